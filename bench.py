"""Benchmark of batched paged-KV decode attention on GB300.

One step = one ``oxd_paged_decode_run`` (the decode kernel; the merge kernel
when a request is split; for a cascade plan also the prefix tiles) over one
batch of the workload, with the plan built and bound to its workspace
beforehand (``oxd_plan_bind_workspace`` copies the work list into the
workspace once, as a server does once per batch and then reuses for every
layer; ``--work-list params`` runs unbound instead).

Default workload: GQA8, Hq=64, Hkv=8, D=128, B=256, KV lengths uniform in
[128, 16384], page size 16, NHD, bf16 ~N(0, 1.5), the first 1024 tokens'
pages shared read-only by groups of 8 consecutive requests, random page
order; out and lse. The workload declares its shared prefixes, so the plan
is the cascade (each group's prefix attended once; ``--plan plain`` for the
other). ``--config`` picks another workload; the default run also measures
the other four (and the default workload on the plain plan) in the same
process under ``workloads``.

Metric: KV-read GB/s and us per step. ``value`` counts the unique KV bytes a
step must read (each shared prefix page once: sum over physical pages in use
of page_size * Hkv * D * 2 (K, V) * 2 B) over the mean step time;
``logical_gbs`` counts every request's pages (sum_b L_b * Hkv * D * 4 B).
Both bases are the same for workloads without shared pages.

Timing: W untimed warm-up steps, then K steps, each between its own pair of
CUDA events on the launching stream; before every step (outside its events)
L2 (129 MB) is flushed by writing a 512 MiB buffer and then reading another
512 MiB buffer (so no dirty flush lines are written back during the step).
The kernel-only time comes from events the library records around the
decode launch. ``warm_l2_us_per_step`` is the median of back-to-back steps
with no flush in between. ``e2e`` repeats the step through the public API
from pinned host buffers: H2D copies of q, the K/V pools and the block
tables, the run, and the D2H read of out and lse, all inside the events;
``e2e_cache_resident`` does the same with the K/V pools left on the device
(q and the tables up, out and lse back). Clocks are sampled with nvidia-smi
during the timed loop.

``parity`` compares the timed run's out and lse with the f64 CPU oracle on
every head (|out - ref| <= 1.5e-2 + 1e-2 |ref|, |lse - ref| <= 1e-3);
``cpu_baseline`` is that oracle's time on the host cores.

``--impl reference`` times the f64 CPU oracle (the reference arm) on a
bounded sample of the same workload on the host cores.

Multi-GPU (torchrun, one rank per GPU): requests are independent, so each rank
decodes its own batch of the workload (weak scaling) with no collective on
the data path; the only collectives are the timing barrier and the max of
the ranks' times.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "paged decode attention: KV-read HBM GB/s (% of GB300 peak), µs per batch step"
DEFAULT_CONFIG = "gqa8_b256_u128to16384_prefix1024x8_ps16_nhd"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["oxd", "reference"], default="oxd")
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=W.CONFIG_ORDER)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target wall time of the oracle baseline sample")
    ap.add_argument("--ref-budget-s", type=float, default=120.0,
                    help="wall-time budget of a whole --impl reference run")
    ap.add_argument("--raw-samples", default=None, metavar="PATH",
                    help="write every timed step's and kernel launch's microseconds (and the "
                         "warm-L2 steps') to PATH as JSON")
    ap.add_argument("--batch", type=int, default=None,
                    help="run only the workload's first N requests (smaller profiling cases)")
    ap.add_argument("--work-list", choices=["bound", "params"], default="bound",
                    help="bound: the plan is bound to its workspace once before the steps; "
                         "params: unbound runs")
    ap.add_argument("--graph", action="store_true",
                    help="capture one run in a CUDA graph and time its replays")
    ap.add_argument("--op", choices=["decode", "rope_append", "prefill", "append_decode"],
                    default="decode",
                    help="rope_append: time the fused RoPE + paged append on the workload's "
                         "tables instead of the decode step; prefill: time the paged causal "
                         "prefill of --prefill-config; append_decode: one engine step, the "
                         "append of each request's new token followed by the decode that reads "
                         "it, with plain launches and with the decode launched as a "
                         "programmatic dependent of the append")
    ap.add_argument("--plan", choices=["auto", "plain", "cascade"], default="auto",
                    help="decode: auto picks the cascade (each sharing group's prefix "
                         "attended once, then the suffixes) for a workload that declares "
                         "shared prefixes, else the plain decode")
    ap.add_argument("--cascade", action="store_true", help="same as --plan cascade")
    ap.add_argument("--no-parity", action="store_true",
                    help="skip the every-head comparison with the f64 oracle")
    ap.add_argument("--no-workloads", action="store_true",
                    help="measure only --config (not the other workloads)")
    ap.add_argument("--record-traffic", nargs=2, metavar=("KEY", "CSV"), default=None,
                    help="no GPU work: read the DRAM bytes of the first paged_decode launch in "
                         "an ncu --csv log of this benchmark and store them in "
                         "profiles/traffic.json under KEY (<workload> or <workload>+cascade), "
                         "keyed to the current decode sources; with --batch, the capture ran "
                         "on that many requests and is scaled to the whole workload by the "
                         "decode kernel's algorithmic bytes")
    ap.add_argument("--prefill-config", default="prefill_gqa4_b8_q2048_kv2048to16384_ps16_nhd",
                    choices=W.PREFILL_ORDER)
    ap.add_argument("--max-splits", type=int, default=0,
                    help="prefill: at most this many pieces per tile (0: the planner decides)")
    ap.add_argument("--tokens-per-request", type=int, default=1,
                    help="rope_append: tokens appended per request in one call (1..64)")
    return ap.parse_args(argv)


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def rank_seed(cfg, rank):
    """Each rank decodes its own batch: same workload shape, seed offset by rank."""
    return cfg.seed + 1000 * rank


def shard_config(cfg, rank):
    import dataclasses

    return dataclasses.replace(cfg, seed=rank_seed(cfg, rank))


def max_over_ranks(ms: float, device=None) -> float:
    """Slowest rank's time (every rank must call this)."""
    import torch
    import torch.distributed as dist

    if not dist.is_initialized() or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank: int, world: int, ms: float) -> float:
    """Aggregate throughput: every rank's bytes over the slowest rank's time."""
    return bytes_per_rank * world / (ms * 1e-3) / 1e9


# ------------------------------------------------------------------ measurement helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a window."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self, steps=None):
        """Samples taken during the marked window (within 60 ms of it: the
        sampling period is 50 ms). With `steps`, also how many timed steps
        each sample strictly inside the window stands for."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:]))
            except (ValueError, IndexError):
                continue
        inside = [r for r in rows if self.t0 - 0.06 <= r[0] <= self.t1 + 0.06]
        used = inside or rows[-3:]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in used for n, v in zip(names, r[3][1:]) if v == "Active"})
        strict = [r for r in rows if self.t0 <= r[0] <= self.t1]
        res = {"sm_mhz": statistics.median(r[1] for r in used), "sm_max_mhz": used[0][2],
               "reasons": reasons, "samples": len(used), "samples_in_window": len(inside),
               "samples_strictly_inside": len(strict),
               "window_ms": (self.t1 - self.t0) * 1e3, "sample_period_ms": 50}
        if steps:
            res["steps_per_sample"] = steps / max(1, len(strict))
        return res


def gpu_id_for_smi(torch, dev):
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return None


DECODE_SOURCES = ("oxd_decode.cu", "oxd_decode_wide.cu", "oxd_host.cpp", "oxd_host_util.h",
                  "oxd_internal.h", "oxd_ptx.cuh", "oxd_tcgen05.cuh")


def strip_comments(src: str) -> str:
    """C/C++ source without its comments (string and character literals kept),
    so that a change of wording alone does not look like a change of code."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return "".join(out)


def source_hash(csrc=None):
    """Hash of the code (comments stripped, white space collapsed) that decides
    a decode launch's DRAM traffic: the planner and the decode kernels with
    their headers (the merge kernel runs in its own launch; the append and
    prefill files never run in a decode step)."""
    h = hashlib.sha256()
    csrc = csrc or os.path.join(ROOT, "paged_kv_decode_attn_gb300", "csrc")
    for name in DECODE_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + " ".join(strip_comments(f.read()).split()).encode())
    return h.hexdigest()[:16]


def ncu_csv_metrics(path, kernel_regex="paged_decode"):
    """Metric name -> value (bytes, or us for durations) of the first launch of a
    kernel matching kernel_regex in an `ncu --csv` log."""
    import csv
    import io
    import re

    txt = open(path).read()
    rows = list(csv.DictReader(io.StringIO(txt[txt.find('"ID"'):])))
    first, vals = None, {}
    for r in rows:
        if not re.search(kernel_regex, r["Kernel Name"]):
            continue
        first = first if first is not None else r["ID"]
        if r["ID"] != first:
            break
        unit, v = r["Metric Unit"], float(r["Metric Value"].replace(",", ""))
        vals[r["Metric Name"]] = v * {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9,
                                      "ns": 1e-3, "nsecond": 1e-3, "us": 1, "usecond": 1,
                                      "ms": 1e3, "msecond": 1e3}.get(unit, 1)
        vals["kernel"] = r["Kernel Name"]
    if not vals:
        raise ValueError(f"no {kernel_regex} launch in {path}")
    return vals


def decode_kernel_bytes(cfg, batch=None):
    """Algorithmic bytes of one decode-kernel launch: the KV bytes it streams
    (a cascade plan's decode kernel skips the shared prefixes of the requests
    it decodes as prefix + suffix; the planner's rule, recomputed on the host)."""
    t = W.make_tables(cfg, batch=batch)
    row = cfg.num_kv_heads * cfg.head_dim * 2 * 2
    return int(t.lengths.sum()) * row


def record_traffic(key, csv_path, batch=None):
    """Store one capture in profiles/traffic.json (see --record-traffic)."""
    name, _, plan = key.partition("+")
    cfg = W.CONFIGS[name]
    v = ncu_csv_metrics(csv_path)
    rd, wr = v["dram__bytes_read.sum"], v["dram__bytes_write.sum"]
    entry = {"source_hash": source_hash(), "kernel": v["kernel"][:80],
             "duration_us_under_ncu": v.get("gpu__time_duration.sum")}
    if batch:
        # the capture ran on the first `batch` requests: scale by the bytes the
        # decode kernel streams (traffic grows with the pages streamed)
        full, part = decode_kernel_bytes(cfg), decode_kernel_bytes(cfg, batch)
        if plan == "cascade":
            full, part = cascade_suffix_bytes(cfg), cascade_suffix_bytes(cfg, batch)
        s = full / part
        entry.update(dram_bytes_per_launch=int((rd + wr) * s), dram_read=int(rd * s),
                     dram_write=int(wr * s), captured_read=int(rd), captured_write=int(wr),
                     captured_algorithmic_bytes=part, full_algorithmic_bytes=full,
                     capture=f"first {batch} requests, one launch; bytes scaled to the whole "
                             f"batch by the decode kernel's algorithmic bytes (x {s:.4f})")
    else:
        entry.update(dram_bytes_per_launch=int(rd + wr), dram_read=int(rd), dram_write=int(wr),
                     capture="full-size workload, one launch")
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        d = {}
    d[key] = entry
    with open(path, "w") as f:
        json.dump(d, f, indent=1)
        f.write("\n")
    print(json.dumps({key: entry}))
    return 0


def cascade_suffix_bytes(cfg, batch=None):
    """Bytes a cascade plan's decode kernel streams: every request's pages after
    the shared prefix when it is decoded as prefix + suffix (longer than the
    prefix, in a group with at least two such requests), else all of them."""
    t = W.make_tables(cfg, batch=batch)
    L = t.lengths
    P, S = cfg.shared_prefix_tokens, cfg.share_group
    tok = 0
    for g0 in range(0, len(L), S):
        grp = L[g0:g0 + S]
        members = grp > P
        if members.sum() >= 2:
            tok += int((grp[members] - P).sum() + grp[~members].sum())
        else:
            tok += int(grp.sum())
    return tok * cfg.num_kv_heads * cfg.head_dim * 2 * 2


def recorded_traffic(workload):
    """DRAM bytes per decode launch from the committed ncu summary, if it still applies.
    A cascade plan's decode kernel streams fewer pages than the plain plan's: its
    entries are keyed "<workload>+cascade"."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("source_hash") == source_hash():
            return e.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


# ------------------------------------------------------------------ the oracle baseline

def oracle_time(case, heads=None, reps=1, nthreads=0, bits=None):
    import oracle

    bits = bits or (W.bf16_bits(case.q), W.bf16_bits(case.k), W.bf16_bits(case.v))
    args = (*bits, case.tables.indptr, case.tables.indices, case.tables.last_page_len)
    kw = dict(num_kv_heads=case.num_kv_heads, page_size=case.page_size,
              layout=0 if case.layout == "NHD" else 1, sm_scale=case.sm_scale, heads=heads,
              nthreads=nthreads)
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.paged_decode(*args, **kw)
    return time.perf_counter() - t0


def cpu_baseline(case, bits, target_s, t_first=None, single_thread=False):
    """Oracle (as it stands) on the whole batch on all host cores, repeated to
    about target_s seconds (t_first: the time of a pass already made, which
    counts as the first repetition); with single_thread, also one pass of the
    batch on one thread. GB/s on the same byte basis as the GPU arm's value
    (unique KV bytes)."""
    cores = os.cpu_count() or 1
    t1 = t_first if t_first is not None else oracle_time(case, bits=bits)
    more = max(0, min(1000, int(math.ceil(target_s / max(t1, 1e-6)))) - 1)
    t = t1 + (oracle_time(case, reps=more, bits=bits) if more > 0 else 0.0)
    reps = more + 1
    per = t / reps
    out = {"value": case.unique_kv_bytes() / per / 1e9, "unit": "GB/s", "cores": cores,
           "kind": "oracle", "ms_per_step": per * 1e3,
           "logical_gbs": case.kv_bytes() / per / 1e9,
           "sample": f"whole workload batch ({case.batch} requests, "
                     f"{case.batch * case.num_qo_heads} heads), f64 oracle over "
                     f"{cores} threads, {reps} repetition(s), {per * 1e3:.1f} ms each",
           "seconds": t}
    if single_thread:
        t_st = oracle_time(case, nthreads=1, bits=bits)
        out["single_thread_value"] = case.unique_kv_bytes() / t_st / 1e9
        out["single_thread_ms_per_step"] = t_st * 1e3
    return out


# ------------------------------------------------------------------ reference arm

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    cfg = W.CONFIGS[args.config]
    case = W.make_case(cfg, device="cpu", batch=args.batch)
    import oracle

    oracle.build()
    L = case.tables.lengths
    # One step = the oracle over a bounded subset of heads, sized so that the
    # whole run (K + W steps) takes about two minutes.
    t_one = oracle_time(case, heads=[(int(np.argmax(L)), 0)])
    per_head = max(t_one, 1e-5)
    budget = args.ref_budget_s / max(1, args.steps + args.warmup)
    n_heads_total = case.batch * case.num_qo_heads
    n = int(max(1, min(n_heads_total, budget / per_head)))
    rng = np.random.default_rng(cfg.seed)
    flat = rng.permutation(n_heads_total)[:n]
    heads = [(int(i // case.num_qo_heads), int(i % case.num_qo_heads)) for i in flat]
    # The metric counts each KV head's bytes once per step; the G query heads of
    # a group read the same K and V, so a sampled query head stands for 1/G of
    # its KV head's bytes.
    G = case.num_qo_heads // case.num_kv_heads
    sample_bytes = sum(int(L[b]) for b, _ in heads) * case.head_dim * 4 / G
    bits = (W.bf16_bits(case.q), W.bf16_bits(case.k), W.bf16_bits(case.v))
    for _ in range(args.warmup):
        oracle_time(case, heads=heads, bits=bits)
    times = [oracle_time(case, heads=heads, bits=bits) for _ in range(args.steps)]
    per = statistics.mean(times)
    # A whole batch step at the sampled rate: the sample stands for
    # sample_bytes of the step's kv_bytes. value is on the GPU arm's basis
    # (unique KV bytes over the step time).
    step_s = per * case.kv_bytes() / sample_bytes
    gbs = case.unique_kv_bytes() / step_s / 1e9
    cores = os.cpu_count() or 1
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(cfg, case),
        "logical_gbs": case.kv_bytes() / step_s / 1e9,
        "sample_ms_per_step": per * 1e3,
        "heads_sampled": n, "heads_total": n_heads_total,
        "ms_per_step_basis": "a whole batch step at the sampled rate: the sampled heads' time "
                             "times the step's KV bytes over the sample's",
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} of {n_heads_total} query heads per step (each head's "
                                   "whole KV sequence), f64 oracle"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_block(cfg, case):
    return {"workload": cfg.name, "batch": case.batch, "num_qo_heads": case.num_qo_heads,
            "num_kv_heads": case.num_kv_heads, "head_dim": case.head_dim,
            "page_size": case.page_size, "layout": case.layout,
            "kv_lengths": list(cfg.lengths), "value_sigma": cfg.sigma,
            "kv_tokens": int(case.tables.lengths.sum()), "kv_bytes_per_step": case.kv_bytes(),
            "unique_kv_bytes_per_step": case.unique_kv_bytes(),
            "shared_prefix_tokens": cfg.shared_prefix_tokens,
            "requests_run": case.batch,
            "l2": "flushed before every timed step, outside its events: 512 MiB write, "
                  "then a 512 MiB read of another buffer"}


# ------------------------------------------------------------------ our arm

ATOL, RTOL, LSE_ATOL = 1.5e-2, 1e-2, 1e-3


def plan_kind_for(cfg, requested):
    """The plan a server would pick: the cascade when the workload declares
    requests that share their leading pages, else the plain decode."""
    can = cfg.shared_prefix_tokens > 0 and cfg.share_group > 1
    if requested == "auto":
        return "cascade" if can else "plain"
    if requested == "cascade" and not can:
        return "plain"
    return requested


def oracle_inputs(case, host=None):
    """Host uint16 views of q, K, V for the oracle (from pinned copies when given)."""
    src = host or {"q": case.q, "k": case.k, "v": case.v}
    return W.bf16_bits(src["q"]), W.bf16_bits(src["k"]), W.bf16_bits(src["v"])


def oracle_full(case, bits, nthreads=0):
    """The f64 oracle on every head of the batch; returns (out, lse, seconds)."""
    import oracle

    t0 = time.perf_counter()
    out, lse = oracle.paged_decode(
        *bits, case.tables.indptr, case.tables.indices, case.tables.last_page_len,
        num_kv_heads=case.num_kv_heads, page_size=case.page_size,
        layout=0 if case.layout == "NHD" else 1, sm_scale=case.sm_scale, nthreads=nthreads)
    return out, lse, time.perf_counter() - t0


def parity_report(out, lse, ref_out, ref_lse):
    """Element-by-element comparison of a run's out/lse with the f64 oracle on
    every head: |out - ref| <= 1.5e-2 + 1e-2 |ref|, |lse - ref| <= 1e-3."""
    o = out.float().cpu().numpy().astype(np.float64)
    err = np.abs(o - ref_out)
    rel = err / (ATOL + RTOL * np.abs(ref_out))
    lg = lse.float().cpu().numpy().astype(np.float64)
    lerr = np.abs(lg - ref_lse)
    ok = bool(np.isfinite(o).all() and np.isfinite(lg).all() and rel.max() <= 1.0 and
              lerr.max() <= LSE_ATOL)
    return {"heads_checked": int(o.shape[0] * o.shape[1]),
            "elements_checked": int(o.size), "max_abs_err": float(err.max()),
            "max_rel_to_bound": float(rel.max()), "max_lse_err": float(lerr.max()),
            "tolerance": "out: 1.5e-2 + 1e-2 |ref|; lse: 1e-3 (f64 oracle, every head)",
            "pass": ok}


class Flusher:
    """Write 512 MiB, then read another 512 MiB: L2 (129 MB) ends up with clean
    lines of neither the workload nor the written buffer, so no write-back of
    flush data lands inside the next timed step."""

    def __init__(self, torch, dev):
        self.w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(128 << 20, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()


def measure_decode(oxd, torch, case, cfg, plan_kind, dev, stream, flush, K, Wm,
                   work_list="bound", graph=False, sampler=None, world=1):
    """Plan, bind and time one workload: K steps after Wm warm-ups, an L2
    flush before each (outside its events); then up to 200 back-to-back steps
    with a warm L2 and the decode kernel alone over up to 200 flushed steps
    (events the library records around its launch)."""
    t = case.tables
    casc = {}
    if plan_kind == "cascade":
        casc = dict(shared_prefix_tokens=cfg.shared_prefix_tokens, share_group=cfg.share_group)
    desc = oxd.make_desc(case.batch, case.num_qo_heads, case.num_kv_heads, case.page_size,
                         case.layout, t.num_pages, **casc)
    tp0 = time.perf_counter()
    plan = oxd.oxd_paged_decode_plan(desc, t.indptr, t.last_page_len, dev.index)
    plan_us = (time.perf_counter() - tp0) * 1e6
    info = plan.info
    indptr = torch.as_tensor(t.indptr, device=dev)
    indices = torch.as_tensor(t.indices, device=dev)
    last = torch.as_tensor(t.last_page_len, device=dev)
    out = torch.empty_like(case.q)
    lse = torch.empty(case.batch, case.num_qo_heads, dtype=torch.float32, device=dev)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    bind_us = None
    if work_list == "bound":
        torch.cuda.synchronize(dev)
        tb0 = time.perf_counter()
        oxd.oxd_plan_bind_workspace(plan, ws, plan.workspace_bytes, stream)
        torch.cuda.synchronize(dev)
        bind_us = (time.perf_counter() - tb0) * 1e6

    def run_once(s):
        oxd.oxd_paged_decode_run(plan, case.q, case.k, case.v, indptr, indices, last,
                                 case.sm_scale, out, lse, ws, plan.workspace_bytes, s)

    g = None
    if graph:
        # one run captured with every pointer fixed; replays re-read the
        # buffers' current contents
        run_once(stream)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run_once(torch.cuda.current_stream(dev))

    def step():
        if g is not None:
            g.replay()
        else:
            run_once(stream)

    for _ in range(Wm):
        flush()
        step()
    if oxd.oxd_read_device_status(ws, stream) != 0:
        raise RuntimeError(f"{cfg.name}: device status error during warm-up")

    # ---- timed steps: the production path, events only around each step
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.mark_start()
    wall0 = time.perf_counter()
    for k in range(K):
        flush()
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if sampler:
        sampler.mark_end()
    if world > 1:
        torch.distributed.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    if oxd.oxd_read_device_status(ws, stream) != 0:
        raise RuntimeError(f"{cfg.name}: device status error during the timed steps")

    # ---- back-to-back steps with a warm L2 (no flush)
    Kw = max(3, min(K, 200))
    wev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(Kw)]
    torch.cuda.synchronize(dev)
    for a, b in wev:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize(dev)
    warm_ms = sorted(a.elapsed_time(b) for a, b in wev)

    # ---- the decode kernel alone (roofline): events the library records
    # around its launch, in a separate loop so they never perturb the steps
    Kk = max(3, min(K, 200))
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(Kk)]
    for a, b in kev:  # materialise the events so their handles exist
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    for k in range(Kk):
        flush()
        oxd.oxd_plan_set_timing_events(plan, kev[k][0], kev[k][1])
        run_once(stream)  # direct runs: the events are recorded by the run itself
    torch.cuda.synchronize(dev)
    oxd.oxd_plan_set_timing_events(plan, None, None)
    kern_ms = [a.elapsed_time(b) for a, b in kev]
    if oxd.oxd_read_device_status(ws, stream) != 0:
        raise RuntimeError(f"{cfg.name}: device status error in the kernel-only loop")

    # Bytes the timed decode kernel reads. In a cascade plan the prefill kernel
    # reads the shared-prefix tokens of the cascade requests (once per group)
    # and the decode kernel the rest of each request's cache.
    kern_bytes = case.kv_bytes()
    if casc:
        kern_bytes -= (info.cascade_requests * cfg.shared_prefix_tokens * case.num_kv_heads *
                       case.head_dim * 2 * 2)
    return dict(plan=plan, info=info, plan_us=plan_us, bind_us=bind_us, out=out, lse=lse,
                ws=ws, indptr=indptr, indices=indices, last=last, step_ms=step_ms,
                warm_ms=warm_ms, kern_ms=kern_ms, kern_launches=Kk, kern_bytes=kern_bytes,
                wall=wall, run_once=run_once, casc=casc)


def summary(case, m, peak, traffic_key, parity):
    """One workload's figures for the bench line."""
    ms = statistics.mean(m["step_ms"])
    kern = statistics.mean(m["kern_ms"])
    srt = sorted(m["step_ms"])
    uniq = case.unique_kv_bytes()
    return {
        "us_per_step": ms * 1e3,
        "us_per_step_p10_p50_p90": [srt[len(srt) // 10] * 1e3, srt[len(srt) // 2] * 1e3,
                                    srt[(9 * len(srt)) // 10] * 1e3],
        "warm_l2_us_per_step": m["warm_ms"][len(m["warm_ms"]) // 2] * 1e3,
        "unique_gbs": uniq / (ms * 1e-3) / 1e9,
        "logical_gbs": case.kv_bytes() / (ms * 1e-3) / 1e9,
        "pct_of_hbm_peak": 100.0 * uniq / (ms * 1e-3) / 1e9 / peak,
        "kv_bytes_per_step": case.kv_bytes(), "unique_kv_bytes_per_step": uniq,
        "kernel_us": kern * 1e3,
        "kernel_frac": m["kern_bytes"] / (kern * 1e-3) / 1e9 / peak,
        "kernel_algorithmic_bytes": m["kern_bytes"],
        "traffic": recorded_traffic(traffic_key),
        "launches_per_step": m["info"].launches_per_run,
        "plan_host_us": m["plan_us"],
        "parity": parity,
    }


def run_oxd(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    import paged_kv_decode_attn_gb300 as oxd

    oxd.build()
    cfg = shard_config(W.CONFIGS[args.config], rank)
    kind = plan_kind_for(cfg, "cascade" if args.cascade else args.plan)
    case = W.make_case(cfg, device=dev, batch=args.batch)
    cfg_block = config_block(cfg, case)
    stream = torch.cuda.current_stream(dev)
    flush = Flusher(torch, dev)
    peak, peak_kind = measured_peaks()
    solo = rank == 0 and world == 1
    check = solo and not args.no_parity
    if check or (solo and not args.no_cpu_baseline):
        import oracle

        oracle.build()  # compiled on the host before any timed region

    sampler = ClockSampler(gpu_id_for_smi(torch, dev)) if rank == 0 else None
    if sampler:
        sampler.start()
    m = measure_decode(oxd, torch, case, cfg, kind, dev, stream, flush, args.steps, args.warmup,
                       work_list=args.work_list, graph=args.graph, sampler=sampler, world=world)
    clocks = sampler.stop(steps=args.steps) if sampler else None
    info, plan, ws, out, lse = m["info"], m["plan"], m["ws"], m["out"], m["lse"]
    timed_out, timed_lse = out.clone(), lse.clone()  # the timed run's results

    ms = max_over_ranks(statistics.mean(m["step_ms"]), dev)
    kv_bytes, uniq = case.kv_bytes(), case.unique_kv_bytes()
    value = whole_job_gbs(uniq, world, ms)
    kern = statistics.mean(m["kern_ms"])
    achieved = m["kern_bytes"] / (kern * 1e-3) / 1e9
    traffic_key = cfg.name + ("+cascade" if kind == "cascade" else "")
    head = summary(case, m, peak, traffic_key, None)
    kern_launches, bind_us, wall = m["kern_launches"], m["bind_us"], m["wall"]
    if args.raw_samples and rank == 0:
        with open(args.raw_samples, "w") as f:
            json.dump({"workload": cfg.name, "plan": kind,
                       "step_us": [x * 1e3 for x in m["step_ms"]],
                       "kernel_us": [x * 1e3 for x in m["kern_ms"]],
                       "warm_l2_step_us": [x * 1e3 for x in m["warm_ms"]]}, f)

    # ---- end to end through the public API from pinned host buffers
    host = {name: x.cpu().pin_memory() for name, x in
            (("q", case.q), ("k", case.k), ("v", case.v), ("indptr", m["indptr"]),
             ("indices", m["indices"]), ("last", m["last"]))}
    out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    lse_h = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    dq, dk, dv = torch.empty_like(case.q), torch.empty_like(case.k), torch.empty_like(case.v)
    dind, dptr, dlast = (torch.empty_like(m["indices"]), torch.empty_like(m["indptr"]),
                         torch.empty_like(m["last"]))
    h2d = sum(x.numel() * x.element_size() for x in host.values())
    d2h = out.numel() * out.element_size() + lse.numel() * lse.element_size()

    def e2e_step():
        dq.copy_(host["q"], non_blocking=True)
        dk.copy_(host["k"], non_blocking=True)
        dv.copy_(host["v"], non_blocking=True)
        dptr.copy_(host["indptr"], non_blocking=True)
        dind.copy_(host["indices"], non_blocking=True)
        dlast.copy_(host["last"], non_blocking=True)
        oxd.oxd_paged_decode_run(plan, dq, dk, dv, dptr, dind, dlast, case.sm_scale, out, lse,
                                 ws, plan.workspace_bytes, stream)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    n_e2e = max(3, min(args.e2e_steps, args.steps))
    e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(n_e2e)]
    for a, b in e_ev:
        flush()
        a.record(stream)
        e2e_step()
        b.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in e_ev), dev)
    if not torch.equal(out_h, out.cpu()):
        raise RuntimeError("e2e output mismatch")

    # ---- the same with the K/V cache resident on the device (as a serving
    # engine keeps it): only q and the block tables go up, out and lse come back
    def e2e_resident_step():
        dq.copy_(host["q"], non_blocking=True)
        dptr.copy_(host["indptr"], non_blocking=True)
        dind.copy_(host["indices"], non_blocking=True)
        dlast.copy_(host["last"], non_blocking=True)
        oxd.oxd_paged_decode_run(plan, dq, case.k, case.v, dptr, dind, dlast, case.sm_scale,
                                 out, lse, ws, plan.workspace_bytes, stream)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)

    for _ in range(3):
        e2e_resident_step()
    r_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(n_e2e)]
    for a, b in r_ev:
        flush()
        a.record(stream)
        e2e_resident_step()
        b.record(stream)
    torch.cuda.synchronize(dev)
    res_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in r_ev), dev)
    if not torch.equal(out_h, out.cpu()):
        raise RuntimeError("e2e (resident cache) output mismatch")
    h2d_res = sum(host[n].numel() * host[n].element_size()
                  for n in ("q", "indptr", "indices", "last"))
    del dq, dk, dv, dind, dptr, dlast

    # ---- parity of the timed run with the f64 oracle on every head, and the
    # oracle's own time on the host cores (the CPU baseline)
    cpu, ref = None, None
    if solo and (check or not args.no_cpu_baseline):
        bits = oracle_inputs(case, host)
        ref_out, ref_lse, t_pass = oracle_full(case, bits)
        ref = (ref_out, ref_lse)
        if check:
            head["parity"] = dict(parity_report(timed_out, timed_lse, ref_out, ref_lse),
                                  oracle_ms=t_pass * 1e3, oracle_cores=os.cpu_count() or 1)
        if not args.no_cpu_baseline:
            cpu = cpu_baseline(case, bits, args.cpu_seconds, t_first=t_pass,
                               single_thread=cfg.name in ("mha8_b1_l512_ps16_nhd",
                                                          "gqa4_b32_u512to4096_ps16_nhd"))
        del bits
    del host, out_h, lse_h

    # ---- the other workloads, measured in the same process (one GPU)
    others = None
    if solo and not args.no_workloads and args.batch is None:
        others = {}
        if kind == "cascade":
            # the same batch on the plain plan, for comparison
            mp = measure_decode(oxd, torch, case, cfg, "plain", dev, stream, flush,
                                args.steps, args.warmup)
            par = parity_report(mp["out"], mp["lse"], *ref) if check else None
            others[cfg.name + "+plain"] = dict(summary(case, mp, peak, cfg.name, par),
                                               plan="plain")
            del mp
        del m, out, lse, timed_out, timed_lse
        case = None
        torch.cuda.empty_cache()
        for name in W.CONFIG_ORDER:
            if name == cfg.name:
                continue
            c2 = W.CONFIGS[name]
            k2 = plan_kind_for(c2, "auto")
            case2 = W.make_case(c2, device=dev)
            m2 = measure_decode(oxd, torch, case2, c2, k2, dev, stream, flush, args.steps,
                                args.warmup)
            par = None
            if check:
                r_out, r_lse, t_o = oracle_full(case2, oracle_inputs(case2))
                par = dict(parity_report(m2["out"], m2["lse"], r_out, r_lse),
                           oracle_ms=t_o * 1e3, oracle_cores=os.cpu_count() or 1)
            key = name + ("+cascade" if k2 == "cascade" else "")
            others[name] = dict(summary(case2, m2, peak, key, par), plan=k2)
            del m2, case2
            torch.cuda.empty_cache()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": cfg_block,
            "value_basis": "unique KV bytes read per step (each shared prefix page once) over "
                           "the mean step time; logical_gbs counts every request's pages",
            "us_per_step": ms * 1e3,
            "us_per_step_p10_p50_p90": head["us_per_step_p10_p50_p90"],
            "warm_l2_us_per_step": head["warm_l2_us_per_step"],
            "unique_gbs": value, "logical_gbs": whole_job_gbs(kv_bytes, world, ms),
            "pct_of_hbm_peak": 100.0 * value / world / peak,
            "pct_of_nominal_hbm": 100.0 * value / world / NOMINAL_HBM_GBS,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind,
                         "traffic": head["traffic"],
                         "kernel": f"paged_decode_kernel variant {info.kernel_variant}",
                         "kernel_us": kern * 1e3, "kernel_timed_launches": kern_launches,
                         "algorithmic_bytes_per_launch": head["kernel_algorithmic_bytes"]},
            "parity": head["parity"],
            "cpu_baseline": cpu,
            "e2e": {"value": whole_job_gbs(uniq, world, e2e_ms), "unit": "GB/s",
                    "ms_per_step": e2e_ms, "steps": n_e2e,
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "inputs": "q, both K/V pools and the block tables copied up every step"},
            "e2e_cache_resident": {
                "value": whole_job_gbs(uniq, world, res_ms), "unit": "GB/s",
                "ms_per_step": res_ms, "steps": n_e2e, "h2d_bytes_per_step": h2d_res,
                "d2h_bytes_per_step": d2h,
                "inputs": "q and the block tables copied up every step; the K/V pools stay "
                          "on the device, as a serving engine keeps its cache"},
            "gpu_launches": args.steps * info.launches_per_run,
            "clocks": clocks,
            "plan": {"kind": kind, "host_us": head["plan_host_us"], "work_list": args.work_list,
                     "bind_us": bind_us, "cuda_graph": bool(args.graph),
                     **info.as_dict()},
            "workloads": others,
            "wall_s_timed_loop": wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


def run_rope_append(args):
    """Fused RoPE + paged append on the workload's shapes: every request gets
    `tokens_per_request` new tokens (its block table already covers them).
    Metric: bytes the operation must move (q read and written, k and v read,
    K and V rows written) per second."""
    import torch

    import paged_kv_decode_attn_gb300 as oxd

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    oxd.build()
    cfg = W.CONFIGS[args.config]
    n_new = args.tokens_per_request
    t0 = W.make_tables(cfg, batch=args.batch)
    lengths = t0.lengths
    case = W.custom_case([int(L) + n_new for L in lengths], num_qo_heads=cfg.num_qo_heads,
                         num_kv_heads=cfg.num_kv_heads, page_size=cfg.page_size,
                         layout=cfg.layout, seed=cfg.seed, device=dev)
    t = case.tables
    B, Hq, Hkv = case.batch, case.num_qo_heads, case.num_kv_heads
    tok = torch.arange(B, dtype=torch.int32, device=dev).repeat_interleave(n_new)
    pos = (torch.as_tensor(lengths, device=dev).to(torch.int32).repeat_interleave(n_new) +
           torch.arange(n_new, dtype=torch.int32, device=dev).repeat(B))
    T = B * n_new
    g = torch.Generator(device=dev).manual_seed(cfg.seed)
    q = torch.randn(T, Hq, 128, generator=g, device=dev).to(torch.bfloat16)
    k = torch.randn(T, Hkv, 128, generator=g, device=dev).to(torch.bfloat16)
    v = torch.randn(T, Hkv, 128, generator=g, device=dev).to(torch.bfloat16)
    q_out = torch.empty_like(q)
    indptr = torch.as_tensor(t.indptr, device=dev)
    indices = torch.as_tensor(t.indices, device=dev)
    refcount = torch.ones(t.num_pages, dtype=torch.int32, device=dev)
    ws = torch.empty(256, dtype=torch.uint8, device=dev)
    desc = oxd.make_rope_append_desc(T, B, Hq, Hkv, case.page_size, case.layout, t.num_pages,
                                     int(t.indptr[-1]))
    stream = torch.cuda.current_stream(dev)
    flush_w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(128 << 20, dtype=torch.float32, device=dev)

    def step():
        oxd.oxd_rope_append(desc, q, k, v, tok, pos, indptr, indices, refcount, q_out, case.k,
                            case.v, ws, 256, stream)

    for _ in range(args.warmup):
        flush_w.zero_()
        flush_r.sum()
        step()
    if oxd.oxd_read_device_status(ws, stream) != 0:
        raise RuntimeError("device status error in the append")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    for a, b in ev:
        flush_w.zero_()
        flush_r.sum()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize(dev)
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    moved = T * (2 * Hq + 4 * Hkv) * 128 * 2
    peak, peak_kind = measured_peaks()
    gbs = moved / (ms * 1e-3) / 1e9
    print(json.dumps({
        "impl": "oxd", "op": "rope_append",
        "metric": "fused RoPE + paged KV append: bytes moved GB/s, us per call",
        "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "us_per_call": ms * 1e3, "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": cfg.name, "batch": B, "tokens_per_request": n_new, "tokens": T,
                   "num_qo_heads": Hq, "num_kv_heads": Hkv, "page_size": case.page_size,
                   "layout": case.layout, "bytes_moved_per_call": moved,
                   "l2": "flushed before every call, outside its events"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                     "frac": gbs / peak, "peak_source": peak_kind},
    }), flush=True)
    return 0


def run_append_decode(args):
    """One engine step of a decode layer: oxd_rope_append writes each request's
    new token (rotated q, K and V rows in their page slots), then
    oxd_paged_decode_run attends over the grown cache. Timed four ways, an L2
    flush before each step: the append alone, the decode alone, the two with
    plain launches, and the two with the decode launched as a programmatic
    dependent of the append (plan pdl = 1). Metric as for decode: unique KV
    bytes per step over the step time."""
    import torch

    import paged_kv_decode_attn_gb300 as oxd

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    oxd.build()
    cfg = W.CONFIGS[args.config]
    kind = plan_kind_for(cfg, "cascade" if args.cascade else args.plan)
    lengths = W.make_tables(cfg, batch=args.batch).lengths
    casc = {}
    if kind == "cascade":
        casc = dict(shared_prefix_tokens=cfg.shared_prefix_tokens, share_group=cfg.share_group)
    case = W.custom_case([int(L) + 1 for L in lengths], num_qo_heads=cfg.num_qo_heads,
                         num_kv_heads=cfg.num_kv_heads, page_size=cfg.page_size,
                         layout=cfg.layout, seed=cfg.seed, sigma=cfg.sigma, device=dev, **casc)
    t = case.tables
    B, Hq, Hkv = case.batch, case.num_qo_heads, case.num_kv_heads
    g = torch.Generator(device=dev).manual_seed(cfg.seed)
    q_new = torch.randn(B, Hq, 128, generator=g, device=dev).to(torch.bfloat16)
    k_new = torch.randn(B, Hkv, 128, generator=g, device=dev).to(torch.bfloat16)
    v_new = torch.randn(B, Hkv, 128, generator=g, device=dev).to(torch.bfloat16)
    tok = torch.arange(B, dtype=torch.int32, device=dev)
    pos = torch.as_tensor(lengths, device=dev).to(torch.int32)
    indptr = torch.as_tensor(t.indptr, device=dev)
    indices = torch.as_tensor(t.indices, device=dev)
    last = torch.as_tensor(t.last_page_len, device=dev)
    # each page's reference count is the number of requests that list it: a
    # token whose slot lies in a page shared with other requests is refused by
    # the append (the pages' write rule; an engine makes that page private
    # first), the others are written
    rc = np.bincount(t.indices, minlength=t.num_pages).astype(np.int32)
    refcount = torch.as_tensor(rc, device=dev)
    slot_page = t.indices[t.indptr[:-1] + np.asarray(lengths) // case.page_size]
    n_shared_slot = int((rc[slot_page] > 1).sum())
    aws = torch.empty(256, dtype=torch.uint8, device=dev)
    adesc = oxd.make_rope_append_desc(B, B, Hq, Hkv, case.page_size, case.layout, t.num_pages,
                                      int(t.indptr[-1]))
    stream = torch.cuda.current_stream(dev)
    plans = {}
    for pdl in (0, 1):
        desc = oxd.make_desc(B, Hq, Hkv, case.page_size, case.layout, t.num_pages, pdl=pdl,
                             **casc)
        plan = oxd.oxd_paged_decode_plan(desc, t.indptr, t.last_page_len, 0)
        ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
        oxd.oxd_plan_bind_workspace(plan, ws, plan.workspace_bytes, stream)
        plans[pdl] = (plan, ws)
    q = torch.empty_like(q_new)
    out = torch.empty_like(q_new)
    lse = torch.empty(B, Hq, device=dev)
    flush = Flusher(torch, dev)

    def append():
        oxd.oxd_rope_append(adesc, q_new, k_new, v_new, tok, pos, indptr, indices, refcount, q,
                            case.k, case.v, aws, 256, stream)

    def decode(pdl):
        plan, ws = plans[pdl]
        oxd.oxd_paged_decode_run(plan, q, case.k, case.v, indptr, indices, last, case.sm_scale,
                                 out, lse, ws, plan.workspace_bytes, stream)

    ways = {"append": append, "decode": lambda: decode(0),
            "append_then_decode": lambda: (append(), decode(0)),
            "append_then_decode_pdl": lambda: (append(), decode(1))}
    times = {}
    K, Wm = args.steps, max(3, args.warmup)
    for r in range(2):  # two rounds, alternating order
        for name in (list(ways) if r == 0 else list(reversed(list(ways)))):
            fn = ways[name]
            for _ in range(Wm):
                flush()
                fn()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(K)]
            torch.cuda.synchronize(dev)
            for a, b_ in ev:
                flush()
                a.record(stream)
                fn()
                b_.record(stream)
            torch.cuda.synchronize(dev)
            times.setdefault(name, []).extend(a.elapsed_time(b_) for a, b_ in ev)
    want = oxd.OXD_DEVICE_SHARED_PAGE if n_shared_slot else oxd.OXD_DEVICE_OK
    if oxd.oxd_read_device_status(aws, stream) != want:
        raise RuntimeError("unexpected device status in the append")
    for _, ws_ in plans.values():
        if oxd.oxd_read_device_status(ws_, stream) != 0:
            raise RuntimeError("device status error in the decode")
    us = {k: statistics.mean(v) * 1e3 for k, v in times.items()}
    uniq = case.unique_kv_bytes()
    step_ms = us["append_then_decode_pdl"] * 1e-3
    peak, peak_kind = measured_peaks()
    print(json.dumps({
        "impl": "oxd", "op": "append_decode",
        "metric": "append + decode step: unique KV-read GB/s, us per step",
        "value": uniq / (step_ms * 1e-3) / 1e9, "unit": "GB/s", "n_gpus": 1,
        "steps": K, "warmup": Wm, "ms_per_step": step_ms, "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg.name, "plan": kind, "batch": B, "new_tokens": B,
                   "tokens_refused_shared_page": n_shared_slot,
                   "kv_bytes_per_step": case.kv_bytes(), "unique_kv_bytes_per_step": uniq,
                   "l2": "flushed before every step, outside its events"},
        "us": us,
        "sum_of_parts_us": us["append"] + us["decode"],
        "pdl_saves_us": us["append_then_decode"] - us["append_then_decode_pdl"],
        "pct_of_hbm_peak": 100.0 * uniq / (step_ms * 1e-3) / 1e9 / peak,
        "gpu_launches": K * (1 + plans[1][0].info.launches_per_run),
    }), flush=True)
    return 0


def run_prefill(args):
    """Paged causal prefill of one prefill workload. A step is one
    oxd_paged_prefill_run on the bound workspace (the prefill kernel and, when
    tiles were split, the merge behind it). Metric: causal attention flops
    (4 D per attended (query token, cached token) pair per query head) per
    second; the roofline is the prefill kernel alone against the measured
    bf16 tensor peak."""
    import torch

    import paged_kv_decode_attn_gb300 as oxd

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    oxd.build()
    cfg = W.PREFILL_CONFIGS[args.prefill_config]
    case = W.make_prefill_case(cfg, device=dev)
    t = case.tables
    desc = oxd.make_prefill_desc(case.batch, case.num_qo_heads, case.num_kv_heads,
                                 case.page_size, case.layout, t.num_pages,
                                 max_splits=args.max_splits)
    h0 = time.perf_counter()
    plan = oxd.oxd_paged_prefill_plan(desc, case.qo_indptr, t.indptr, t.last_page_len)
    host_us = (time.perf_counter() - h0) * 1e6
    info = plan.info
    qo = torch.as_tensor(case.qo_indptr, device=dev)
    indptr = torch.as_tensor(t.indptr, device=dev)
    indices = torch.as_tensor(t.indices, device=dev)
    last = torch.as_tensor(t.last_page_len, device=dev)
    out = torch.empty_like(case.q)
    lse = torch.empty(case.q.shape[:2], device=dev)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    oxd.oxd_prefill_plan_bind_workspace(plan, ws, stream=stream)
    flush_w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(128 << 20, dtype=torch.float32, device=dev)

    def flush():
        flush_w.zero_()
        flush_r.sum()

    def step():
        oxd.oxd_paged_prefill_run(plan, case.q, case.k, case.v, qo, indptr, indices, last,
                                  case.sm_scale, out, lse, ws, stream=stream)

    W_ = max(3, args.warmup)
    for _ in range(W_):
        flush()
        step()
    if oxd.oxd_read_device_status(ws, stream) != 0:
        raise RuntimeError("device status error in the prefill warm-up")
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    sampler = ClockSampler(gpu_id_for_smi(torch, dev))
    sampler.start()
    torch.cuda.synchronize(dev)
    sampler.mark_start()
    for a, b in ev:
        flush()
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize(dev)
    sampler.mark_end()
    clocks = sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    if oxd.oxd_read_device_status(ws, stream) != 0:
        raise RuntimeError("device status error during the timed steps")
    # the prefill kernel alone (events the library records around its launch)
    Kk = max(3, min(K, 200))
    kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(Kk)]
    for a, b in kev:  # materialise the events so their handles exist
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    for a, b in kev:
        flush()
        oxd.oxd_prefill_plan_set_timing_events(plan, a, b)
        step()
    torch.cuda.synchronize(dev)
    oxd.oxd_prefill_plan_set_timing_events(plan, None, None)
    kern = [a.elapsed_time(b) for a, b in kev]
    ms = statistics.mean(step_ms)
    k_ms = statistics.mean(kern)
    flops = case.flops()
    tfs = flops / (ms * 1e-3) / 1e12
    k_tfs = flops / (k_ms * 1e-3) / 1e12
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        peak = float(json.load(f)["bf16_tflops"])
    line = {
        "impl": "oxd", "op": "prefill",
        "metric": "paged causal prefill: attention TFLOP/s (4 D flops per attended pair per "
                  "query head), us per call",
        "value": tfs, "unit": "TFLOP/s", "n_gpus": 1, "steps": K, "warmup": W_,
        "ms_per_step": ms, "us_per_call": ms * 1e3,
        "us_p10_p90": [float(np.percentile(step_ms, 10)) * 1e3,
                       float(np.percentile(step_ms, 90)) * 1e3],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": cfg.name, "batch": case.batch, "q_lens": list(cfg.q_lens),
                   "kv_lens": list(cfg.kv_lens), "num_qo_heads": case.num_qo_heads,
                   "num_kv_heads": case.num_kv_heads, "page_size": case.page_size,
                   "layout": case.layout, "flops_per_call": flops,
                   "causal_pairs_per_head": case.causal_pairs(),
                   "l2": "flushed before every call, outside its events"},
        "plan": dict(info.as_dict(), host_us=host_us),
        "roofline": {"bound": "tensor", "achieved": k_tfs, "peak": peak, "unit": "TFLOP/s",
                     "frac": k_tfs / peak, "kernel_us": k_ms * 1e3,
                     "peak_source": "measured bf16 burst"},
        "gpu_launches": K * info.launches_per_run,
        "clocks": clocks,
    }
    if cfg.name.startswith("prefill_gqa4_q32+64"):
        line["context"] = {"pages_h20_us": {"oxide": 46.60, "flashinfer": 23.21},
                           "note": "other hardware (H20): context, not a target"}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.record_traffic:
        return record_traffic(args.record_traffic[0], args.record_traffic[1], args.batch)
    if args.impl == "reference":
        return run_reference(args)
    if args.op == "rope_append":
        return run_rope_append(args)
    if args.op == "prefill":
        return run_prefill(args)
    if args.op == "append_decode":
        return run_append_decode(args)
    return run_oxd(args)


if __name__ == "__main__":
    sys.exit(main())
