"""Host-side logic of bench.py: multi-rank aggregation (gloo, world size 2) and
the oracle reference arm, without a GPU.

Requests are independent, so N ranks each decode their own batch (weak
scaling); the only collective is the max of the ranks' step times, and the
whole-job value counts every rank's bytes over that slowest time.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench
    import workloads as W

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = bench.shard_config(W.CONFIGS["gqa4_b32_u512to4096_ps16_nhd"], rank)
        t = W.make_tables(cfg)
        local_ms = 1.0 + rank  # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms)
        q.put((rank, cfg.seed, int(t.lengths.sum()), ms,
               bench.whole_job_gbs(1_000_000_000, world, ms)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_distinct_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    (r0, seed0, tok0, ms0, gbs0), (r1, seed1, tok1, ms1, gbs1) = res
    assert ms0 == ms1 == 2.0                  # max over ranks
    assert gbs0 == gbs1 == pytest.approx(2 * 1e9 / 2e-3 / 1e9)
    assert seed0 != seed1 and tok0 != tok1    # each rank decodes its own batch


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    r = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
         "--warmup", "1", "--ref-budget-s", "3", "--config", "gqa4_b32_u512to4096_ps16_nhd"],
        capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [line for line in r.stdout.splitlines() if line.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"] == "gqa4_b32_u512to4096_ps16_nhd"


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
         "--warmup", "1"], capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_counts_each_kv_head_once():
    # Every query head of a two-request batch sampled: the arm's GB/s must be the
    # metric's logical KV bytes per step over its time, although the G = 4 query
    # heads of a group each read their KV head's whole sequence.
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    r = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
         "--warmup", "1", "--batch", "2", "--ref-budget-s", "30", "--config",
         "gqa4_b32_u512to4096_ps16_nhd"],
        capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["cpu_baseline"]["sample"].startswith("64 of 64 ")
    kv = d["config"]["kv_bytes_per_step"]
    assert d["value"] == pytest.approx(kv / (d["ms_per_step"] * 1e-3) / 1e9, rel=1e-9)
    assert d["ms_per_step"] == pytest.approx(d["sample_ms_per_step"], rel=1e-9)


def test_reference_arm_reports_unique_bytes_and_a_whole_step_on_shared_prefixes():
    # Nine requests of the GQA8 workload: a group of eight sharing 1024 tokens
    # and one more. value counts each shared page once, logical_gbs every
    # request's pages; ms_per_step stands for the whole batch (here all heads
    # are sampled, so it equals the sample's time).
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    r = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
         "--warmup", "1", "--batch", "9", "--ref-budget-s", "60"],
        capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    c = d["config"]
    assert c["workload"] == "gqa8_b256_u128to16384_prefix1024x8_ps16_nhd"
    assert c["unique_kv_bytes_per_step"] < c["kv_bytes_per_step"]
    assert d["heads_sampled"] == d["heads_total"] == 9 * 64
    step_s = d["ms_per_step"] * 1e-3
    assert d["value"] == pytest.approx(c["unique_kv_bytes_per_step"] / step_s / 1e9, rel=1e-9)
    assert d["logical_gbs"] == pytest.approx(c["kv_bytes_per_step"] / step_s / 1e9, rel=1e-9)


def test_default_run_is_the_largest_workload_on_the_cascade_plan():
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W

    args = bench.parse_args([])
    cfg = W.CONFIGS[args.config]
    assert args.config == "gqa8_b256_u128to16384_prefix1024x8_ps16_nhd"
    assert max(W.CONFIGS.values(), key=lambda c: W.make_tables(c).lengths.sum()) is cfg
    assert bench.plan_kind_for(cfg, args.plan) == "cascade"
    assert bench.plan_kind_for(W.CONFIGS["gqa4_b32_u512to4096_ps16_nhd"], "auto") == "plain"
    assert bench.plan_kind_for(W.CONFIGS["mqa32_b16_l32768_ps64_nhd"], "cascade") == "plain"


def test_parity_report_flags_an_element_outside_the_bound():
    import numpy as np
    import torch

    sys.path.insert(0, ROOT)
    import bench

    rng = np.random.default_rng(1)
    ref = rng.standard_normal((3, 4, 128))
    ref_lse = rng.standard_normal((3, 4))
    out = torch.as_tensor(ref, dtype=torch.float32).to(torch.bfloat16)
    lse = torch.as_tensor(ref_lse, dtype=torch.float32)
    good = bench.parity_report(out, lse, ref, ref_lse)
    assert good["pass"] and good["heads_checked"] == 12 and good["max_rel_to_bound"] < 1.0
    bad = out.clone()
    bad[2, 3, 7] = float(ref[2, 3, 7]) + 0.05 + 0.02 * abs(float(ref[2, 3, 7]))
    assert not bench.parity_report(bad, lse, ref, ref_lse)["pass"]
    assert not bench.parity_report(out, lse + 2e-3, ref, ref_lse)["pass"]
