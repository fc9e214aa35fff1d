"""Randomised decode cases against the f64 oracle, every head of every request.

A hundred seeded draws over the whole descriptor space the decode accepts: group
sizes 1..32 (every kernel variant and both tensor paths for wide groups),
page sizes 8..64, NHD and HND, batches of 1..24 requests whose lengths mix
one-token, one-page, page-aligned and long requests, unused pool pages, scales
other than 1/sqrt(D), value spreads, split settings (planner's choice, forced
splits, a cap, never split), with and without LSE, on bound and unbound
workspaces. Each case is small enough for the oracle to check in well under a
second.
"""
import os

import numpy as np
import pytest
import torch

import paged_kv_decode_attn_gb300 as oxd
import workloads as W
from gpu_helpers import DeviceTables, assert_parity, oracle_ref, plan_case

pytestmark = pytest.mark.gpu

# OXD_FUZZ_SCALE=k draws k times as many cases (new seeds after the first 100).
N_CASES = 100 * int(os.environ.get("OXD_FUZZ_SCALE", "1"))


@pytest.fixture(scope="module", autouse=True)
def setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oxd.build()


def draw(i):
    rng = np.random.default_rng(9000 + i)
    G = int(rng.choice([1, 2, 3, 4, 5, 8, 12, 16, 17, 24, 32]))
    Hkv = int(rng.choice([1, 2, 4, 8])) if G <= 16 else int(rng.choice([1, 2]))
    ps = int(rng.choice([8, 16, 32, 64]))
    layout = str(rng.choice(["NHD", "HND"]))
    B = int(rng.integers(1, 25))
    kinds = rng.integers(0, 5, size=B)
    lengths = []
    for kd in kinds:
        if kd == 0:
            lengths.append(1)                               # a one-token context
        elif kd == 1:
            lengths.append(int(rng.integers(1, ps + 1)))     # within one page
        elif kd == 2:
            lengths.append(ps * int(rng.integers(1, 40)))    # a full last page
        else:
            lengths.append(int(rng.integers(1, 3000)))
    splits = rng.integers(0, 4)
    kw = {}
    if splits == 1:
        kw["force_splits"] = int(rng.integers(2, 12))
    elif splits == 2:
        kw["max_splits"] = int(rng.integers(1, 6))
    if G > 16:
        kw["tensor_path"] = int(rng.integers(0, 2))
    case = W.custom_case(lengths, num_qo_heads=G * Hkv, num_kv_heads=Hkv, page_size=ps,
                         layout=layout, seed=9100 + i, sigma=float(rng.choice([0.5, 1.0, 2.0])),
                         device="cuda", sm_scale=float(rng.choice([0.05, 0.0884, 0.2])),
                         extra_pages=int(rng.integers(0, 4)))
    want_lse = bool(rng.integers(0, 4) > 0)
    bind = bool(rng.integers(0, 2))
    return case, kw, want_lse, bind


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case_matches_oracle(i):
    case, kw, want_lse, bind = draw(i)
    plan = plan_case(case, **kw)
    tables = DeviceTables(case)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    if bind:
        oxd.oxd_plan_bind_workspace(plan, ws)
    out = torch.empty_like(case.q)
    lse = (torch.empty(case.batch, case.num_qo_heads, dtype=torch.float32, device="cuda")
           if want_lse else None)
    oxd.oxd_paged_decode_run(plan, case.q, case.k, case.v, tables.indptr, tables.indices,
                             tables.last, case.sm_scale, out, lse, ws, plan.workspace_bytes)
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
    ref_out, ref_lse = oracle_ref(case)
    what = (f"case {i}: G={case.num_qo_heads // case.num_kv_heads} Hkv={case.num_kv_heads} "
            f"ps={case.page_size} {case.layout} B={case.batch} {kw} lse={want_lse} bind={bind}")
    assert_parity(out, ref_out, lse, ref_lse if want_lse else None, what)
