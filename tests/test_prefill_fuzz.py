"""Randomised paged causal prefill cases against the f64 oracle, every row.

Sixty seeded draws: both tile sizes (256 rows on the two-half kernel, 128 on
the narrow one, or the planner's pick), group sizes 1..128 (tiles of 256 down to
one query token, and tiles that leave rows idle), page sizes 8..64, NHD and HND, one to four
requests whose query counts run from zero to the whole cache, split settings
(planner's choice, never split, a cap), bound and unbound workspaces, and
scales other than 1/sqrt(D). Each case is small enough for the oracle to
check every output row in well under a second.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_attn_gb300 as oxd
import workloads as W
from gpu_helpers import assert_parity
from test_prefill import Prefill, oracle_rows

pytestmark = pytest.mark.gpu

# OXD_FUZZ_SCALE=k draws k times as many cases (new seeds after the first 60).
N_CASES = 60 * int(os.environ.get("OXD_FUZZ_SCALE", "1"))


@pytest.fixture(scope="module", autouse=True)
def setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oxd.build()
    oracle.build()


def draw(i):
    rng = np.random.default_rng(7000 + i)
    G = int(rng.choice([1, 2, 3, 4, 5, 8, 16, 32, 64, 128]))
    Hkv = int(rng.choice([1, 2, 4])) if G <= 32 else 1
    ps = int(rng.choice([8, 16, 32, 64]))
    layout = str(rng.choice(["NHD", "HND"]))
    B = int(rng.integers(1, 5))
    kv = [int(rng.integers(1, 600)) for _ in range(B)]
    q = []
    for L in kv:
        kind = rng.integers(0, 4)
        q.append(0 if kind == 0 else min(L, 200) if kind == 1
                 else int(rng.integers(1, min(L, 200) + 1)))
    if sum(q) == 0:
        q[0] = 1
    max_splits = int(rng.choice([0, 0, 1, 3]))
    bind = bool(rng.integers(0, 2))
    case = W.prefill_case(tuple(q), tuple(kv), G * Hkv, Hkv, ps, layout, seed=7100 + i,
                          device="cuda", sm_scale=float(rng.choice([0.05, 0.0884, 0.15])))
    tile_rows = int(rng.choice([0, 128, 256]))
    return case, max_splits, bind, tile_rows


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_prefill_matches_oracle(i):
    case, max_splits, bind, tile_rows = draw(i)
    run = Prefill(case, max_splits=max_splits, bind=bind, tile_rows=tile_rows)
    run.run()
    torch.cuda.synchronize()
    assert run.status() == oxd.OXD_DEVICE_OK
    ref_o, ref_l = oracle_rows(case)
    what = (f"case {i}: G={case.num_qo_heads // case.num_kv_heads} Hkv={case.num_kv_heads} "
            f"ps={case.page_size} {case.layout} q={tuple(case.qo_indptr[1:] - case.qo_indptr[:-1])} "
            f"max_splits={max_splits} bind={bind} tile_rows={run.plan.info.tile_rows}")
    assert_parity(run.out, ref_o, run.lse, ref_l, what)
