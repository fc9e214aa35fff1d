"""Randomised fused RoPE + paged append cases against the f64 oracle.

Forty seeded draws: group sizes 1..32 and KV head counts 1..16 (head counts
that split a token's rows across warps included), page sizes 8..64, NHD and
HND, four to twelve requests appending two to 64 tokens each in shuffled order,
rotary bases other than 10^4, and pools with shared pages (reference count
above one) that must stay untouched. q_out and the K pool agree with the oracle
to one bf16 step (almost all exact), V and every byte not written bitwise, and
the device status is the oracle's.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_attn_gb300 as oxd
from test_rope_append import (_append_inputs, _bits, _grown_case, _oracle_append, _run_append,
                              _ulp_close)

pytestmark = pytest.mark.gpu

# OXD_FUZZ_SCALE=k draws k times as many cases (new seeds after the first 40).
N_CASES = 40 * int(os.environ.get("OXD_FUZZ_SCALE", "1"))


@pytest.fixture(scope="module", autouse=True)
def setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oxd.build()
    oracle.build()


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_append_matches_oracle(i):
    rng = np.random.default_rng(5000 + i)
    G = int(rng.choice([1, 2, 3, 4, 8, 32]))
    Hkv = int(rng.choice([1, 2, 5, 8, 16])) if G < 32 else 1
    ps = int(rng.choice([8, 16, 32, 64]))
    layout = str(rng.choice(["NHD", "HND"]))
    B = int(rng.integers(4, 13))
    lengths = [int(x) for x in rng.integers(0, 400, B)]
    add = [int(x) for x in rng.integers(2, 65 if B <= 5 else 9, B)]
    theta = float(rng.choice([10000.0, 500000.0, 1000.0]))
    case = _grown_case(lengths, add, G, Hkv, ps, layout, seed=5100 + i)
    k_before, v_before = _bits(case.k), _bits(case.v)
    q, k, v, tr, pos = _append_inputs(lengths, add, G * Hkv, Hkv, seed=5200 + i)
    perm = torch.randperm(q.shape[0], generator=torch.Generator().manual_seed(i)).cuda()
    q, k, v, tr, pos = q[perm], k[perm], v[perm], tr[perm], pos[perm]
    refcount = torch.ones(case.tables.num_pages, dtype=torch.int32, device="cuda")
    if rng.integers(0, 2):
        # some pages shared: tokens aimed at them write nothing and are reported
        shared = rng.choice(case.tables.num_pages, size=max(1, case.tables.num_pages // 8),
                            replace=False)
        refcount[torch.as_tensor(shared, device="cuda")] = 2
    q_out, status = _run_append(case, q, k, v, tr, pos, refcount, theta=theta)
    rq, rk, rv, rst = _oracle_append(case, k_before, v_before, q, k, v, tr, pos, refcount,
                                     theta=theta)
    what = f"case {i}: G={G} Hkv={Hkv} ps={ps} {layout} B={B} theta={theta}"
    if (rst == 0).all():
        assert status == oxd.OXD_DEVICE_OK, what
    else:
        assert status == oxd.OXD_DEVICE_SHARED_PAGE, what
    _ulp_close(_bits(q_out), rq, what + " q_out")
    _ulp_close(_bits(case.k), rk, what + " K pool")
    assert np.array_equal(_bits(case.v), rv), what + " V pool"
