"""Fused RoPE + paged KV append through the C ABI against the f64 oracle.

Each token's query heads are rotated into q_out and its K (rotated) and V
rows land in its page slot. The GPU rotates in float with the angle carried
as a two-float number of turns; the oracle rotates in f64. Both round once
to bf16, so K and q_out agree bit for bit except where the exact value sits
next to a rounding boundary. The bound applied to every element: within one
bf16 step of the oracle, or within the oracle's bf16 step plus 2^-20 of the
rotated pair's norm, the float arithmetic's own error (about 2.5e-7 of the
norm) with a margin of four, which matters where a rotated value sits near
zero; and at least 99 % of the elements bitwise equal.
V rows are copies and every other pool byte is untouched: both bitwise.
Tokens aimed at shared pages (reference count not one), past the request's
pages or at out-of-pool pages write nothing and set the status word; a
decode after an append attends to the appended tokens.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_attn_gb300 as oxd
import workloads as W
from gpu_helpers import DeviceTables, assert_parity, oracle_ref, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oxd.build()
    oracle.build()


def _ordered(bits):
    """bf16 bit patterns mapped to integers in the order of their values."""
    b = np.asarray(bits, np.uint16).astype(np.int32)
    return np.where(b & 0x8000, 0x8000 - b, b + 0x8000)


def _f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _ulp_close(gpu_bits, ref_bits, what):
    """Within one bf16 step of the oracle, or, where the rotated value sits
    near zero, within the float arithmetic's own error: the angle is good to
    about 2^-25 turns (2e-7 rad) and the products round at 2^-24, so the
    float result is off by at most about 2.5e-7 times the pair's norm
    sqrt(y_i^2 + y_(i+64)^2) (a rotation keeps it, so it is read off the
    oracle's output); 2^-20 of it leaves a margin of four."""
    g, r = np.asarray(gpu_bits), np.asarray(ref_bits)
    d = np.abs(_ordered(g) - _ordered(r))
    rv = _f32(r)
    norm = np.sqrt(rv[..., :64] ** 2 + rv[..., 64:] ** 2)
    norm = np.concatenate([norm, norm], axis=-1)
    step = np.abs(_f32(r) - _f32(r ^ 1)).clip(min=0)  # bf16 step at the oracle's value
    ok = (d <= 1) | (np.abs(_f32(g) - rv) <= step + 2.0 ** -20 * norm)
    assert ok.all(), (f"{what}: {int((~ok).sum())} elements off, worst {int(d[~ok].max())} "
                      f"bf16 steps")
    assert (d == 0).mean() >= 0.99, f"{what}: only {(d == 0).mean():.4f} exact"


def _bits(t):
    return W.bf16_bits(t)


def _grown_case(lengths, add, G, Hkv, ps, layout, seed, extra_pages=4):
    """A case whose block tables already cover `add` more tokens per request."""
    grown = [L + a for L, a in zip(lengths, add)]
    case = W.custom_case(grown, num_qo_heads=G * Hkv, num_kv_heads=Hkv, page_size=ps,
                         layout=layout, seed=seed, device="cuda", extra_pages=extra_pages)
    return case


def _append_inputs(lengths, add, Hq, Hkv, seed):
    tok_req, pos = [], []
    for b, (L, a) in enumerate(zip(lengths, add)):
        for i in range(a):
            tok_req.append(b)
            pos.append(L + i)
    T = len(pos)
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn(T, Hq, 128, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(T, Hkv, 128, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(T, Hkv, 128, generator=g, device="cuda").to(torch.bfloat16)
    return (q, k, v, torch.tensor(tok_req, dtype=torch.int32, device="cuda"),
            torch.tensor(pos, dtype=torch.int32, device="cuda"))


def _run_append(case, q, k, v, tr, pos, refcount, q_out=None, theta=10000.0):
    t = case.tables
    desc = oxd.make_rope_append_desc(q.shape[0], case.batch, case.num_qo_heads,
                                     case.num_kv_heads, case.page_size, case.layout,
                                     t.num_pages, int(t.indptr[-1]), rope_theta=theta)
    tables = DeviceTables(case)
    if q_out is None:
        q_out = torch.empty_like(q)
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    oxd.oxd_rope_append(desc, q, k, v, tr, pos, tables.indptr, tables.indices, refcount, q_out,
                        case.k, case.v, ws)
    torch.cuda.synchronize()
    return q_out, oxd.oxd_read_device_status(ws)


def _oracle_append(case, k_before, v_before, q, k, v, tr, pos, refcount, theta=10000.0):
    t = case.tables
    return oracle.rope_append(_bits(q), _bits(k), _bits(v), tr.cpu().numpy(), pos.cpu().numpy(),
                              t.indptr, t.indices, refcount.cpu().numpy(), k_before, v_before,
                              page_size=case.page_size,
                              layout=0 if case.layout == "NHD" else 1, theta=theta)


@pytest.mark.parametrize("layout,ps", [("NHD", 16), ("HND", 16), ("NHD", 64), ("HND", 8)])
@pytest.mark.parametrize("G", [1, 4, 32])
def test_append_matches_oracle(G, layout, ps):
    Hkv = 8 if G < 32 else 1
    lengths = [1, 15, 16, 100, 333, 64]
    add = [1, 1, 3, 1, 2, 64]          # up to 64 tokens of one request in one call
    case = _grown_case(lengths, add, G, Hkv, ps, layout, seed=31 + G + ps)
    k_before, v_before = _bits(case.k), _bits(case.v)
    q, k, v, tr, pos = _append_inputs(lengths, add, G * Hkv, Hkv, seed=5)
    # scramble the token order: any order is allowed
    perm = torch.randperm(q.shape[0], generator=torch.Generator().manual_seed(3)).cuda()
    q, k, v, tr, pos = q[perm], k[perm], v[perm], tr[perm], pos[perm]
    refcount = torch.ones(case.tables.num_pages, dtype=torch.int32, device="cuda")
    q_out, status = _run_append(case, q, k, v, tr, pos, refcount)
    assert status == oxd.OXD_DEVICE_OK
    rq, rk, rv, rst = _oracle_append(case, k_before, v_before, q, k, v, tr, pos, refcount)
    assert (rst == 0).all()
    _ulp_close(_bits(q_out), rq, "q_out")
    _ulp_close(_bits(case.k), rk, "K pool")
    assert np.array_equal(_bits(case.v), rv), "V pool"


@pytest.mark.parametrize("G,Hkv", [(2, 10), (3, 3), (5, 16), (1, 17)])
def test_head_counts_across_warp_chunks(G, Hkv):
    # a warp takes up to eight heads of one token: head counts that are not
    # multiples of eight, and more than eight KV heads, split a token's rows
    lengths, add = [5, 70, 31], [2, 1, 33]
    case = _grown_case(lengths, add, G, Hkv, 16, "HND" if Hkv % 2 else "NHD", seed=50 + Hkv)
    k_before, v_before = _bits(case.k), _bits(case.v)
    q, k, v, tr, pos = _append_inputs(lengths, add, G * Hkv, Hkv, seed=9)
    refcount = torch.ones(case.tables.num_pages, dtype=torch.int32, device="cuda")
    q_out, status = _run_append(case, q, k, v, tr, pos, refcount)
    assert status == oxd.OXD_DEVICE_OK
    rq, rk, rv, rst = _oracle_append(case, k_before, v_before, q, k, v, tr, pos, refcount)
    assert (rst == 0).all()
    _ulp_close(_bits(q_out), rq, "q_out")
    _ulp_close(_bits(case.k), rk, "K pool")
    assert np.array_equal(_bits(case.v), rv), "V pool"


@pytest.mark.parametrize("B", [1000, 4200])
def test_batches_of_thousands_of_requests(B):
    # One new token for each of B requests of 1..40 cached tokens, in
    # shuffled order: every token's walk through a large indptr.
    rng = np.random.default_rng(B)
    lengths = [int(x) for x in rng.integers(1, 41, size=B)]
    add = [1] * B
    case = _grown_case(lengths, add, 4, 2, 16, "NHD", seed=B)
    k_before, v_before = _bits(case.k), _bits(case.v)
    q, k, v, tr, pos = _append_inputs(lengths, add, 8, 2, seed=B + 1)
    perm = torch.randperm(q.shape[0], generator=torch.Generator().manual_seed(B)).cuda()
    q, k, v, tr, pos = q[perm], k[perm], v[perm], tr[perm], pos[perm]
    refcount = torch.ones(case.tables.num_pages, dtype=torch.int32, device="cuda")
    q_out, status = _run_append(case, q, k, v, tr, pos, refcount)
    assert status == oxd.OXD_DEVICE_OK
    rq, rk, rv, rst = _oracle_append(case, k_before, v_before, q, k, v, tr, pos, refcount)
    assert (rst == 0).all()
    _ulp_close(_bits(q_out), rq, "q_out")
    _ulp_close(_bits(case.k), rk, "K pool")
    assert np.array_equal(_bits(case.v), rv), "V pool"


def test_positions_up_to_the_limit():
    # tokens at positions near 2^24 - 1: the angle must stay accurate there
    ps = 64
    big = (1 << 24) - 3
    pages = big // ps + 2
    # one request whose logical page j is physical page j % 4 (the four
    # tokens below land in distinct slots), so the pool stays small
    n_phys = 4
    indptr = np.array([0, pages], np.int32)
    indices = (np.arange(pages) % n_phys).astype(np.int32)
    last = np.array([ps], np.int32)
    tables = W.BlockTables(lengths=np.array([pages * ps]), indptr=indptr, indices=indices,
                           last_page_len=last, num_pages=n_phys, page_size=ps)
    Hkv, Hq = 1, 2
    k_pool = torch.zeros(n_phys, ps, Hkv, 128, dtype=torch.bfloat16, device="cuda")
    v_pool = torch.zeros_like(k_pool)
    case = W.Case(1, Hq, Hkv, 128, ps, "NHD", 1.0, tables, None, k_pool, v_pool)
    pos = torch.tensor([big, big - 1, 12345678, 3], dtype=torch.int32, device="cuda")
    tr = torch.zeros(4, dtype=torch.int32, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(4)
    q = torch.randn(4, Hq, 128, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(4, Hkv, 128, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(4, Hkv, 128, generator=g, device="cuda").to(torch.bfloat16)
    k_before, v_before = _bits(k_pool), _bits(v_pool)
    refcount = torch.ones(n_phys, dtype=torch.int32, device="cuda")
    q_out, status = _run_append(case, q, k, v, tr, pos, refcount)
    assert status == oxd.OXD_DEVICE_OK
    rq, rk, rv, rst = _oracle_append(case, k_before, v_before, q, k, v, tr, pos, refcount)
    assert (rst == 0).all()
    _ulp_close(_bits(q_out), rq, "q_out at large positions")
    _ulp_close(_bits(k_pool), rk, "K at large positions")


def test_positions_outside_the_limit_are_refused():
    # positions of 2^24 or more, or negative, write no K/V row even where the
    # block table covers them; their q_out rows are rotated at p & (2^24 - 1)
    ps, n_phys = 64, 4
    pages = (1 << 24) // ps + 4
    indptr = np.array([0, pages], np.int32)
    indices = (np.arange(pages) % n_phys).astype(np.int32)
    tables = W.BlockTables(lengths=np.array([pages * ps]), indptr=indptr, indices=indices,
                           last_page_len=np.array([ps], np.int32), num_pages=n_phys, page_size=ps)
    Hkv, Hq = 2, 4
    g = torch.Generator(device="cuda").manual_seed(14)
    k_pool = torch.randn(n_phys, Hkv, ps, 128, generator=g, device="cuda").to(torch.bfloat16)
    v_pool = torch.randn(n_phys, Hkv, ps, 128, generator=g, device="cuda").to(torch.bfloat16)
    case = W.Case(1, Hq, Hkv, 128, ps, "HND", 1.0, tables, None, k_pool, v_pool)
    pos = torch.tensor([1 << 24, (1 << 24) + 70, -1, -5], dtype=torch.int32, device="cuda")
    tr = torch.zeros(4, dtype=torch.int32, device="cuda")
    q = torch.randn(4, Hq, 128, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(4, Hkv, 128, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(4, Hkv, 128, generator=g, device="cuda").to(torch.bfloat16)
    k_before, v_before = _bits(k_pool), _bits(v_pool)
    refcount = torch.ones(n_phys, dtype=torch.int32, device="cuda")
    q_out, status = _run_append(case, q, k, v, tr, pos, refcount)
    assert status == oxd.OXD_DEVICE_BAD_POSITION
    assert np.array_equal(_bits(k_pool), k_before) and np.array_equal(_bits(v_pool), v_before)
    masked = pos & ((1 << 24) - 1)
    rq, _, _, _ = _oracle_append(case, k_before, v_before, q, k, v, tr, masked, refcount)
    _ulp_close(_bits(q_out), rq, "q_out at masked positions")


def test_shared_pages_and_bad_positions_are_not_written():
    lengths = [30, 50, 7]
    add = [2, 1, 1]
    case = _grown_case(lengths, add, 4, 8, 16, "NHD", seed=9)
    k_before, v_before = _bits(case.k), _bits(case.v)
    q, k, v, tr, pos = _append_inputs(lengths, add, 32, 8, seed=6)
    # token 2 (request 1) goes past its pages; request 0's target page is shared
    pos[2] = int(case.tables.indptr[2] - case.tables.indptr[1]) * 16
    t = case.tables
    page0 = int(t.indices[t.indptr[0] + lengths[0] // 16])
    refcount = torch.ones(t.num_pages, dtype=torch.int32, device="cuda")
    refcount[page0] = 2
    q_out, status = _run_append(case, q, k, v, tr, pos, refcount)
    assert status in (oxd.OXD_DEVICE_SHARED_PAGE, oxd.OXD_DEVICE_BAD_POSITION)
    rq, rk, rv, rst = _oracle_append(case, k_before, v_before, q, k, v, tr, pos, refcount)
    assert list(rst) == [1, 1, 2, 0]
    _ulp_close(_bits(q_out), rq, "q_out")       # every q row is still written
    _ulp_close(_bits(case.k), rk, "K pool")
    assert np.array_equal(_bits(case.v), rv)
    # only the third token differs from the untouched pools at all
    assert np.array_equal(_bits(case.k)[page0], k_before[page0])


def test_in_place_query_rotation():
    lengths, add = [10, 40], [1, 1]
    case = _grown_case(lengths, add, 4, 8, 16, "HND", seed=12)
    k_before, v_before = _bits(case.k), _bits(case.v)
    q, k, v, tr, pos = _append_inputs(lengths, add, 32, 8, seed=7)
    q0 = q.clone()
    refcount = torch.ones(case.tables.num_pages, dtype=torch.int32, device="cuda")
    _, status = _run_append(case, q, k, v, tr, pos, refcount, q_out=q)
    assert status == oxd.OXD_DEVICE_OK
    rq, _, _, _ = _oracle_append(case, k_before, v_before, q0, k, v, tr, pos, refcount)
    _ulp_close(_bits(q), rq, "q rotated in place")


def test_decode_after_append_sees_the_new_tokens():
    # grow every request by one token through the append, then decode with
    # the longer tables: the result matches the oracle on the grown cache
    lengths = [100, 257, 16, 1]
    add = [1, 1, 1, 1]
    case = _grown_case(lengths, add, 4, 2, 16, "NHD", seed=13)
    k_before, v_before = _bits(case.k), _bits(case.v)
    q, k, v, tr, pos = _append_inputs(lengths, add, 8, 2, seed=8)
    refcount = torch.ones(case.tables.num_pages, dtype=torch.int32, device="cuda")
    q_rot, status = _run_append(case, q, k, v, tr, pos, refcount)
    assert status == oxd.OXD_DEVICE_OK
    case.q.copy_(q_rot)  # one new token per request, in request order
    # the oracle's inputs are the oracle's own append of the same tokens to
    # host copies of the pools taken before the GPU append
    rq, rk, rv, st = _oracle_append(case, k_before, v_before, q, k, v, tr, pos, refcount)
    assert (st == oracle.APPEND_WRITTEN).all()
    t = case.tables
    ref_out, ref_lse = oracle.paged_decode(rq, rk, rv, t.indptr, t.indices, t.last_page_len,
                                           num_kv_heads=2, page_size=16, layout=0,
                                           sm_scale=case.sm_scale)
    out, lse, _, _ = run_decode(case)
    assert_parity(out, ref_out, lse, ref_lse, "decode after append")
