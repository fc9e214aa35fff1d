"""Pins of the f64 oracle against facts fixed outside the oracle itself.

The source pages print no numeric values for decode attention, so the oracle is
pinned by closed forms worked by hand (``tests/golden``), invariants of the
definition (one-token context, identical keys, page permutation, layout and
head-grouping consistency, split-and-merge), and brute-force dense attention on
tiny inputs written independently of the oracle's gather code. A plausible
slip in the oracle (a wrong head mapping, a dropped last-page mask, log2 for
ln, a missing sm_scale, a transposed pool index) fails at least one of them;
``test_oracle_mutants.py`` checks that claim by planting such slips.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def to_bits(x) -> np.ndarray:
    """float array -> bf16 bit patterns (round to nearest even)."""
    t = torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def run_case(oracle_mod, case: W.Case, **kw):
    return oracle_mod.paged_decode(
        W.bf16_bits(case.q), W.bf16_bits(case.k), W.bf16_bits(case.v), case.tables.indptr,
        case.tables.indices, case.tables.last_page_len, num_kv_heads=case.num_kv_heads,
        page_size=case.page_size, layout=0 if case.layout == "NHD" else 1,
        sm_scale=case.sm_scale, **kw)


def dense_kv(pool_bits, layout, indices_b, L, h):
    """Materialise K (or V) of one request and KV head as [L, D] float64.

    Written without the oracle's offset arithmetic: index whole pages out of
    the pool tensor, move the token axis next to the page axis, flatten.
    """
    pool = bits_to_f64(pool_bits)
    pages = pool[np.asarray(indices_b)]                 # [P, ps, Hkv, D] or [P, Hkv, ps, D]
    if layout == "HND":
        pages = pages.transpose(0, 2, 1, 3)             # -> [P, ps, Hkv, D]
    P, ps, Hkv, D = pages.shape
    return pages.reshape(P * ps, Hkv, D)[:L, h, :]


def brute_force(case: W.Case):
    """Dense two-pass softmax without max shift (small logits only)."""
    t = case.tables
    q = bits_to_f64(W.bf16_bits(case.q))
    kb, vb = W.bf16_bits(case.k), W.bf16_bits(case.v)
    G = case.group_size
    out = np.zeros((case.batch, case.num_qo_heads, case.head_dim))
    lse = np.zeros((case.batch, case.num_qo_heads))
    for b in range(case.batch):
        ind = t.indices[t.indptr[b]:t.indptr[b + 1]]
        L = int(t.lengths[b])
        for hq in range(case.num_qo_heads):
            K = dense_kv(kb, case.layout, ind, L, hq // G)
            V = dense_kv(vb, case.layout, ind, L, hq // G)
            e = np.exp(case.sm_scale * (K @ q[b, hq]))
            out[b, hq] = (e[:, None] * V).sum(0) / e.sum()
            lse[b, hq] = math.log(e.sum())
    return out, lse


# ---------------------------------------------------------------- worked examples

@pytest.mark.parametrize("fname", ["two_token_worked_example.json",
                                   "three_token_two_page_example.json"])
def test_golden_worked_examples(oracle_mod, fname):
    with open(os.path.join(GOLDEN, fname)) as f:
        g = json.load(f)
    scale = {"ln(3)": math.log(3.0), "ln(2)": math.log(2.0)}[g["sm_scale_expr"]]
    exp_lse = {"ln(4)": math.log(4.0), "ln(7)": math.log(7.0)}[g["expected_lse_expr"]]
    q, k, v = (to_bits(g[n]) for n in ("q", "k_pages", "v_pages"))
    assert np.array_equal(bits_to_f64(k), np.asarray(g["k_pages"], np.float64))  # exact in bf16
    out, lse = oracle_mod.paged_decode(
        q, k, v, g["indptr"], g["indices"], g["last_page_len"], num_kv_heads=g["Hkv"],
        page_size=g["page_size"], layout=0, sm_scale=scale)
    np.testing.assert_allclose(out, np.asarray(g["expected_out"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, [[exp_lse]], rtol=0, atol=1e-13)


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("G", [1, 4])
def test_one_token_context_returns_that_v(oracle_mod, layout, G):
    case = W.custom_case([1, 1, 1], num_qo_heads=4 * G, num_kv_heads=4, page_size=16,
                         layout=layout, seed=3)
    out, lse = run_case(oracle_mod, case)
    t = case.tables
    q = bits_to_f64(W.bf16_bits(case.q))
    for b in range(case.batch):
        page = int(t.indices[t.indptr[b]])
        for hq in range(case.num_qo_heads):
            h = hq // G
            if layout == "NHD":
                v0 = bits_to_f64(W.bf16_bits(case.v[page, 0, h]))
                k0 = bits_to_f64(W.bf16_bits(case.k[page, 0, h]))
            else:
                v0 = bits_to_f64(W.bf16_bits(case.v[page, h, 0]))
                k0 = bits_to_f64(W.bf16_bits(case.k[page, h, 0]))
            assert np.array_equal(out[b, hq], v0)          # exact: weight is exactly 1
            assert lse[b, hq] == pytest.approx(case.sm_scale * float(q[b, hq] @ k0), abs=1e-12)


def _fill_identical_keys(case, key_row):
    k = case.k
    if case.layout == "NHD":
        k[:] = key_row.view(1, 1, -1, case.head_dim)
    else:
        k[:] = key_row.view(1, -1, 1, case.head_dim)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_identical_keys_give_mean_of_v(oracle_mod, layout):
    lengths = [37, 16, 5]
    case = W.custom_case(lengths, num_qo_heads=8, num_kv_heads=2, page_size=16, layout=layout,
                         seed=5)
    key = torch.randn(case.num_kv_heads, case.head_dim).to(torch.bfloat16)
    _fill_identical_keys(case, key)
    out, lse = run_case(oracle_mod, case)
    t = case.tables
    q = bits_to_f64(W.bf16_bits(case.q))
    kk = bits_to_f64(W.bf16_bits(key))
    vb = W.bf16_bits(case.v)
    for b, L in enumerate(lengths):
        ind = t.indices[t.indptr[b]:t.indptr[b + 1]]
        for hq in range(case.num_qo_heads):
            h = hq // case.group_size
            V = dense_kv(vb, layout, ind, L, h)
            np.testing.assert_allclose(out[b, hq], V.mean(0), rtol=1e-13, atol=1e-13)
            s = case.sm_scale * float(q[b, hq] @ kk[h])
            assert lse[b, hq] == pytest.approx(s + math.log(L), abs=1e-12)


def test_zero_scale_gives_mean_of_v_and_log_length(oracle_mod):
    lengths = [40, 3]
    case = W.custom_case(lengths, num_qo_heads=4, num_kv_heads=4, page_size=8, seed=6,
                         sm_scale=0.0)
    out, lse = run_case(oracle_mod, case)
    t = case.tables
    vb = W.bf16_bits(case.v)
    for b, L in enumerate(lengths):
        ind = t.indices[t.indptr[b]:t.indptr[b + 1]]
        for hq in range(4):
            np.testing.assert_allclose(out[b, hq], dense_kv(vb, "NHD", ind, L, hq).mean(0),
                                       rtol=1e-13, atol=1e-13)
            assert lse[b, hq] == pytest.approx(math.log(L), abs=1e-13)


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("D", [4, 128])
@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("heads", [(2, 2), (4, 2), (3, 1)])
def test_matches_dense_brute_force(oracle_mod, D, layout, heads):
    Hq, Hkv = heads
    case = W.custom_case([1, 17, 40], num_qo_heads=Hq, num_kv_heads=Hkv, page_size=8,
                         layout=layout, head_dim=D, seed=7 + D, sigma=0.5)
    out, lse = run_case(oracle_mod, case)
    ref_out, ref_lse = brute_force(case)
    np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- invariants

def test_page_permutation_leaves_output_bitwise_unchanged(oracle_mod):
    case = W.custom_case([50, 33, 7, 16], num_qo_heads=8, num_kv_heads=2, page_size=16, seed=8)
    out0, lse0 = run_case(oracle_mod, case)
    rng = np.random.default_rng(9)
    perm = rng.permutation(case.tables.num_pages)        # new position of each page
    inv = np.argsort(perm)
    case.k = case.k[torch.as_tensor(inv)].contiguous()
    case.v = case.v[torch.as_tensor(inv)].contiguous()
    case.tables.indices = perm[case.tables.indices].astype(np.int32)
    out1, lse1 = run_case(oracle_mod, case)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def test_nhd_and_hnd_storage_of_one_cache_agree_bitwise(oracle_mod):
    case = W.custom_case([29, 64, 3], num_qo_heads=6, num_kv_heads=3, page_size=16, seed=10)
    out0, lse0 = run_case(oracle_mod, case)
    case.k = case.k.permute(0, 2, 1, 3).contiguous()
    case.v = case.v.permute(0, 2, 1, 3).contiguous()
    case.layout = "HND"
    out1, lse1 = run_case(oracle_mod, case)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def test_gqa_equals_mha_on_repeated_kv_heads(oracle_mod):
    G = 4
    case = W.custom_case([21, 48], num_qo_heads=8, num_kv_heads=2, page_size=16, seed=11)
    out_g, lse_g = run_case(oracle_mod, case)
    # Repeat each KV head G times consecutively: MHA head hq then reads KV head hq // G.
    mha = W.Case(case.batch, 8, 8, case.head_dim, case.page_size, "NHD", case.sm_scale,
                 case.tables, case.q, case.k.repeat_interleave(G, dim=2),
                 case.v.repeat_interleave(G, dim=2))
    out_m, lse_m = run_case(oracle_mod, mha)
    assert np.array_equal(out_g, out_m) and np.array_equal(lse_g, lse_m)


def test_unused_tail_slots_of_last_page_are_ignored(oracle_mod):
    case = W.custom_case([19, 5, 32], num_qo_heads=4, num_kv_heads=2, page_size=16, seed=12)
    out0, lse0 = run_case(oracle_mod, case)
    t = case.tables
    for b in range(case.batch):
        last_page = int(t.indices[t.indptr[b + 1] - 1])
        n = int(t.last_page_len[b])
        case.k[last_page, n:] = 3.0e4
        case.v[last_page, n:] = -3.0e4
    out1, lse1 = run_case(oracle_mod, case)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


def test_shared_pages_read_by_several_requests(oracle_mod):
    # Two requests whose block tables list the same physical pages attend over
    # the same tokens, so equal queries give equal results.
    case = W.custom_case([40, 40, 70], num_qo_heads=2, num_kv_heads=2, page_size=16, seed=13,
                         shared_prefix_tokens=48, share_group=3)
    t = case.tables
    assert t.shared_pages == 3
    assert np.array_equal(t.indices[0:3], t.indices[3:6])
    case.q[1] = case.q[0]
    out, lse = run_case(oracle_mod, case)
    assert np.array_equal(out[0], out[1]) and np.array_equal(lse[0], lse[1])


def test_thread_count_does_not_change_result(oracle_mod):
    case = W.custom_case([100, 3, 77, 16, 1], num_qo_heads=8, num_kv_heads=4, page_size=16,
                         seed=14)
    out1, lse1 = run_case(oracle_mod, case, nthreads=1)
    out8, lse8 = run_case(oracle_mod, case, nthreads=7)
    assert np.array_equal(out1, out8) and np.array_equal(lse1, lse8)


def test_head_subset_matches_full_run(oracle_mod):
    case = W.custom_case([30, 70], num_qo_heads=8, num_kv_heads=2, page_size=16, seed=15)
    out, lse = run_case(oracle_mod, case)
    heads = [(1, 7), (0, 0), (1, 2)]
    o2, l2 = run_case(oracle_mod, case, heads=heads)
    for i, (b, hq) in enumerate(heads):
        assert np.array_equal(o2[i], out[b, hq]) and l2[i] == lse[b, hq]


# ---------------------------------------------------------------- split-K and merge

def test_split_states_merge_to_unsplit(oracle_mod):
    case = W.custom_case([97, 300], num_qo_heads=4, num_kv_heads=1, page_size=16, seed=16)
    out, lse = run_case(oracle_mod, case)
    rng = np.random.default_rng(17)
    args = (W.bf16_bits(case.q), W.bf16_bits(case.k), W.bf16_bits(case.v), case.tables.indptr,
            case.tables.indices, case.tables.last_page_len)
    for b, L in enumerate(case.tables.lengths):
        for hq in range(4):
            cuts = np.sort(rng.choice(np.arange(1, L), size=min(5, L - 1), replace=False))
            edges = [0, *cuts.tolist(), int(L)]
            vs, ss = [], []
            for a, e in zip(edges[:-1], edges[1:]):
                o, s = oracle_mod.partial_state(*args, num_kv_heads=1, page_size=16, layout=0,
                                                sm_scale=case.sm_scale, b=b, hq=hq,
                                                tok_begin=a, tok_end=e)
                vs.append(o)
                ss.append(s)
            mo, ml = oracle_mod.merge_states(np.stack(vs), np.asarray(ss))
            np.testing.assert_allclose(mo, out[b, hq], rtol=1e-12, atol=1e-13)
            assert ml == pytest.approx(lse[b, hq], rel=1e-12, abs=1e-12)


def test_merge_closed_forms(oracle_mod):
    rng = np.random.default_rng(18)
    v = rng.normal(size=(3, 8))
    # single state: identity
    o, s = oracle_mod.merge_states(v[:1], np.array([0.7]))
    assert np.array_equal(o, v[0]) and s == pytest.approx(0.7, abs=1e-15)
    # equal LSEs: plain average, lse + ln S
    o, s = oracle_mod.merge_states(v, np.full(3, -2.0))
    np.testing.assert_allclose(o, v.mean(0), rtol=1e-14, atol=1e-15)
    assert s == pytest.approx(-2.0 + math.log(3.0), abs=1e-14)
    # weights e^s: lse ln 1 and ln 3 -> 1/4, 3/4
    o, s = oracle_mod.merge_states(v[:2], np.log([1.0, 3.0]))
    np.testing.assert_allclose(o, 0.25 * v[0] + 0.75 * v[1], rtol=1e-14, atol=1e-15)
    assert s == pytest.approx(math.log(4.0), abs=1e-14)
    # -inf states carry no weight; all -inf gives zeros and -inf
    o, s = oracle_mod.merge_states(v, np.array([-np.inf, 1.0, -np.inf]))
    assert np.array_equal(o, v[1]) and s == 1.0
    o, s = oracle_mod.merge_states(v, np.full(3, -np.inf))
    assert np.array_equal(o, np.zeros(8)) and s == -np.inf


def test_empty_partial_range_is_neutral(oracle_mod):
    case = W.custom_case([10], num_qo_heads=1, num_kv_heads=1, page_size=16, seed=19)
    o, s = oracle_mod.partial_state(
        W.bf16_bits(case.q), W.bf16_bits(case.k), W.bf16_bits(case.v), case.tables.indptr,
        case.tables.indices, case.tables.last_page_len, num_kv_heads=1, page_size=16,
        layout=0, sm_scale=1.0, b=0, hq=0, tok_begin=4, tok_end=4)
    assert s == -np.inf and not o.any()


# ---------------------------------------------------------------- rejection

@pytest.mark.parametrize("mutation", ["page_oob", "negative_page", "last_zero", "last_big",
                                      "empty_request"])
def test_invalid_block_tables_are_rejected(oracle_mod, mutation):
    case = W.custom_case([20, 9], num_qo_heads=2, num_kv_heads=1, page_size=16, seed=20)
    t = case.tables
    ind, ptr, last = t.indices.copy(), t.indptr.copy(), t.last_page_len.copy()
    if mutation == "page_oob":
        ind[1] = t.num_pages
    elif mutation == "negative_page":
        ind[0] = -1
    elif mutation == "last_zero":
        last[0] = 0
    elif mutation == "last_big":
        last[1] = 17
    elif mutation == "empty_request":
        ptr = np.array([0, 0, len(ind)], np.int32)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.paged_decode(W.bf16_bits(case.q), W.bf16_bits(case.k), W.bf16_bits(case.v),
                                ptr, ind, last, num_kv_heads=1, page_size=16, layout=0,
                                sm_scale=1.0)
