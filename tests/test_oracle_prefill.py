"""Pins of the oracle's paged causal prefill (CPU only).

What pins it, other than its own formula:
  * a closed form worked by hand (tests/golden/causal_prefill_worked_example.json):
    the query tokens sit at the end of the cache and see nothing past their
    own position;
  * dense causal attention on tiny inputs, written here with plain indexing of
    whole pages and an explicit mask (no page arithmetic from the oracle);
  * reductions to the independently pinned decode oracle: with one query token
    per request prefill is decode, and the last query token of any request
    sees the whole cache, so both agree bit for bit;
  * causality: changing K/V past a row's position leaves that row unchanged;
  * identical keys: the output is the mean of the visible V rows and
    lse = s + ln(position + 1);
  * a row subset and any thread count give the same bits as the full run;
  * planted mistakes (causal off by one, top-left alignment, the query row of
    the wrong request, modulo head mapping, the owner search off by one, a
    dropped sm_scale) each fail this battery.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "oxd_oracle.c")
GOLDEN = os.path.join(HERE, "golden", "causal_prefill_worked_example.json")


def _bits(x):
    t = torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _layout(case):
    return 0 if case.layout == "NHD" else 1


def _prefill(lib, case, **kw):
    t = case.tables
    return oracle.paged_prefill(W.bf16_bits(case.q), W.bf16_bits(case.k), W.bf16_bits(case.v),
                                case.qo_indptr, t.indptr, t.indices, t.last_page_len,
                                num_kv_heads=case.num_kv_heads, page_size=case.page_size,
                                layout=_layout(case), sm_scale=case.sm_scale, lib=lib, **kw)


def _dense(pool_bits, layout, idx, L, h):
    """[L, D] of one request and KV head: whole pages picked out of the pool,
    the token axis moved next to the page axis, flattened."""
    pages = _f64(pool_bits)[np.asarray(idx)]
    if layout == "HND":
        pages = pages.transpose(0, 2, 1, 3)
    P, ps, H, D = pages.shape
    return pages.reshape(P * ps, H, D)[:L, h, :]


def _brute(case):
    """Dense causal attention with an explicit lower-triangular mask."""
    t = case.tables
    q = _f64(W.bf16_bits(case.q))
    kb, vb = W.bf16_bits(case.k), W.bf16_bits(case.v)
    G = case.group_size
    out = np.zeros(q.shape)
    lse = np.zeros(q.shape[:2])
    for b in range(case.batch):
        idx = t.indices[t.indptr[b]:t.indptr[b + 1]]
        L = int(t.lengths[b])
        q0, q1 = int(case.qo_indptr[b]), int(case.qo_indptr[b + 1])
        n = q1 - q0
        # row i of the block may see columns 0 .. L - n + i
        mask = np.arange(L)[None, :] <= (L - n + np.arange(n))[:, None]
        for hq in range(case.num_qo_heads):
            K = _dense(kb, case.layout, idx, L, hq // G)
            V = _dense(vb, case.layout, idx, L, hq // G)
            s = case.sm_scale * (q[q0:q1, hq] @ K.T)
            s = np.where(mask, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            e = np.exp(s - m)
            out[q0:q1, hq] = (e @ V) / e.sum(axis=1, keepdims=True)
            lse[q0:q1, hq] = m[:, 0] + np.log(e.sum(axis=1))
    return out, lse


def _small(q_lens, kv_lens, Hq, Hkv, ps, layout, D, seed):
    return W.prefill_case(q_lens, kv_lens, Hq, Hkv, ps, layout, head_dim=D, seed=seed,
                          sm_scale=0.3)


# ------------------------------------------------------------------ the pin battery

def prefill_pins(lib):
    bad = []

    # closed form worked by hand
    g = json.load(open(GOLDEN))
    out, lse = oracle.paged_prefill(
        _bits(g["q"]), _bits(g["k_pages"]), _bits(g["v_pages"]), g["qo_indptr"], g["indptr"],
        g["indices"], g["last_page_len"], num_kv_heads=g["Hkv"], page_size=g["page_size"],
        layout=0, sm_scale=math.log(3.0), lib=lib)
    want_lse = [math.log(4.0), math.log(11.0)]
    if not (np.allclose(out, np.asarray(g["expected_out"]), rtol=0, atol=1e-12)
            and np.allclose(lse[:, 0], want_lse, rtol=0, atol=1e-12)):
        bad.append(f"worked example: out {out.tolist()} lse {lse.tolist()}")

    # dense causal attention
    for (ql, kl, Hq, Hkv, ps, layout, D) in [
            ((3, 1, 5), (7, 1, 12), 4, 2, 4, "NHD", 8),
            ((2, 6), (9, 6), 3, 1, 2, "HND", 4),
            ((4, 0, 2), (4, 3, 17), 2, 2, 8, "NHD", 128)]:
        case = _small(ql, kl, Hq, Hkv, ps, layout, D, seed=sum(kl))
        o1, l1 = _prefill(lib, case)
        o2, l2 = _brute(case)
        if not (np.allclose(o1, o2, rtol=0, atol=1e-12) and np.allclose(l1, l2, rtol=0, atol=1e-12)):
            bad.append(f"dense causal attention differs for q_lens {ql}, kv_lens {kl}")

    # one query token per request is decode; the last token of a request sees
    # the whole cache
    case = _small((1, 1, 1), (5, 17, 2), 8, 2, 4, "NHD", 16, seed=3)
    o1, l1 = _prefill(lib, case)
    t = case.tables
    o2, l2 = oracle.paged_decode(W.bf16_bits(case.q), W.bf16_bits(case.k), W.bf16_bits(case.v),
                                 t.indptr, t.indices, t.last_page_len, num_kv_heads=2, page_size=4,
                                 layout=0, sm_scale=case.sm_scale, lib=lib)
    if not (np.array_equal(o1, o2) and np.array_equal(l1, l2)):
        bad.append("one query token per request differs from decode")
    case = _small((3, 4), (6, 9), 4, 4, 2, "HND", 8, seed=4)
    o1, l1 = _prefill(lib, case)
    last = case.qo_indptr[1:] - 1
    t = case.tables
    qb = W.bf16_bits(case.q)[last]
    o2, l2 = oracle.paged_decode(qb, W.bf16_bits(case.k), W.bf16_bits(case.v), t.indptr,
                                 t.indices, t.last_page_len, num_kv_heads=4, page_size=2,
                                 layout=1, sm_scale=case.sm_scale, lib=lib)
    if not (np.array_equal(o1[last], o2) and np.array_equal(l1[last], l2)):
        bad.append("last query token differs from decode over the whole cache")

    # causality: K/V past the first query token's position do not reach it
    case = _small((4,), (10,), 2, 1, 4, "NHD", 8, seed=5)
    o1, l1 = _prefill(lib, case)
    kb, vb = W.bf16_bits(case.k).copy(), W.bf16_bits(case.v).copy()
    t = case.tables
    pos0 = 10 - 4
    for j in range(pos0 + 1, 10):   # tokens after query 0's position
        page, slot = int(t.indices[j // 4]), j % 4
        kb[page, slot] = _bits(np.full(8, 3.0))
        vb[page, slot] = _bits(np.full(8, -5.0))
    o2, l2 = oracle.paged_prefill(W.bf16_bits(case.q), kb, vb, case.qo_indptr, t.indptr,
                                  t.indices, t.last_page_len, num_kv_heads=1, page_size=4,
                                  layout=0, sm_scale=case.sm_scale, lib=lib)
    if not (np.array_equal(o1[0], o2[0]) and np.array_equal(l1[0], l2[0])):
        bad.append("a row sees tokens past its position")
    if np.array_equal(o1[3], o2[3]):
        bad.append("the last row ignores tokens before its position")

    # identical keys: mean of the visible values, lse = s + ln(p + 1)
    case = _small((3,), (5,), 1, 1, 2, "NHD", 4, seed=6)
    key = _bits([0.5, -1.0, 0.25, 2.0])
    kb = W.bf16_bits(case.k).copy()
    kb[...] = key
    o1, l1 = oracle.paged_prefill(W.bf16_bits(case.q), kb, W.bf16_bits(case.v), case.qo_indptr,
                                  case.tables.indptr, case.tables.indices,
                                  case.tables.last_page_len, num_kv_heads=1, page_size=2,
                                  layout=0, sm_scale=case.sm_scale, lib=lib)
    V = _dense(W.bf16_bits(case.v), "NHD", case.tables.indices, 5, 0)
    qf = _f64(W.bf16_bits(case.q))
    for i in range(3):
        p = 2 + i
        s = case.sm_scale * float(qf[i, 0] @ _f64(key))
        if not (np.allclose(o1[i, 0], V[:p + 1].mean(0), rtol=0, atol=1e-12)
                and math.isclose(l1[i, 0], s + math.log(p + 1), abs_tol=1e-12)):
            bad.append(f"identical keys: row {i}")

    # a row subset gives the same bits as the full run, at any thread count
    case = _small((5, 2), (11, 3), 4, 2, 4, "HND", 8, seed=7)
    o1, l1 = _prefill(lib, case)
    rows = [(6, 3), (0, 0), (4, 1), (2, 2)]
    o2, l2 = _prefill(lib, case, rows=rows, nthreads=3)
    for n, (tk, hq) in enumerate(rows):
        if not (np.array_equal(o2[n], o1[tk, hq]) and l2[n] == l1[tk, hq]):
            bad.append(f"row subset differs at {tk, hq}")
    o3, l3 = _prefill(lib, case, nthreads=1)
    if not (np.array_equal(o3, o1) and np.array_equal(l3, l1)):
        bad.append("thread count changes the result")
    return bad


# ------------------------------------------------------------------ tests

def test_prefill_pins():
    assert prefill_pins(None) == []


@pytest.mark.parametrize("mutation", ["q_len_above_kv_len", "qo_start", "qo_decreasing"])
def test_invalid_prefill_tables_are_rejected(mutation):
    case = _small((2, 3), (4, 5), 2, 1, 4, "NHD", 8, seed=8)
    qo = case.qo_indptr.copy()
    qb = W.bf16_bits(case.q)
    if mutation == "q_len_above_kv_len":
        case = _small((2, 3), (4, 3), 2, 1, 4, "NHD", 8, seed=8)
        qo = np.array([0, 2, 6], np.int32)  # request 1: 4 query tokens over 3 cached
        qb = np.zeros((6, 2, 8), np.uint16)
    elif mutation == "qo_start":
        qo = qo + 1
        qb = np.zeros((int(qo[-1]), 2, 8), np.uint16)
    else:
        qo = np.array([0, 3, 2], np.int32)
        qb = np.zeros((2, 2, 8), np.uint16)
    t = case.tables
    with pytest.raises(oracle.OracleError):
        oracle.paged_prefill(qb, W.bf16_bits(case.k), W.bf16_bits(case.v), qo, t.indptr,
                             t.indices, t.last_page_len, num_kv_heads=1, page_size=4, layout=0,
                             sm_scale=0.3)


PREFILL_MUTANTS = {
    "causal_off_by_one": ("row_state(P, qrow, b, hq / G, pos + 1,",
                          "row_state(P, qrow, b, hq / G, pos,"),
    "top_left_alignment": ("const int64_t pos = L - q_len + (t - J->qo_indptr[b]);",
                           "const int64_t pos = (t - J->qo_indptr[b]);"),
    "query_row_of_request": (
        "P->q + ((size_t)t * (size_t)P->Hq + (size_t)hq) * (size_t)P->D;",
        "P->q + ((size_t)(t - J->qo_indptr[b]) * (size_t)P->Hq + (size_t)hq) * (size_t)P->D;"),
    "kv_head_modulo": ("row_state(P, qrow, b, hq / G,", "row_state(P, qrow, b, hq % P->Hkv,"),
    "owner_search": ("while (J->qo_indptr[b + 1] <= t) ++b;",
                     "while (J->qo_indptr[b + 1] < t) ++b;"),
    "prefill_scale_dropped": ("        s[j] = P->sm_scale * dot;", "        s[j] = dot;"),
}


@pytest.mark.parametrize("name", sorted(PREFILL_MUTANTS))
def test_pins_reject_planted_mistakes(name, tmp_path):
    old, new = PREFILL_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    mutated = tmp_path / "oxd_oracle.c"
    mutated.write_text(src.replace(old, new))
    (tmp_path / "oxd_oracle.h").write_text(open(SRC[:-1] + "h").read())
    lib = oracle.bind(oracle.compile_library(str(mutated), str(tmp_path / f"lib_{name}.so")))
    try:
        failures = prefill_pins(lib)
    except Exception as e:  # a mutant may also crash the battery
        failures = [repr(e)]
    assert failures, f"mutant {name} passed every pin"
