"""The oracle's pins catch plausible slips.

Each mutant is a copy of ``oracle/oxd_oracle.c`` with one deliberate mistake
planted (in the oracle, on the CPU): a wrong head mapping, a dropped
``last_page_len`` mask, log2 instead of ln, a missing ``sm_scale``, a
transposed pool index, a wrong sign, a skipped block-table lookup, a dropped
normalisation, a merge that forgets the max shift. The test builds each mutant
and requires that the battery of pins (hand-derived closed forms, brute force,
invariants) rejects it, while the unmodified source passes the same battery.
"""
import json
import math
import os
import shutil

import numpy as np
import pytest
import torch

import oracle
import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "oxd_oracle.c")

MUTANTS = {
    "head_mapping_modulo": ("int h = hq / G;", "int h = hq % P->Hkv;"),
    "ignores_last_page_len": (
        "return (pages - 1) * (int64_t)page_size + (int64_t)last_page_len[b];",
        "return pages * (int64_t)page_size;"),
    "lse_in_log2": ("*lse = M + log(Z);", "*lse = M + log2(Z);"),
    "missing_sm_scale": ("s[j - t0] = P->sm_scale * dot;", "s[j - t0] = dot;"),
    "nhd_index_transposed": (
        "return (((size_t)page * (size_t)page_size + (size_t)t) * (size_t)Hkv + (size_t)h) *",
        "return (((size_t)page * (size_t)Hkv + (size_t)h) * (size_t)page_size + (size_t)t) *"),
    "softmax_sign_flipped": ("Z += exp(s[j] - M);", "Z += exp(M - s[j]);"),
    "no_block_table_lookup": (
        "int64_t page = P->indices[P->indptr[b] + j / P->page_size];",
        "int64_t page = P->indptr[b] + j / P->page_size;"),
    "unnormalised_weights": ("double w = exp(s[j] - M) / Z;", "double w = exp(s[j] - M);"),
    "merge_without_max_shift": ("for (int i = 0; i < S; ++i) W += exp(s[i] - M);",
                                "for (int i = 0; i < S; ++i) W += exp(s[i]);"),
    "token_off_by_one": ("int t = (int)(j % P->page_size);",
                         "int t = (int)((j + 1) % P->page_size);"),
}


def _bits(x):
    t = torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _decode(lib, case, **kw):
    return oracle.paged_decode(
        W.bf16_bits(case.q), W.bf16_bits(case.k), W.bf16_bits(case.v), case.tables.indptr,
        case.tables.indices, case.tables.last_page_len, num_kv_heads=case.num_kv_heads,
        page_size=case.page_size, layout=0 if case.layout == "NHD" else 1,
        sm_scale=case.sm_scale, lib=lib, **kw)


def _brute(case):
    t = case.tables
    q = _f64(W.bf16_bits(case.q))
    kb, vb = _f64(W.bf16_bits(case.k)), _f64(W.bf16_bits(case.v))
    if case.layout == "HND":
        kb, vb = kb.transpose(0, 2, 1, 3), vb.transpose(0, 2, 1, 3)
    out = np.zeros((case.batch, case.num_qo_heads, case.head_dim))
    lse = np.zeros((case.batch, case.num_qo_heads))
    for b in range(case.batch):
        ind = t.indices[t.indptr[b]:t.indptr[b + 1]]
        L = int(t.lengths[b])
        K = kb[ind].reshape(-1, case.num_kv_heads, case.head_dim)[:L]
        V = vb[ind].reshape(-1, case.num_kv_heads, case.head_dim)[:L]
        for hq in range(case.num_qo_heads):
            h = hq // case.group_size
            e = np.exp(case.sm_scale * (K[:, h] @ q[b, hq]))
            out[b, hq] = (e[:, None] * V[:, h]).sum(0) / e.sum()
            lse[b, hq] = math.log(e.sum())
    return out, lse


def _pins(lib) -> list:
    """Run the pin battery against one oracle build; return the names that failed."""
    failed = []

    def check(name, fn):
        try:
            ok = fn()
        except Exception:  # a crash or a rejected input counts as a caught slip
            ok = False
        if not ok:
            failed.append(name)

    def golden():
        ok = True
        for fname in ("two_token_worked_example.json", "three_token_two_page_example.json"):
            with open(os.path.join(HERE, "golden", fname)) as f:
                g = json.load(f)
            scale = {"ln(3)": math.log(3.0), "ln(2)": math.log(2.0)}[g["sm_scale_expr"]]
            want = {"ln(4)": math.log(4.0), "ln(7)": math.log(7.0)}[g["expected_lse_expr"]]
            out, lse = oracle.paged_decode(
                _bits(g["q"]), _bits(g["k_pages"]), _bits(g["v_pages"]), g["indptr"],
                g["indices"], g["last_page_len"], num_kv_heads=1, page_size=g["page_size"],
                layout=0, sm_scale=scale, lib=lib)
            ok &= np.allclose(out, g["expected_out"], rtol=0, atol=1e-12)
            ok &= abs(lse[0, 0] - want) < 1e-12
        return ok

    def brute(layout):
        def f():
            case = W.custom_case([1, 17, 40], num_qo_heads=4, num_kv_heads=2, page_size=8,
                                 layout=layout, head_dim=4, seed=31, sigma=0.5)
            out, lse = _decode(lib, case)
            ro, rl = _brute(case)
            return np.allclose(out, ro, rtol=1e-12, atol=1e-12) and np.allclose(
                lse, rl, rtol=1e-12, atol=1e-12)
        return f

    def merge_forms():
        v = np.random.default_rng(3).normal(size=(2, 4))
        o, s = oracle.merge_states(v, np.log([1.0, 3.0]), lib=lib)
        return np.allclose(o, 0.25 * v[0] + 0.75 * v[1], atol=1e-14) and abs(
            s - math.log(4.0)) < 1e-14

    check("golden", golden)
    check("brute_nhd", brute("NHD"))
    check("brute_hnd", brute("HND"))
    check("merge", merge_forms)
    return failed


@pytest.fixture(scope="module")
def workdir(tmp_path_factory):
    return str(tmp_path_factory.mktemp("oracle_mutants"))


def test_unmodified_oracle_passes_battery(workdir):
    lib = oracle.bind(oracle.compile_library(SRC, os.path.join(workdir, "lib_orig.so")))
    assert _pins(lib) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_each_planted_slip_is_caught(workdir, name):
    old, new = MUTANTS[name]
    with open(SRC) as f:
        text = f.read()
    assert old in text, f"mutant {name}: anchor not found in the oracle source"
    src = os.path.join(workdir, f"{name}.c")
    with open(src, "w") as f:
        f.write(text.replace(old, new))
    shutil.copy(os.path.join(os.path.dirname(SRC), "oxd_oracle.h"), workdir)
    lib = oracle.bind(oracle.compile_library(src, os.path.join(workdir, f"lib_{name}.so")))
    assert _pins(lib), f"mutant {name} passed every pin"
