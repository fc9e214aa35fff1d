"""Shared helpers of the GPU tests: run the C-ABI path, query the oracle, compare.

The tolerance is the one fixed for this operation: every bf16 output element
within 1.5e-2 absolute + 1e-2 relative of the f64 oracle, every LSE within
1e-3 absolute.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_decode_attn_gb300 as oxd
import workloads as W

ATOL = 1.5e-2
RTOL = 1e-2
LSE_ATOL = 1e-3


def plan_case(case: W.Case, **kw) -> oxd.Plan:
    t = case.tables
    desc = oxd.make_desc(case.batch, case.num_qo_heads, case.num_kv_heads, case.page_size,
                         case.layout, t.num_pages, head_dim=case.head_dim, **kw)
    return oxd.oxd_paged_decode_plan(desc, t.indptr, t.last_page_len,
                                     torch.cuda.current_device())


class DeviceTables:
    def __init__(self, case: W.Case, device="cuda"):
        t = case.tables
        self.indptr = torch.as_tensor(t.indptr, device=device)
        self.indices = torch.as_tensor(t.indices, device=device)
        self.last = torch.as_tensor(t.last_page_len, device=device)


def run_decode(case: W.Case, plan: oxd.Plan | None = None, tables: DeviceTables | None = None,
               want_lse=True, workspace=None, out=None, lse=None, **plan_kw):
    """One decode step through the C ABI; returns (out bf16, lse f32 or None, plan, ws)."""
    dev = case.q.device
    plan = plan or plan_case(case, **plan_kw)
    tables = tables or DeviceTables(case, dev)
    if out is None:
        out = torch.empty_like(case.q)
    if lse is None and want_lse:
        lse = torch.empty(case.batch, case.num_qo_heads, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=dev)
    oxd.oxd_paged_decode_run(plan, case.q, case.k, case.v, tables.indptr, tables.indices,
                             tables.last, case.sm_scale, out, lse, workspace,
                             plan.workspace_bytes)
    return out, lse, plan, workspace


def oracle_ref(case: W.Case, heads=None, nthreads=0):
    return oracle.paged_decode(
        W.bf16_bits(case.q), W.bf16_bits(case.k), W.bf16_bits(case.v), case.tables.indptr,
        case.tables.indices, case.tables.last_page_len, num_kv_heads=case.num_kv_heads,
        page_size=case.page_size, layout=0 if case.layout == "NHD" else 1,
        sm_scale=case.sm_scale, heads=heads, nthreads=nthreads)


def assert_parity(out_gpu, ref_out, lse_gpu=None, ref_lse=None, what=""):
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    err = np.abs(o - ref_out)
    bound = ATOL + RTOL * np.abs(ref_out)
    bad = err > bound
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} output elements outside tolerance; worst at {i}: "
            f"gpu {o[i]!r} ref {ref_out[i]!r} (max err {err.max():.3e})")
    if lse_gpu is not None:
        lg = lse_gpu.float().cpu().numpy().astype(np.float64)
        lerr = np.abs(lg - ref_lse)
        assert np.isfinite(lg).all(), f"{what}: non-finite lse"
        assert lerr.max() <= LSE_ATOL, f"{what}: max lse err {lerr.max():.3e}"
    return float(err.max())


def gpu_heads(out, lse, heads):
    """Gather [n, D] / [n] rows of (b, hq) pairs from full GPU outputs."""
    idx_b = torch.as_tensor([h[0] for h in heads], device=out.device)
    idx_h = torch.as_tensor([h[1] for h in heads], device=out.device)
    return out[idx_b, idx_h], (lse[idx_b, idx_h] if lse is not None else None)
