"""Runs on a workspace bound to their plan (``oxd_plan_bind_workspace``).

A bound run reads the work list from the workspace instead of the kernels'
parameter buffers and copies nothing, so it must give bitwise the same out
and lse as the unbound run of the same plan, for every kind of list: one that
fits the parameter buffers, one too long for them (uploaded by unbound runs),
one with split (request, KV head) streams and their merge entries, and the
paired 16-row CTAs of a 32-head group.

A binding ends on the device when anything else writes the workspace's list
or stamp. The kernels then compute nothing and record a plan mismatch; a
list that still carries the stamp but holds values outside the plan (a
damaged list) is reported the same way, with every access kept inside the
caller's buffers by the kernels' own bounds checks on each unit.
"""
import numpy as np
import pytest
import torch

import paged_kv_decode_attn_gb300 as oxd
import workloads as W
from gpu_helpers import DeviceTables, plan_case, run_decode

pytestmark = pytest.mark.gpu

HEADER = 256  # bytes of the workspace header; the unit array follows it


@pytest.fixture(scope="module", autouse=True)
def setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oxd.build()


def _case(kind):
    if kind == "gqa4_nhd":
        return W.custom_case([1, 40, 700, 2500, 129], num_qo_heads=32, num_kv_heads=8,
                             page_size=16, layout="NHD", seed=71, device="cuda"), {}
    if kind == "mha_hnd":
        return W.custom_case([17, 333, 1024], num_qo_heads=8, num_kv_heads=8, page_size=16,
                             layout="HND", seed=72, device="cuda"), {}
    if kind == "mqa32_pairs":
        return W.custom_case([5000, 64, 1], num_qo_heads=32, num_kv_heads=1, page_size=64,
                             layout="NHD", seed=73, device="cuda"), {}
    if kind == "mqa32_mma_pairs":  # each piece on two 16-row CTAs, one per row half
        return W.custom_case([5000, 64, 1], num_qo_heads=32, num_kv_heads=1, page_size=64,
                             layout="NHD", seed=73, device="cuda"), {"tensor_path": 1}
    if kind == "forced_splits":
        return W.custom_case([3000, 900, 77], num_qo_heads=32, num_kv_heads=8, page_size=16,
                             layout="NHD", seed=74, device="cuda"), {"force_splits": 5}
    if kind == "long_list":
        return W.custom_case([64] * 600, num_qo_heads=8, num_kv_heads=8, page_size=16,
                             layout="NHD", seed=75, device="cuda"), {"max_splits": 1}
    raise ValueError(kind)


def _bound_run(case, plan, tables, ws, fill=float("nan")):
    out = torch.full_like(case.q, fill)
    lse = torch.full((case.batch, case.num_qo_heads), fill, device="cuda")
    oxd.oxd_paged_decode_run(plan, case.q, case.k, case.v, tables.indptr, tables.indices,
                             tables.last, case.sm_scale, out, lse, ws, plan.workspace_bytes)
    return out, lse


@pytest.mark.parametrize("kind", ["gqa4_nhd", "mha_hnd", "mqa32_pairs", "mqa32_mma_pairs",
                                  "forced_splits", "long_list"])
def test_bound_runs_equal_unbound_runs_bitwise(kind):
    case, kw = _case(kind)
    plan = plan_case(case, **kw)
    info = plan.info
    if kind == "long_list":
        assert info.upload_bytes > 0
    if kind == "forced_splits":
        assert info.num_split_requests > 0
    tables = DeviceTables(case)
    ref_out, ref_lse, _, _ = run_decode(case, plan=plan, tables=tables)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    oxd.oxd_plan_bind_workspace(plan, ws)
    for _ in range(2):
        out, lse = _bound_run(case, plan, tables, ws)
        assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))


def test_overwritten_stamp_ends_the_binding():
    case, kw = _case("forced_splits")
    plan = plan_case(case, **kw)
    tables = DeviceTables(case)
    ref_out, _, _, _ = run_decode(case, plan=plan, tables=tables)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    oxd.oxd_plan_bind_workspace(plan, ws)
    ws.zero_()  # someone else's write into the workspace
    out, lse = _bound_run(case, plan, tables, ws)
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_PLAN_MISMATCH
    assert bool(torch.isnan(out.float()).all()) and bool(torch.isnan(lse).all())
    oxd.oxd_plan_bind_workspace(plan, ws)  # binding again restores it
    out, _ = _bound_run(case, plan, tables, ws)
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))


def test_binding_another_plan_to_the_workspace_ends_the_first_binding():
    case_a, _ = _case("gqa4_nhd")
    case_b, _ = _case("mha_hnd")
    plan_a, plan_b = plan_case(case_a), plan_case(case_b)
    tab_a, tab_b = DeviceTables(case_a), DeviceTables(case_b)
    ref_b, _, _, _ = run_decode(case_b, plan=plan_b, tables=tab_b)
    nbytes = max(plan_a.workspace_bytes, plan_b.workspace_bytes)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    oxd.oxd_plan_bind_workspace(plan_a, ws)
    oxd.oxd_plan_bind_workspace(plan_b, ws)
    out_a, _ = _bound_run(case_a, plan_a, tab_a, ws)
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_PLAN_MISMATCH
    assert bool(torch.isnan(out_a.float()).all())
    out_b, _ = _bound_run(case_b, plan_b, tab_b, ws)
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
    assert torch.equal(out_b.view(torch.int16), ref_b.view(torch.int16))


def test_unbound_upload_run_of_another_plan_ends_the_binding():
    case_a, _ = _case("gqa4_nhd")
    case_b, kw_b = _case("long_list")
    plan_a, plan_b = plan_case(case_a), plan_case(case_b, **kw_b)
    assert plan_b.info.upload_bytes > 0
    tab_a, tab_b = DeviceTables(case_a), DeviceTables(case_b)
    nbytes = max(plan_a.workspace_bytes, plan_b.workspace_bytes)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    oxd.oxd_plan_bind_workspace(plan_a, ws)
    run_decode(case_b, plan=plan_b, tables=tab_b, workspace=ws)  # uploads B's list
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
    out_a, _ = _bound_run(case_a, plan_a, tab_a, ws)
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_PLAN_MISMATCH
    assert bool(torch.isnan(out_a.float()).all())


def test_unbound_run_of_another_plan_ends_the_binding():
    # the other plan's list rides in its kernels' parameters, but its run
    # still writes partial states over the bound list: the binding ends
    case_a, _ = _case("long_list")
    case_b, kw_b = _case("forced_splits")
    plan_a, plan_b = plan_case(case_a, max_splits=1), plan_case(case_b, **kw_b)
    assert plan_b.info.upload_bytes == 0
    tab_a, tab_b = DeviceTables(case_a), DeviceTables(case_b)
    ref_a, _, _, _ = run_decode(case_a, plan=plan_a, tables=tab_a)
    nbytes = max(plan_a.workspace_bytes, plan_b.workspace_bytes)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    oxd.oxd_plan_bind_workspace(plan_a, ws)
    run_decode(case_b, plan=plan_b, tables=tab_b, workspace=ws)
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
    out_a, _ = _bound_run(case_a, plan_a, tab_a, ws)
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_PLAN_MISMATCH
    assert bool(torch.isnan(out_a.float()).all())
    oxd.oxd_plan_bind_workspace(plan_a, ws)
    out_a, _ = _bound_run(case_a, plan_a, tab_a, ws)
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
    assert torch.equal(out_a.view(torch.int16), ref_a.view(torch.int16))


def _align256(x):
    return (x + 255) // 256 * 256


@pytest.mark.parametrize("region", ["unit_array", "cta_records", "everything_after_header"])
def test_damaged_list_is_reported_not_followed(region):
    # The workspace list: a 256-byte header, the unit array (16 bytes a
    # unit), then at the next 256-byte boundary one 32-byte record per CTA
    # (its unit range and a copy of its first unit). Damaged bytes read
    # 0x7f7f7f7f in every field: a unit's first page then lies far beyond the
    # index array, a CTA range beyond the unit count, a merge entry beyond the
    # output rows, and the kernels reject each before any access it governs.
    case, kw = _case("long_list")                 # about 16 units a CTA
    plan = plan_case(case, **kw)
    info = plan.info
    assert info.num_split_requests == 0
    tables = DeviceTables(case)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    oxd.oxd_plan_bind_workspace(plan, ws)
    units_end = HEADER + 16 * info.num_work_items
    rec_begin = _align256(units_end)
    rec_end = rec_begin + 32 * info.grid_ctas
    lo, hi = {"unit_array": (HEADER, units_end), "cta_records": (rec_begin, rec_end),
              "everything_after_header": (HEADER, plan.workspace_bytes)}[region]
    ws[lo:hi].fill_(0x7F)
    out, lse = _bound_run(case, plan, tables, ws)
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_PLAN_MISMATCH
    nan = torch.isnan(out.float())
    if region == "unit_array":
        # each CTA's first unit comes from its intact record; the rest are
        # rejected
        assert bool(nan.any()) and not bool(nan.all())
    else:
        assert bool(nan.all()) and bool(torch.isnan(lse).all())


def test_runs_on_another_workspace_are_unaffected_by_a_binding():
    case, kw = _case("forced_splits")
    plan = plan_case(case, **kw)
    tables = DeviceTables(case)
    ws_bound = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    oxd.oxd_plan_bind_workspace(plan, ws_bound)
    ref_out, ref_lse, _, ws_other = run_decode(case, plan=plan, tables=tables)
    assert oxd.oxd_read_device_status(ws_other) == oxd.OXD_DEVICE_OK
    out, lse = _bound_run(case, plan, tables, ws_bound)
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
