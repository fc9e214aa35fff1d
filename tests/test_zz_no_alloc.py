"""The allocation-free entry point against the oracle and the workspace entry point.

``oxd_paged_decode_run_static_workspace`` serves callers that cannot call
cudaMalloc (a process that reserves all device memory at start-up, or a
plugin host that passes only input and output tensors); it runs the same
decode in a scratch array that the library itself holds on each GPU. Two
calls in a row must each match the f64 oracle and the regular entry point
within the decode tolerance (the second call reuses the array the first one
left behind), and a call after the first must leave the device's free memory
and torch's allocation count unchanged. Its device status is read with
``oxd_read_static_workspace_status``: a page index outside the pool shows
there as OXD_DEVICE_BAD_PAGE, and the next good call reads OK again.
This file is collected last, so a failure here comes after every other test.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_attn_gb300 as oxd
import workloads as W
from gpu_helpers import (ATOL, LSE_ATOL, RTOL, DeviceTables, assert_parity, oracle_ref,
                         plan_case, run_decode)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oxd.build()
    oracle.build()


def _close(a, b):
    a = a.float()
    b = b.float()
    return bool(((a - b).abs() <= ATOL + RTOL * b.abs()).all())


def _static_run(case, plan, tables, out, lse):
    oxd.oxd_paged_decode_run_static_workspace(plan, case.q, case.k, case.v, tables.indptr,
                                              tables.indices, tables.last, case.sm_scale,
                                              out, lse)


@pytest.mark.parametrize("G,layout,ps", [(4, "NHD", 16), (1, "HND", 16), (32, "NHD", 64)])
def test_static_workspace_matches_oracle_and_workspace_entry_twice(G, layout, ps):
    Hkv = 8 if G < 32 else 1
    case = W.custom_case([1, 40, 700, 2500, 129], num_qo_heads=G * Hkv, num_kv_heads=Hkv,
                         page_size=ps, layout=layout, seed=21 + G, device="cuda")
    plan = plan_case(case)
    assert plan.workspace_bytes <= 32 << 20
    tables = DeviceTables(case)
    ref_out, ref_lse, _, _ = run_decode(case, plan=plan, tables=tables)
    f64_out, f64_lse = oracle_ref(case)
    out = torch.empty_like(case.q)
    lse = torch.empty(case.batch, case.num_qo_heads, device="cuda")
    for call in range(2):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        torch.cuda.synchronize()
        alloc0 = torch.cuda.memory_allocated()
        free0 = torch.cuda.mem_get_info()[0]
        _static_run(case, plan, tables, out, lse)
        assert oxd.oxd_read_static_workspace_status() == oxd.OXD_DEVICE_OK
        torch.cuda.synchronize()
        if call == 1:
            # the first call loaded the kernels; from then on nothing is allocated
            assert torch.cuda.memory_allocated() == alloc0, "torch allocation changed"
            assert torch.cuda.mem_get_info()[0] == free0, "device free memory changed"
        assert_parity(out, f64_out, lse, f64_lse, f"call {call} against the oracle")
        assert _close(out, ref_out), f"call {call}: output differs from the workspace entry"
        assert float((lse - ref_lse).abs().max()) <= LSE_ATOL, f"call {call}: lse differs"


def test_static_workspace_reports_a_bad_page_through_its_status_reader():
    case = W.custom_case([300, 40, 1000], num_qo_heads=32, num_kv_heads=8, page_size=16,
                         seed=31, device="cuda")
    plan = plan_case(case)
    bad = DeviceTables(case)
    bad.indices[3] = case.tables.num_pages + 5   # outside the pool
    out = torch.empty_like(case.q)
    lse = torch.empty(case.batch, case.num_qo_heads, device="cuda")
    _static_run(case, plan, bad, out, lse)
    assert oxd.oxd_read_static_workspace_status() == oxd.OXD_DEVICE_BAD_PAGE
    assert torch.isfinite(out.float()).all()   # page 0 was read in its place
    good = DeviceTables(case)
    _static_run(case, plan, good, out, lse)
    assert oxd.oxd_read_static_workspace_status() == oxd.OXD_DEVICE_OK
    ref_out, ref_lse = oracle_ref(case)
    assert_parity(out, ref_out, lse, ref_lse, "after the bad call")


def test_static_workspace_rejects_plans_beyond_its_size():
    # 64 requests x 64 forced splits x 32 heads of partial states need more
    # than 32 MiB of scratch; the call must refuse before touching the device.
    lengths = np.full(64, 8192, np.int64)
    pages = lengths // 16
    indptr = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
    last = np.full(64, 16, np.int32)
    desc = oxd.make_desc(64, 32, 8, 16, "NHD", int(pages.sum()), force_splits=64)
    plan = oxd.oxd_paged_decode_plan(desc, indptr, last, torch.cuda.current_device())
    assert plan.workspace_bytes > 32 << 20
    fake = 1 << 40
    with pytest.raises(oxd.OxdError) as e:
        oxd.oxd_paged_decode_run_static_workspace(plan, fake, fake, fake, fake, fake, fake, 1.0,
                                                  fake, None, 0)
    assert e.value.status == oxd.OXD_ERR_WORKSPACE_TOO_SMALL
