"""The allocation-free decode entry point agrees with the workspace entry point.

``oxd_paged_decode_run_static_workspace`` serves callers that cannot call
cudaMalloc (a process that reserves all device memory at start-up, or a
plugin host that passes only input and output tensors); it runs the same
decode in a scratch array that the library itself holds on each GPU. Two
calls in a row must each match the regular entry point within the decode
tolerance: the second call reuses the array the first one left behind.
This file is collected last, so a failure here comes after every other test.
"""
import numpy as np
import pytest
import torch

import paged_kv_decode_attn_gb300 as oxd
import workloads as W
from gpu_helpers import ATOL, LSE_ATOL, RTOL, DeviceTables, plan_case, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oxd.build()


def _close(a, b):
    a = a.float()
    b = b.float()
    return bool(((a - b).abs() <= ATOL + RTOL * b.abs()).all())


@pytest.mark.parametrize("G,layout,ps", [(4, "NHD", 16), (1, "HND", 16), (32, "NHD", 64)])
def test_static_workspace_matches_workspace_entry_twice(G, layout, ps):
    Hkv = 8 if G < 32 else 1
    case = W.custom_case([1, 40, 700, 2500, 129], num_qo_heads=G * Hkv, num_kv_heads=Hkv,
                         page_size=ps, layout=layout, seed=21 + G, device="cuda")
    plan = plan_case(case)
    assert plan.workspace_bytes <= 32 << 20
    tables = DeviceTables(case)
    ref_out, ref_lse, _, _ = run_decode(case, plan=plan, tables=tables)
    for call in range(2):
        out = torch.full_like(case.q, float("nan"))
        lse = torch.full((case.batch, case.num_qo_heads), float("nan"), device="cuda")
        oxd.oxd_paged_decode_run_static_workspace(plan, case.q, case.k, case.v, tables.indptr,
                                                  tables.indices, tables.last, case.sm_scale,
                                                  out, lse)
        torch.cuda.synchronize()
        assert _close(out, ref_out), f"call {call}: output differs"
        assert float((lse - ref_lse).abs().max()) <= LSE_ATOL, f"call {call}: lse differs"


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
