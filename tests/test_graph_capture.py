"""A decode run on a bound workspace captured in a CUDA graph and replayed.

A run on the workspace bound to its plan enqueues only kernel launches (the
decode kernel, and the merge kernel with a programmatic dependency when some
stream is split), with every pointer fixed at the call. Captured once, the
graph replays the step on whatever the fixed buffers hold at replay time: new
query values and new page indices (the same lengths) give the same result as
a direct run on them, bitwise.
"""
import dataclasses

import pytest
import torch

import paged_kv_decode_attn_gb300 as oxd
import workloads as W
from gpu_helpers import DeviceTables, assert_parity, oracle_ref, plan_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oxd.build()


def _run(plan, case, tables, out, lse, ws, stream=None):
    oxd.oxd_paged_decode_run(plan, case.q, case.k, case.v, tables.indptr, tables.indices,
                             tables.last, case.sm_scale, out, lse, ws, plan.workspace_bytes,
                             stream)


@pytest.mark.parametrize("G,force", [(4, 0), (4, 3), (32, 0), (1, 12)])
def test_captured_run_replays_with_new_inputs(G, force):
    Hkv = 8 if G < 32 else 1
    case = W.custom_case([700, 33, 2500, 129], num_qo_heads=G * Hkv, num_kv_heads=Hkv,
                         page_size=16, layout="NHD", seed=40 + G, device="cuda")
    plan = plan_case(case, force_splits=force)
    if force > 1:
        assert plan.info.launches_per_run == 2
    tables = DeviceTables(case)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    oxd.oxd_plan_bind_workspace(plan, ws)
    out = torch.empty_like(case.q)
    lse = torch.empty(case.batch, case.num_qo_heads, device="cuda")
    _run(plan, case, tables, out, lse, ws)  # sets up the kernels before capture
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _run(plan, case, tables, out, lse, ws, torch.cuda.current_stream())

    gen = torch.Generator(device="cuda")
    for rep in range(3):
        # new inputs in the captured buffers: query values and a permuted
        # page order (same lengths, so the plan still holds)
        gen.manual_seed(1000 + rep)
        case.q.copy_(torch.randn(case.q.shape, generator=gen, device="cuda").to(torch.bfloat16))
        perm = torch.randperm(case.k.shape[0], generator=gen, device="cuda")
        inv = torch.empty_like(perm)
        inv[perm] = torch.arange(perm.numel(), device="cuda")
        case.k.copy_(case.k[perm].clone())
        case.v.copy_(case.v[perm].clone())
        tables.indices.copy_(inv[tables.indices.long()].to(torch.int32))
        graph.replay()
        torch.cuda.synchronize()
        assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
        ref_out = torch.empty_like(out)
        ref_lse = torch.empty_like(lse)
        _run(plan, case, tables, ref_out, ref_lse, ws)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), f"replay {rep}"
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))
    # and the last replay against the oracle on the final inputs
    case_now = dataclasses.replace(case, tables=_tables_on_host(case.tables, tables))
    o_ref, l_ref = oracle_ref(case_now)
    assert_parity(out, o_ref, lse, l_ref, f"graph G{G} force {force}")


def _tables_on_host(t, dev_tables):
    return dataclasses.replace(t, indices=dev_tables.indices.cpu().numpy())
