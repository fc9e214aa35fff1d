"""Small batches merged inside thread-block clusters (GPU).

When every (request, KV head) stream of a batch can be cut into C >= 2 pieces
and the batch then fits the resident CTAs, the plan runs stream k on the C
CTAs of cluster k and the cluster's first CTA merges the pieces: one launch,
no merge kernel. These cases check the result against the f64 oracle for
the kernel variants that take this path (G = 1, 2 and 3..8), NHD and HND,
clusters of 2..8 CTAs, with and without LSE; bitwise equality of bound and
unbound runs and of repeated runs; a CUDA-graph replay with new inputs; and
the device status for a bad page index (the merge still ends, no hang).
"""
import numpy as np
import pytest
import torch

import paged_kv_decode_attn_gb300 as oxd
import workloads as W
from gpu_helpers import DeviceTables, assert_parity, oracle_ref, plan_case, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oxd.build()


def _case(lengths, G, Hkv, layout="NHD", ps=16, seed=1):
    return W.custom_case(lengths, num_qo_heads=G * Hkv, num_kv_heads=Hkv, page_size=ps,
                         layout=layout, seed=seed, device="cuda", extra_pages=2)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("G,Hkv", [(1, 8), (1, 1), (2, 4), (2, 12), (3, 2), (4, 8), (8, 4)])
def test_cluster_merge_matches_oracle(G, Hkv, layout):
    case = _case([512, 200, 1000], G, Hkv, layout, seed=G)
    ref_out, ref_lse = oracle_ref(case)
    out, lse, plan, ws = run_decode(case)
    info = plan.info
    assert info.cluster_size == 8 and info.launches_per_run == 1
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
    assert_parity(out, ref_out, lse, ref_lse, f"cluster G={G} {layout}")


@pytest.mark.parametrize("lengths,C", [([33, 300], 3), ([20, 250, 64], 2), ([160] * 3, 8),
                                       ([81, 300], 6)])
def test_cluster_sizes(lengths, C):
    case = _case(lengths, 1, 4, "NHD", seed=C)
    ref_out, ref_lse = oracle_ref(case)
    out, lse, plan, ws = run_decode(case)
    assert plan.info.cluster_size == C
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
    assert_parity(out, ref_out, lse, ref_lse, f"clusters of {C}")


def test_cluster_merge_without_lse_and_bound_runs_bitwise():
    case = _case([512, 400], 4, 8, "HND", seed=11)
    plan = plan_case(case)
    assert plan.info.cluster_size == 8
    tables = DeviceTables(case)
    ref_out, ref_lse, _, _ = run_decode(case, plan=plan, tables=tables)
    out0, _, _, _ = run_decode(case, plan=plan, tables=tables, want_lse=False)
    assert torch.equal(out0.view(torch.int16), ref_out.view(torch.int16))
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    oxd.oxd_plan_bind_workspace(plan, ws)
    for _ in range(3):
        out = torch.full_like(case.q, float("nan"))
        lse = torch.full((case.batch, case.num_qo_heads), float("nan"), device="cuda")
        oxd.oxd_paged_decode_run(plan, case.q, case.k, case.v, tables.indptr, tables.indices,
                                 tables.last, case.sm_scale, out, lse, ws, plan.workspace_bytes)
        assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32))


def test_cluster_merge_replays_in_a_cuda_graph():
    case = _case([512, 300, 96], 8, 2, "NHD", seed=21)
    plan = plan_case(case)
    assert plan.info.cluster_size == 6
    tables = DeviceTables(case)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    oxd.oxd_plan_bind_workspace(plan, ws)
    q = case.q.clone()
    out = torch.empty_like(q)
    lse = torch.empty(case.batch, case.num_qo_heads, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        oxd.oxd_paged_decode_run(plan, q, case.k, case.v, tables.indptr, tables.indices,
                                 tables.last, case.sm_scale, out, lse, ws, plan.workspace_bytes, s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        oxd.oxd_paged_decode_run(plan, q, case.k, case.v, tables.indptr, tables.indices,
                                 tables.last, case.sm_scale, out, lse, ws, plan.workspace_bytes, s)
    for seed in (5, 6):
        gen = torch.Generator(device="cuda").manual_seed(seed)
        q.copy_(torch.randn(q.shape, generator=gen, device="cuda").to(q.dtype))
        g.replay()
        torch.cuda.synchronize()
        case_now = W.Case(case.batch, case.num_qo_heads, case.num_kv_heads, case.head_dim,
                          case.page_size, case.layout, case.sm_scale, case.tables, q, case.k,
                          case.v, True, "custom")
        ref_out, ref_lse = oracle_ref(case_now)
        assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
        assert_parity(out, ref_out, lse, ref_lse, f"graph replay {seed}")


def test_bad_page_index_in_a_cluster_is_reported():
    case = _case([512, 256], 4, 8, "NHD", seed=31)
    plan = plan_case(case)
    assert plan.info.cluster_size == 8
    tables = DeviceTables(case)
    tables.indices[5] = case.tables.num_pages + 7  # outside the pool
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    out, lse, _, _ = run_decode(case, plan=plan, tables=tables, workspace=ws)
    torch.cuda.synchronize()
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_BAD_PAGE
    assert bool(torch.isfinite(out.float()).all())
