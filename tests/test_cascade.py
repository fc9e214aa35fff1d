"""Cascade (shared-prefix) decode through the C ABI against the f64 oracle (GPU).

A plan given shared_prefix_tokens and share_group attends each sharing group's
requests to their common prefix once (prefill kernel, no mask), decodes only
the pages after it, and merges the two states. The result must match the
oracle of the plain decode (|out - ref| <= 1.5e-2 + 1e-2 |ref|, lse 1e-3) and
the plain decode itself within the same bound; runs on a bound workspace are
bitwise equal to unbound ones and a captured graph replays. Cases cover every
decode kernel variant (G = 1, 4, 8, 32 on both tensor paths), NHD and HND,
requests no longer than the prefix (decoded whole), a group with one longer
request, groups wider than one prefix tile, forced splits of the suffixes, and
the full GQA8 workload whose groups of eight share 1024 tokens.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_attn_gb300 as oxd
import workloads as W
from gpu_helpers import DeviceTables, assert_parity, gpu_heads, oracle_ref, plan_case, run_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oxd.build()
    oracle.build()


def _shared_case(lengths, G, Hkv, ps, layout, prefix, group, seed):
    return W.custom_case(lengths, num_qo_heads=G * Hkv, num_kv_heads=Hkv, page_size=ps,
                         layout=layout, seed=seed, device="cuda", shared_prefix_tokens=prefix,
                         share_group=group)


@pytest.mark.parametrize("G,Hkv,tensor_path", [(1, 8, 0), (4, 8, 0), (8, 4, 0), (32, 1, 0),
                                               (32, 1, 1)])
@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_cascade_matches_oracle_and_plain_decode(G, Hkv, tensor_path, layout):
    # two groups of four: group 0 all longer than the prefix, group 1 with a
    # request exactly at the prefix and one below it (both decoded whole)
    lengths = [700, 129, 3000, 256, 128, 90, 1500, 400]
    case = _shared_case(lengths, G, Hkv, 16, layout, 128, 4, seed=60 + G)
    plan = plan_case(case, shared_prefix_tokens=128, share_group=4, tensor_path=tensor_path)
    info = plan.info
    assert info.cascade_requests == 4 + 2 and info.launches_per_run == 3
    out, lse, _, ws = run_decode(case, plan)
    torch.cuda.synchronize()
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
    ref_o, ref_l = oracle_ref(case)
    assert_parity(out, ref_o, lse, ref_l, f"cascade G{G} {layout}")
    o2, l2, _, _ = run_decode(case, tensor_path=tensor_path)
    torch.cuda.synchronize()
    assert_parity(out, o2.float().cpu().numpy().astype(np.float64), lse,
                  l2.cpu().numpy().astype(np.float64), "cascade vs plain decode")


def test_group_with_one_long_request_and_wide_groups():
    # group of 40 (three prefix tiles at G = 8) and a group whose only longer
    # request is decoded whole
    lengths = [300 + 37 * i for i in range(40)] + [100, 64, 500, 32]
    case = _shared_case(lengths, 8, 2, 16, "NHD", 256, 40, seed=71)
    plan = plan_case(case, shared_prefix_tokens=256, share_group=40)
    assert plan.info.cascade_units == 3 * 2 and plan.info.cascade_requests == 40
    out, lse, _, ws = run_decode(case, plan)
    torch.cuda.synchronize()
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
    ref_o, ref_l = oracle_ref(case)
    assert_parity(out, ref_o, lse, ref_l, "wide groups")


@pytest.mark.parametrize("force", [1, 3])
def test_forced_suffix_splits(force):
    case = _shared_case([2000, 1200, 900, 4000], 4, 8, 16, "HND", 512, 4, seed=72)
    plan = plan_case(case, shared_prefix_tokens=512, share_group=4, force_splits=force)
    out, lse, _, ws = run_decode(case, plan)
    torch.cuda.synchronize()
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
    ref_o, ref_l = oracle_ref(case)
    assert_parity(out, ref_o, lse, ref_l, f"force {force}")


def test_bound_workspace_matches_unbound_and_graph_replays():
    case = _shared_case([900, 300, 1700, 260, 2000, 1000, 700, 1300], 4, 8, 16, "NHD", 256, 4,
                        seed=73)
    plan = plan_case(case, shared_prefix_tokens=256, share_group=4)
    tables = DeviceTables(case)
    out1, lse1, _, _ = run_decode(case, plan, tables)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    oxd.oxd_plan_bind_workspace(plan, ws)
    out2, lse2, _, _ = run_decode(case, plan, tables, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(lse1.view(torch.int32), lse2.view(torch.int32))
    out3 = torch.empty_like(out1)
    lse3 = torch.empty_like(lse1)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        oxd.oxd_paged_decode_run(plan, case.q, case.k, case.v, tables.indptr, tables.indices,
                                 tables.last, case.sm_scale, out3, lse3, ws, plan.workspace_bytes,
                                 torch.cuda.current_stream())
    gen = torch.Generator(device="cuda").manual_seed(9)
    case.q.copy_(torch.randn(case.q.shape, generator=gen, device="cuda").to(torch.bfloat16))
    graph.replay()
    torch.cuda.synchronize()
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
    ref_o, ref_l = oracle_ref(case)
    assert_parity(out3, ref_o, lse3, ref_l, "graph replay")


def test_full_gqa8_workload_sampled_heads():
    cfg = W.CONFIGS["gqa8_b256_u128to16384_prefix1024x8_ps16_nhd"]
    case = W.make_case(cfg, device="cuda")
    plan = plan_case(case, shared_prefix_tokens=1024, share_group=8)
    assert plan.info.cascade_requests > 200
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    oxd.oxd_plan_bind_workspace(plan, ws)
    out, lse, _, _ = run_decode(case, plan, workspace=ws)
    torch.cuda.synchronize()
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    rng = np.random.default_rng(8)
    heads = [(int(b), int(h)) for b, h in zip(rng.integers(0, case.batch, 48),
                                              rng.integers(0, case.num_qo_heads, 48))]
    heads += [(0, 0), (7, 63), (case.batch - 1, 5)]
    ref_o, ref_l = oracle_ref(case, heads=heads)
    go, gl = gpu_heads(out, lse, heads)
    assert_parity(go, ref_o, gl, ref_l, "GQA8 cascade")
