"""Decode launched as a programmatic dependent of the kernel before it (GPU).

In an engine step the fused RoPE + paged append writes each request's new
token (its rotated q, its K and V rows in their page slots) and the decode
reads them ("FlashInfer parity matrix", "Admitted attention matrix": "Fused
RoPE plus paged append" before "Paged batch decode"). A plan with pdl = 1
launches the decode's first kernel as a programmatic dependent of the kernel
before it on the stream: its CTAs may be scheduled while the append is still
running and wait for it (griddepcontrol.wait) before touching memory.

Each case checks the step against the oracle run on host copies (the
oracle's own append, then its decode over the grown cache) and bitwise
against the same step with plain launches: every decode kernel family, the
cascade and the cluster merge; and a loop of decode runs on one workspace,
each launched behind the previous run's merge, which reads the workspace
the next run writes.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_attn_gb300 as oxd
import workloads as W
from gpu_helpers import DeviceTables, assert_parity, plan_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oxd.build()
    oracle.build()


def _step_case(lengths, G, Hkv, seed, **kw):
    """A batch whose tables already cover one more token per request, the
    new token's q/k/v, and host copies of the pools before the append."""
    grown = [L + 1 for L in lengths]
    case = W.custom_case(grown, num_qo_heads=G * Hkv, num_kv_heads=Hkv, page_size=16,
                         layout="NHD", seed=seed, device="cuda", **kw)
    g = torch.Generator(device="cuda").manual_seed(seed + 1)
    B = len(lengths)
    new = [torch.randn(B, h, 128, generator=g, device="cuda").to(torch.bfloat16)
           for h in (G * Hkv, Hkv, Hkv)]
    tr = torch.arange(B, dtype=torch.int32, device="cuda")
    pos = torch.tensor(lengths, dtype=torch.int32, device="cuda")
    return case, new, tr, pos, (W.bf16_bits(case.k), W.bf16_bits(case.v))


def _oracle_step(case, new, tr, pos, before):
    t = case.tables
    refcount = np.ones(t.num_pages, np.int32)
    q_rot, kp, vp, st = oracle.rope_append(
        W.bf16_bits(new[0]), W.bf16_bits(new[1]), W.bf16_bits(new[2]), tr.cpu().numpy(),
        pos.cpu().numpy(), t.indptr, t.indices, refcount, before[0], before[1],
        page_size=case.page_size, layout=0)
    assert (st == oracle.APPEND_WRITTEN).all()
    return oracle.paged_decode(q_rot, kp, vp, t.indptr, t.indices, t.last_page_len,
                               num_kv_heads=case.num_kv_heads, page_size=case.page_size,
                               layout=0, sm_scale=case.sm_scale)


def _run_step(case, new, tr, pos, before, pdl, plan_kw):
    """Restore the pools, then append + decode back to back on one stream."""
    case.k.copy_(torch.from_numpy(before[0].view(np.int16)).view(torch.bfloat16).view_as(case.k))
    case.v.copy_(torch.from_numpy(before[1].view(np.int16)).view(torch.bfloat16).view_as(case.v))
    t = case.tables
    tables = DeviceTables(case)
    plan = plan_case(case, pdl=pdl, **plan_kw)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    oxd.oxd_plan_bind_workspace(plan, ws)
    aws = torch.empty(256, dtype=torch.uint8, device="cuda")
    desc = oxd.make_rope_append_desc(case.batch, case.batch, case.num_qo_heads,
                                     case.num_kv_heads, case.page_size, case.layout,
                                     t.num_pages, int(t.indptr[-1]))
    refcount = torch.ones(t.num_pages, dtype=torch.int32, device="cuda")
    q = torch.empty_like(new[0])
    out = torch.empty_like(new[0])
    lse = torch.empty(case.batch, case.num_qo_heads, device="cuda")
    torch.cuda.synchronize()
    oxd.oxd_rope_append(desc, new[0], new[1], new[2], tr, pos, tables.indptr, tables.indices,
                        refcount, q, case.k, case.v, aws)
    oxd.oxd_paged_decode_run(plan, q, case.k, case.v, tables.indptr, tables.indices,
                             tables.last, case.sm_scale, out, lse, ws)
    torch.cuda.synchronize()
    assert oxd.oxd_read_device_status(aws) == oxd.OXD_DEVICE_OK
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
    return out, lse, plan.info


CASES = {
    "fma_g1": (1, 8, [100, 257, 16, 1, 3000], {}),
    "mma8_g4": (4, 8, [100, 257, 16, 1, 3000, 4095, 64], {}),
    "mma16_g16": (16, 2, [700, 33, 2048], {}),
    "tcgen05_g32": (32, 1, [4000, 65, 1, 900], {}),
    "cluster_g1": (1, 8, [511], {}),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_decode_behind_append_matches_oracle_and_plain_launch(name):
    G, Hkv, lengths, plan_kw = CASES[name]
    case, new, tr, pos, before = _step_case(lengths, G, Hkv, seed=len(name) * 7 + G)
    ref_out, ref_lse = _oracle_step(case, new, tr, pos, before)
    out1, lse1, info = _run_step(case, new, tr, pos, before, 1, plan_kw)
    if name.startswith("cluster"):
        assert info.cluster_size >= 2
    assert_parity(out1, ref_out, lse1, ref_lse, f"{name} behind the append")
    out0, lse0, _ = _run_step(case, new, tr, pos, before, 0, plan_kw)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1), "pdl changed the result"


def test_cascade_behind_append_matches_oracle_and_plain_launch():
    lengths = [700, 129, 3000, 256, 1500, 400, 2000, 900]
    case, new, tr, pos, before = _step_case(lengths, 8, 2, seed=41, shared_prefix_tokens=128,
                                            share_group=4)
    kw = dict(shared_prefix_tokens=128, share_group=4)
    ref_out, ref_lse = _oracle_step(case, new, tr, pos, before)
    out1, lse1, info = _run_step(case, new, tr, pos, before, 1, kw)
    assert info.cascade_units > 0
    assert_parity(out1, ref_out, lse1, ref_lse, "cascade behind the append")
    out0, lse0, _ = _run_step(case, new, tr, pos, before, 0, kw)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


@pytest.mark.parametrize("G,Hkv", [(4, 8), (32, 1)])
def test_layer_loop_on_one_workspace(G, Hkv):
    # Eight "layers" of decode on one bound workspace with split requests, each
    # run launched behind the previous run's merge kernel (which reads the
    # partial states the next run overwrites); every layer has its own q.
    case = W.custom_case([3000, 700, 4096, 64, 1500], num_qo_heads=G * Hkv, num_kv_heads=Hkv,
                         page_size=16, layout="NHD", seed=77 + G, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(5)
    qs = [torch.randn(tuple(case.q.shape), generator=g, device="cuda").to(torch.bfloat16)
          for _ in range(8)]
    tables = DeviceTables(case)
    results = []
    for pdl in (1, 0):
        plan = plan_case(case, pdl=pdl)
        assert plan.info.num_split_requests > 0
        ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
        oxd.oxd_plan_bind_workspace(plan, ws)
        outs = [torch.empty_like(case.q) for _ in qs]
        lses = [torch.empty(case.batch, case.num_qo_heads, device="cuda") for _ in qs]
        torch.cuda.synchronize()
        for q, o, ls in zip(qs, outs, lses):
            oxd.oxd_paged_decode_run(plan, q, case.k, case.v, tables.indptr, tables.indices,
                                     tables.last, case.sm_scale, o, ls, ws)
        torch.cuda.synchronize()
        assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
        results.append((outs, lses))
    for layer in range(len(qs)):
        assert torch.equal(results[0][0][layer], results[1][0][layer]), f"layer {layer}"
        assert torch.equal(results[0][1][layer], results[1][1][layer]), f"layer {layer}"
    t = case.tables
    for layer in (0, len(qs) - 1):
        ref_o, ref_l = oracle.paged_decode(
            W.bf16_bits(qs[layer]), W.bf16_bits(case.k), W.bf16_bits(case.v), t.indptr,
            t.indices, t.last_page_len, num_kv_heads=Hkv, page_size=16, layout=0,
            sm_scale=case.sm_scale)
        assert_parity(results[0][0][layer], ref_o, results[0][1][layer], ref_l, f"layer {layer}")
