"""GPU parity of the CUDA path (through the C ABI) against the f64 oracle.

Covers the "Paged batch decode" device matrix named on the "FlashInfer parity
matrix" page ("Admitted attention matrix"): MHA, MQA, GQA, mixed lengths, page
order, read-only page reuse; NHD and HND layouts ("Domain coverage"); split
partitions with their merge; invalid-page rejection as a device status. The
five full-size workloads are checked on sampled heads in the launch
configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_attn_gb300 as oxd
import workloads as W
from gpu_helpers import (DeviceTables, assert_parity, gpu_heads, oracle_ref, plan_case,
                         run_decode)

pytestmark = pytest.mark.gpu

LENGTHS = [1, 15, 16, 17, 63, 64, 65, 200, 777]  # one token .. several stages, ragged tails


@pytest.fixture(scope="module", autouse=True)
def setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oxd.build()
    oracle.build()


def small_case(G, layout="NHD", ps=16, lengths=LENGTHS, Hkv=2, seed=0, sigma=1.0, **kw):
    return W.custom_case(lengths, num_qo_heads=G * Hkv, num_kv_heads=Hkv, page_size=ps,
                         layout=layout, seed=seed + 100 * G + ps, sigma=sigma, device="cuda",
                         **kw)


# ------------------------------------------------------------------ small parity sweep

@pytest.mark.parametrize("ps", [8, 16, 32, 64])
@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("G", [1, 2, 3, 4, 8, 12, 16, 24, 32])
def test_parity_small(G, layout, ps):
    case = small_case(G, layout, ps)
    ref_out, ref_lse = oracle_ref(case)
    out, lse, plan, _ = run_decode(case)
    assert_parity(out, ref_out, lse, ref_lse, f"G{G} {layout} ps{ps} auto")
    out1, lse1, _, _ = run_decode(case, max_splits=1)
    assert_parity(out1, ref_out, lse1, ref_lse, f"G{G} {layout} ps{ps} unsplit")


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("G,Hkv", [(1, 64), (2, 32), (4, 16), (8, 16), (32, 4)])
def test_many_kv_heads(G, Hkv, layout):
    # KV heads beyond the workloads' eight (a 64-head MHA model, GQA with 16
    # or 32 KV heads, MQA-like groups over four KV heads): a head's rows and
    # pages at large head strides, auto and unsplit plans
    case = small_case(G, layout, 16, lengths=[900, 1, 33, 2500], Hkv=Hkv, seed=14)
    ref_out, ref_lse = oracle_ref(case)
    out, lse, _, _ = run_decode(case)
    assert_parity(out, ref_out, lse, ref_lse, f"G{G} Hkv{Hkv} {layout} auto")
    out1, lse1, _, _ = run_decode(case, max_splits=1)
    assert_parity(out1, ref_out, lse1, ref_lse, f"G{G} Hkv{Hkv} {layout} unsplit")


@pytest.mark.parametrize("ps", [16, 64])
@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("G", [17, 32])
def test_both_tensor_paths_for_large_groups(G, layout, ps):
    # groups over 16 heads: tcgen05 (default) and mma.sync on paired CTAs
    case = small_case(G, layout, ps)
    ref_out, ref_lse = oracle_ref(case)
    for path in (0, 1):
        for force in (0, 3):
            out, lse, plan, _ = run_decode(case, tensor_path=path, force_splits=force)
            assert plan.info.kernel_variant == (5 if path == 0 else 4)
            assert_parity(out, ref_out, lse, ref_lse, f"G{G} {layout} ps{ps} path {path}")


@pytest.mark.parametrize("G,force", [(32, 0), (32, 2), (4, 0), (1, 0)])
def test_scores_growing_along_the_sequence(G, force):
    # Keys grow with their position, so each row's running maximum keeps
    # rising by many units of log2 from stage to stage: the online softmax
    # rescales again and again (the tcgen05 path only when the rise exceeds
    # 2^8, which this case forces every few stages).
    Hkv = 1 if G == 32 else 8
    case = small_case(G, "NHD", 16, lengths=[1500, 700, 129], Hkv=Hkv, seed=12,
                      sm_scale=0.5)
    t = case.tables
    ps = case.page_size
    for b in range(case.batch):
        for lp in range(int(t.indptr[b + 1] - t.indptr[b])):
            phys = int(t.indices[t.indptr[b] + lp])
            case.k[phys] *= 1.0 + lp * ps / 64.0
    ref_out, ref_lse = oracle_ref(case)
    out, lse, plan, _ = run_decode(case, force_splits=force)
    assert_parity(out, ref_out, lse, ref_lse, f"growing scores G{G} force {force}")


@pytest.mark.parametrize("path", [0, 1])
def test_many_short_units_per_cta_large_group(path):
    # 600 MQA requests of 1..300 tokens, planned for one SM: every CTA runs
    # hundreds of units back to back (query tile reloads, per-unit epilogues,
    # split and whole units interleaved)
    rng = np.random.default_rng(5)
    lengths = [int(x) for x in rng.integers(1, 301, 600)]
    case = small_case(32, "NHD", 16, lengths=lengths, Hkv=1, seed=6)
    ref_out, ref_lse = oracle_ref(case)
    out, lse, plan, ws = run_decode(case, num_sms=1, tensor_path=path)
    assert plan.info.grid_ctas <= 4 and plan.info.num_work_items >= 600
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
    assert_parity(out, ref_out, lse, ref_lse, f"many units path {path}")


@pytest.mark.parametrize("G", [1, 4, 32])
def test_forced_splits_agree(G):
    case = small_case(G, "NHD", 16, lengths=[1000, 333, 64, 1, 129], seed=3)
    ref_out, ref_lse = oracle_ref(case)
    outs = []
    for force in (1, 2, 3, 7, 8, 9, 64):
        out, lse, plan, _ = run_decode(case, force_splits=force)
        assert plan.info.max_chunks == min(force, 63)
        assert plan.info.launches_per_run == (2 if force > 1 else 1)
        assert_parity(out, ref_out, lse, ref_lse, f"force {force}")
        outs.append(out.float())
        # the same plan on a bound workspace: bitwise the same, run after run
        ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
        oxd.oxd_plan_bind_workspace(plan, ws)
        for _ in range(2):
            out_b, lse_b, _, _ = run_decode(case, plan=plan, workspace=ws)
            assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
            assert torch.equal(out_b.view(torch.int16), out.view(torch.int16)), f"bound {force}"
            assert torch.equal(lse_b.view(torch.int32), lse.view(torch.int32))
    for o in outs[1:]:
        d = (o - outs[0]).abs()
        assert (d <= 1.5e-2 + 1e-2 * outs[0].abs()).all()


def test_without_lse_output():
    case = small_case(4)
    ref_out, _ = oracle_ref(case)
    out, lse, _, _ = run_decode(case, want_lse=False)
    assert lse is None
    assert_parity(out, ref_out, what="no lse")


# ------------------------------------------------------------------ invariants

@pytest.mark.parametrize("G", [1, 2, 4, 32])
@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_one_token_context_returns_that_v_bitwise(G, layout):
    case = small_case(G, layout, 16, lengths=[1, 1, 1, 1], seed=5)
    out, lse, _, _ = run_decode(case)
    t = case.tables
    for b in range(case.batch):
        page = int(t.indices[t.indptr[b]])
        for hq in range(case.num_qo_heads):
            h = hq // G
            v0 = case.v[page, 0, h] if layout == "NHD" else case.v[page, h, 0]
            assert torch.equal(out[b, hq], v0), (b, hq)
    _, ref_lse = oracle_ref(case)
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= 1e-3


@pytest.mark.parametrize("G", [1, 8])
def test_identical_keys_give_mean_of_v(G):
    case = small_case(G, "NHD", 16, lengths=[300, 17, 64], seed=6)
    key = torch.randn(case.num_kv_heads, 128, device="cuda").to(torch.bfloat16)
    case.k[:] = key.view(1, 1, -1, 128)
    out, lse, _, _ = run_decode(case)
    t = case.tables
    for b in range(case.batch):
        ids = torch.as_tensor(t.indices[t.indptr[b]:t.indptr[b + 1]], device="cuda")
        L = int(t.lengths[b])
        for hq in range(case.num_qo_heads):
            V = case.v[ids][:, :, hq // G].reshape(-1, 128)[:L].double()
            mean = V.mean(0)
            assert ((out[b, hq].double() - mean).abs() <= 1.5e-2 + 1e-2 * mean.abs()).all()
    ref_out, ref_lse = oracle_ref(case)
    assert_parity(out, ref_out, lse, ref_lse, "identical keys")


@pytest.mark.parametrize("G", [1, 4, 32])
def test_page_permutation_leaves_output_bitwise_unchanged(G):
    case = small_case(G, "HND", 16, lengths=[500, 77, 16, 240], seed=7)
    out0, lse0, _, _ = run_decode(case)
    perm = np.random.default_rng(1).permutation(case.tables.num_pages)
    inv = torch.as_tensor(np.argsort(perm), device="cuda")
    case.k = case.k[inv].contiguous()
    case.v = case.v[inv].contiguous()
    case.tables.indices = perm[case.tables.indices].astype(np.int32)
    out1, lse1, _, _ = run_decode(case)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


@pytest.mark.parametrize("name", ["fma_g1", "mma8_g4", "mma16_g16", "tcgen05_g32", "paired_g32",
                                  "cluster_g1", "cascade_g8"])
def test_runs_are_bitwise_deterministic(name):
    # Sixty runs of one plan on one workspace, split streams included: the
    # device status is OK after every run and out and lse equal the first
    # run's bit for bit (a race between a CTA's warps, or a barrier phase taken
    # a phase late, would show as a differing or timed-out run).
    G = int(name.split("_g")[1])
    lengths = [2000, 1, 700, 45, 3000, 129]
    kw = {}
    if name == "cluster_g1":
        lengths = [511]
    elif name == "tcgen05_g32":
        kw = dict(tensor_path=0)
    elif name == "paired_g32":
        kw = dict(tensor_path=1)
    elif name == "cascade_g8":
        lengths = [700, 129, 3000, 256, 1500, 400, 2000, 900]
    extra = dict(shared_prefix_tokens=128, share_group=4) if name == "cascade_g8" else {}
    case = small_case(G, "NHD", 16, lengths=lengths, Hkv=8 if G == 1 else 2, seed=8, **extra)
    plan = plan_case(case, **kw, **extra)
    if name == "cluster_g1":
        assert plan.info.cluster_size >= 2
    if name == "cascade_g8":
        assert plan.info.cascade_units > 0
    tables = DeviceTables(case)
    out = torch.empty_like(case.q)
    lse = torch.empty(case.batch, case.num_qo_heads, device="cuda")
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device="cuda")
    first = None
    for i in range(60):
        out.fill_(float("nan"))
        run_decode(case, plan=plan, tables=tables, workspace=ws, out=out, lse=lse)
        assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK, f"run {i}"
        if first is None:
            first = (out.clone(), lse.clone())
        else:
            assert torch.equal(out, first[0]) and torch.equal(lse, first[1]), f"run {i}"
    ref_out, ref_lse = oracle_ref(case)
    assert_parity(out, ref_out, lse, ref_lse, name)


@pytest.mark.parametrize("scale", [0.0, -0.09])
@pytest.mark.parametrize("name", ["fma_g1", "mma8_g4", "mma16_g16", "tcgen05_g32", "paired_g32",
                                  "cluster_g1", "cascade_g8"])
def test_zero_and_negative_scales(name, scale):
    # sm_scale is any finite number: 0 gives every visible token the same
    # weight (out = the mean of V, lse = ln L), a negative scale reverses the
    # ranking of the scores; no kernel may take the maximum of raw scores as
    # the maximum of scaled ones then.
    G = int(name.split("_g")[1])
    lengths = [2000, 1, 700, 45, 3000, 129]
    kw = {}
    if name == "cluster_g1":
        lengths = [511]
    elif name == "tcgen05_g32":
        kw = dict(tensor_path=0)
    elif name == "paired_g32":
        kw = dict(tensor_path=1)
    elif name == "cascade_g8":
        lengths = [700, 129, 3000, 256, 1500, 400, 2000, 900]
    extra = dict(shared_prefix_tokens=128, share_group=4) if name == "cascade_g8" else {}
    case = small_case(G, "NHD", 16, lengths=lengths, Hkv=8 if G == 1 else 2, seed=12,
                      sm_scale=scale, **extra)
    plan = plan_case(case, **kw, **extra)
    out, lse, _, ws = run_decode(case, plan=plan)
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
    ref_out, ref_lse = oracle_ref(case)
    assert_parity(out, ref_out, lse, ref_lse, f"{name} scale {scale}")


@pytest.mark.parametrize("G", [1, 2, 8, 32])
def test_nan_in_unused_tail_slots_is_ignored(G):
    case = small_case(G, "NHD", 16, lengths=[19, 5, 33, 100], seed=9)
    out0, lse0, _, _ = run_decode(case)
    t = case.tables
    for b in range(case.batch):
        page = int(t.indices[t.indptr[b + 1] - 1])
        n = int(t.last_page_len[b])
        case.k[page, n:] = float("nan")
        case.v[page, n:] = float("inf")
    out1, lse1, _, _ = run_decode(case)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_shared_pages_are_read_only_and_reused():
    case = small_case(8, "NHD", 16, lengths=[1024, 700, 1500, 2000, 1024, 64, 1100, 300],
                      shared_prefix_tokens=1024, share_group=4, seed=10)
    assert case.tables.shared_pages > 0
    k0, v0 = case.k.clone(), case.v.clone()
    ref_out, ref_lse = oracle_ref(case)
    out, lse, _, _ = run_decode(case)
    assert_parity(out, ref_out, lse, ref_lse, "shared prefix")
    assert torch.equal(case.k, k0) and torch.equal(case.v, v0)


def test_runs_on_the_callers_stream():
    case = small_case(4, "NHD", 16, seed=11)
    ref_out, ref_lse = oracle_ref(case)
    s = torch.cuda.Stream()
    plan = plan_case(case)
    tables = DeviceTables(case)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        out = torch.empty_like(case.q)
        lse = torch.empty(case.batch, case.num_qo_heads, device="cuda")
        ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
        oxd.oxd_paged_decode_run(plan, case.q, case.k, case.v, tables.indptr, tables.indices,
                                 tables.last, case.sm_scale, out, lse, ws, stream=s)
    s.synchronize()
    assert_parity(out, ref_out, lse, ref_lse, "side stream")


def test_guard_bands_around_outputs_are_untouched():
    case = small_case(4, "NHD", 16, seed=12)
    plan = plan_case(case)
    pad = 4096
    n_out = case.q.numel() * 2
    n_lse = case.batch * case.num_qo_heads * 4
    ws_bytes = plan.workspace_bytes
    total = pad + n_out + pad + n_lse + pad + ws_bytes + pad
    total = (total + 255) // 256 * 256
    buf = torch.full((total,), 0xA5, dtype=torch.uint8, device="cuda")
    o0 = pad
    l0 = (o0 + n_out + pad + 255) // 256 * 256
    w0 = (l0 + n_lse + pad + 255) // 256 * 256
    base = buf.data_ptr()
    tables = DeviceTables(case)
    oxd.oxd_paged_decode_run(plan, case.q, case.k, case.v, tables.indptr, tables.indices,
                             tables.last, case.sm_scale, base + o0, base + l0, base + w0,
                             ws_bytes)
    torch.cuda.synchronize()
    host = buf.cpu().numpy()
    mask = np.ones(total, bool)
    mask[o0:o0 + n_out] = False
    mask[l0:l0 + n_lse] = False
    mask[w0:w0 + ws_bytes] = False
    assert (host[mask] == 0xA5).all()
    out = buf[o0:o0 + n_out].view(torch.bfloat16).view_as(case.q)
    ref_out, _ = oracle_ref(case)
    assert_parity(out, ref_out, what="guard bands")


# ------------------------------------------------------------------ device-side failures

def test_bad_page_index_reports_status_without_fault():
    case = small_case(4, "NHD", 16, lengths=[300, 40], seed=13)
    plan = plan_case(case)
    tables = DeviceTables(case)
    tables.indices[3] = case.tables.num_pages + 7   # out of the pool
    tables.indices[-1] = -2
    out, lse, _, ws = run_decode(case, plan=plan, tables=tables)
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_BAD_PAGE
    assert torch.isfinite(out.float()).all()
    # the next run with good tables resets the status word
    good = DeviceTables(case)
    out2, lse2, _, _ = run_decode(case, plan=plan, tables=good, workspace=ws)
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
    ref_out, ref_lse = oracle_ref(case)
    assert_parity(out2, ref_out, lse2, ref_lse, "after recovery")


def test_device_tables_differing_from_the_plan_report_status():
    case = small_case(4, "NHD", 16, lengths=[300, 40], seed=14)
    plan = plan_case(case)
    tables = DeviceTables(case)
    tables.last[1] = 1 if int(case.tables.last_page_len[1]) != 1 else 2
    _, _, _, ws = run_decode(case, plan=plan, tables=tables)
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_PLAN_MISMATCH


def test_workspace_too_small_is_refused_on_device_run():
    case = small_case(4, seed=15)
    plan = plan_case(case)
    tables = DeviceTables(case)
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    with pytest.raises(oxd.OxdError) as e:
        oxd.oxd_paged_decode_run(plan, case.q, case.k, case.v, tables.indptr, tables.indices,
                                 tables.last, case.sm_scale, torch.empty_like(case.q), None, ws,
                                 plan.workspace_bytes - 256)
    assert e.value.status == oxd.OXD_ERR_WORKSPACE_TOO_SMALL


# ------------------------------------------------------------------ state merge

@pytest.mark.parametrize("S", [1, 2, 5, 16, 17, 32, 40])
def test_merge_states_matches_oracle(S):
    N, H, D = 3, 4, 128
    g = torch.Generator(device="cuda").manual_seed(S)
    v = torch.randn(N, S, H, D, generator=g, device="cuda")
    s = torch.randn(N, S, H, generator=g, device="cuda") * 3
    s[0, 0, 1] = float("-inf")
    s[1, :, 2] = float("-inf")        # a head with no weight at all
    out = torch.empty(N, H, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(N, H, device="cuda")
    oxd.oxd_merge_states(v, s, N, S, H, D, out, lse)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.merge_states_batched(v.double().cpu().numpy(),
                                               s.double().cpu().numpy())
    assert_parity(out, ref_o, what="merge")
    lg = lse.cpu().numpy()
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(lg), fin)
    assert np.abs(lg[fin] - ref_l[fin]).max() <= 1e-4
    assert (out[1, 2] == 0).all() and lg[1, 2] == -np.inf


def test_merge_of_split_partials_equals_decode():
    # Attention states of two halves of each request (oracle partials), merged
    # on the GPU, match the unsplit decode.
    case = small_case(4, "NHD", 16, lengths=[100, 257], seed=16)
    args = (W.bf16_bits(case.q), W.bf16_bits(case.k), W.bf16_bits(case.v),
            case.tables.indptr, case.tables.indices, case.tables.last_page_len)
    B, H = case.batch, case.num_qo_heads
    v = np.zeros((B, 2, H, 128))
    s = np.zeros((B, 2, H))
    for b in range(B):
        L = int(case.tables.lengths[b])
        for h in range(H):
            for i, (a, e) in enumerate([(0, L // 3), (L // 3, L)]):
                v[b, i, h], s[b, i, h] = oracle.partial_state(
                    *args, num_kv_heads=case.num_kv_heads, page_size=16, layout=0,
                    sm_scale=case.sm_scale, b=b, hq=h, tok_begin=a, tok_end=e)
    vt = torch.as_tensor(v, dtype=torch.float32, device="cuda")
    st = torch.as_tensor(s, dtype=torch.float32, device="cuda")
    out = torch.empty(B, H, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, H, device="cuda")
    oxd.oxd_merge_states(vt, st, B, 2, H, 128, out, lse)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle_ref(case)
    assert_parity(out, ref_out, lse, ref_lse, "merged halves")


# ------------------------------------------------------------------ full-size workloads

@pytest.mark.slow
@pytest.mark.parametrize("name", W.CONFIG_ORDER)
def test_full_size_workloads_on_every_head(name):
    # Each of the five workloads at full size, in the benchmark's launch
    # configuration (the plan bound to its workspace), element by element on
    # every head (B * Hq rows of 128 and B * Hq LSEs) against the f64 oracle;
    # a workload that declares shared prefixes also on the cascade plan.
    cfg = W.CONFIGS[name]
    case = W.make_case(cfg, device="cuda")
    ref_out, ref_lse = oracle_ref(case)
    assert ref_out.shape == (case.batch, case.num_qo_heads, 128)
    plans = [{}]
    if cfg.shared_prefix_tokens > 0:
        plans.append(dict(shared_prefix_tokens=cfg.shared_prefix_tokens,
                          share_group=cfg.share_group))
    for kw in plans:
        plan = plan_case(case, **kw)
        ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
        oxd.oxd_plan_bind_workspace(plan, ws)
        out, lse, plan, ws = run_decode(case, plan=plan, workspace=ws)
        assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
        if kw:
            assert plan.info.cascade_units > 0
        assert_parity(out, ref_out, lse, ref_lse, f"{name} {'cascade' if kw else 'plain'}")


@pytest.mark.slow
def test_largest_batch_the_work_units_encode():
    # 2^19 - 1 requests, the most a work unit's 19-bit request field holds, of
    # 1..24 tokens each (one to three pages of 8): about 1.05 M pages, 4.3 GB of
    # K and V. Checked on sampled heads, always including the last requests.
    B = (1 << 19) - 1
    lengths = np.random.default_rng(77).integers(1, 25, size=B).tolist()
    case = W.custom_case(lengths, num_qo_heads=2, num_kv_heads=1, page_size=8, layout="NHD",
                         seed=77, device="cuda")
    plan = plan_case(case)
    assert plan.info.num_work_items == B
    ws = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device="cuda")
    oxd.oxd_plan_bind_workspace(plan, ws)
    out, lse, plan, ws = run_decode(case, plan=plan, workspace=ws)
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
    rng = np.random.default_rng(78)
    heads = {(int(b), int(h)) for b, h in zip(rng.integers(0, B, 40), rng.integers(0, 2, 40))}
    heads |= {(0, 0), (B - 1, 0), (B - 1, 1), (B - 2, 1), ((1 << 18), 0)}
    heads = sorted(heads)
    ref_out, ref_lse = oracle_ref(case, heads=heads)
    go, gl = gpu_heads(out, lse, heads)
    assert_parity(go, ref_out, gl, ref_lse, "largest batch")


@pytest.mark.slow
@pytest.mark.parametrize("G", [1, 8, 32])
def test_one_long_request_split_over_every_cta(G):
    # One request of 2^21 tokens (32768 pages of 64, 1 GB of K and V) is cut into
    # one piece a resident CTA (304 states a row), so the merge takes its
    # multi-pass path for rows of more than 32 states.
    case = W.custom_case([1 << 21], num_qo_heads=G, num_kv_heads=1, page_size=64, layout="NHD",
                         seed=80 + G, device="cuda")
    plan = plan_case(case)
    assert plan.info.num_split_requests == 1 and plan.info.max_chunks > 32
    out, lse, plan, ws = run_decode(case, plan=plan)
    assert oxd.oxd_read_device_status(ws) == oxd.OXD_DEVICE_OK
    heads = [(0, h) for h in (range(G) if G <= 8 else (0, 1, 15, 16, 30, 31))]
    ref_out, ref_lse = oracle_ref(case, heads=heads)
    go, gl = gpu_heads(out, lse, heads)
    assert_parity(go, ref_out, gl, ref_lse, f"one long request G={G}")
