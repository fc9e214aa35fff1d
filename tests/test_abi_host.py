"""C-ABI checks that need no GPU: exported symbols, planning, operand rejection.

Planning with ``num_sms > 0`` makes no CUDA call, and ``oxd_paged_decode_run``
/ ``oxd_merge_states`` check every operand before touching the device, so the
negative cases run here with fake (never dereferenced) addresses. These are
the pages' "lifetime and negative gates" ("Oxide Infer" README, "Evidence
before claims") and the "checked span, alignment, alias, and capacity rules"
of "Providers".
"""
import ctypes
import math
import os
import re

import numpy as np
import pytest

import paged_kv_decode_attn_gb300 as oxd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE = 1 << 40  # fake device addresses, far apart and 256-byte aligned


@pytest.fixture(scope="module", autouse=True)
def built():
    oxd.build()


def declared_functions():
    with open(os.path.join(ROOT, "include", "oxd.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(oxd_[a-z_]+)\s*\(", text)))


def test_every_declared_function_is_exported():
    names = declared_functions()
    assert set(names) == set(oxd.EXPORTED_SYMBOLS)
    L = ctypes.CDLL(oxd.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n
    assert oxd.oxd_version().startswith("oxd ")


def test_status_strings_cover_every_code():
    seen = {oxd.oxd_status_string(s) for s in range(10)}
    assert len(seen) == 10 and "unknown status" not in seen
    assert oxd.oxd_status_string(99) == "unknown status"
    assert {oxd.oxd_device_status_string(c) for c in range(4)} >= {"ok"}


def host_plan(lengths, Hq=32, Hkv=8, ps=16, layout="NHD", num_pages=None, **kw):
    lengths = np.asarray(lengths, np.int64)
    pages = (lengths + ps - 1) // ps
    indptr = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
    last = (lengths - (pages - 1) * ps).astype(np.int32)
    desc = oxd.make_desc(len(lengths), Hq, Hkv, ps, layout,
                         int(pages.sum()) if num_pages is None else num_pages,
                         num_sms=kw.pop("num_sms", 152), **kw)
    return oxd.oxd_paged_decode_plan(desc, indptr, last), indptr, last


# ------------------------------------------------------------------ planning

def test_balanced_partition_spreads_work_over_the_grid():
    plan, indptr, _ = host_plan([4096] * 32)
    info = plan.info
    assert info.kernel_variant == 2                       # G = 4: tensor-core variant
    assert info.grid_ctas == 152 * info.ctas_per_sm       # every resident CTA gets a share
    total_pages = int(indptr[-1]) * 8
    assert abs(info.chunk_pages - total_pages / info.grid_ctas) <= 1  # share per CTA, pages
    assert info.num_work_items >= info.grid_ctas
    assert info.num_split_requests > 0 and info.max_chunks > 1
    # partial states: one [G][128] f32 block + [G] lse per split piece
    part = info.num_slots * 4 * 128 * 4 + info.num_slots * 4 * 4
    assert info.workspace_bytes >= part
    assert info.workspace_bytes == plan.workspace_bytes
    assert info.launches_per_run == 2          # decode + merge of the split streams
    assert info.upload_bytes == 0              # the work list fits the parameter buffer
    assert info.total_kv_tokens == 32 * 4096


def test_short_batch_is_not_split_when_splitting_is_off():
    plan, _, _ = host_plan([100, 5000, 17], max_splits=1)
    info = plan.info
    assert info.num_split_requests == 0 and info.num_work_items == 3 * 8
    assert info.launches_per_run == 1 and info.num_slots == 0
    assert info.grid_ctas == 3 * 8


def test_tiny_batch_uses_one_stage_per_cta_at_least():
    plan, _, _ = host_plan([512], Hq=8, Hkv=8)   # 8 streams of 32 pages
    info = plan.info
    assert 32 <= info.grid_ctas <= 8 * 32 // 4    # at least one 64-token stage per CTA
    assert info.num_work_items >= info.grid_ctas


def test_small_batch_merges_inside_clusters():
    # 8 streams of 32 pages: each cut into 8 pieces on the 8 CTAs of a cluster,
    # whose first CTA merges them (no merge launch)
    plan, _, _ = host_plan([512], Hq=8, Hkv=8)
    info = plan.info
    assert info.cluster_size == 8 and info.grid_ctas == 8 * 8
    assert info.launches_per_run == 1 and info.num_slots == 64
    assert info.num_split_requests == 8 and info.max_chunks == 8
    # the shortest stream bounds the cluster size (3 pages: clusters of 3)
    plan, _, _ = host_plan([40, 300, 129], Hq=4, Hkv=2)
    assert plan.info.cluster_size == 3 and plan.info.grid_ctas == 3 * 2 * 3


@pytest.mark.parametrize("lengths,Hq,Hkv,kw", [
    ([4096] * 32, 32, 8, {}),                 # many streams: line partition + merge kernel
    ([32768], 32, 8, {}),                     # few long streams: pieces would be too long
    ([512, 1, 300], 8, 8, {}),                # a one-page stream: no pieces to spread
    ([512], 8, 8, {"force_splits": 4}),       # the caller fixed the split
    ([512], 8, 8, {"max_splits": 2}),
    ([4000, 4000], 32, 1, {}),                # 32-head groups: other kernels
    ([512], 96, 8, {}),                       # groups of 12: states do not fit rank 0
])
def test_cluster_merge_only_where_it_pays(lengths, Hq, Hkv, kw):
    plan, _, _ = host_plan(lengths, Hq=Hq, Hkv=Hkv, **kw)
    assert plan.info.cluster_size == 0


@pytest.mark.parametrize("lengths,H", [([1], 8), ([1], 32), ([16], 32), ([100] * 4, 32)])
def test_short_streams_get_a_cta_each_and_need_no_merge(lengths, H):
    # one-token or one-page contexts: every (request, head) stream on its own
    # CTA (they used to queue on the few CTAs their token count asked for)
    plan, _, _ = host_plan(lengths, Hq=H, Hkv=H)
    info = plan.info
    assert info.grid_ctas == len(lengths) * H == info.num_work_items
    assert info.launches_per_run == 1 and info.num_split_requests == 0
    assert info.cluster_size == 0


def test_many_short_streams_share_the_resident_ctas():
    plan, _, _ = host_plan([40] * 100, Hq=8, Hkv=8)   # 800 streams of 3 pages
    info = plan.info
    assert info.grid_ctas == 152 * info.ctas_per_sm and info.num_work_items == 800
    assert info.launches_per_run == 1


@pytest.mark.parametrize("force", [1, 2, 3, 7])
def test_forced_splits(force):
    lengths = [1, 16, 17, 100, 1000]
    plan, indptr, _ = host_plan(lengths, force_splits=force)
    pages = np.diff(indptr)
    chunks = np.minimum(force, pages)
    info = plan.info
    assert info.num_work_items == chunks.sum() * 8
    assert info.num_split_requests == int((chunks > 1).sum()) * 8   # split (request, head) streams
    assert info.num_slots == int(chunks[chunks > 1].sum()) * 8
    assert info.max_chunks == chunks.max()


def test_long_work_lists_are_uploaded():
    plan, _, _ = host_plan([64] * 600, Hq=8, Hkv=8, max_splits=1)
    info = plan.info
    assert info.num_work_items == 600 * 8 and info.upload_bytes >= 600 * 8 * 16
    assert info.launches_per_run == 1


def test_max_splits_caps_chunks():
    plan, _, _ = host_plan([32768] * 4, Hq=32, Hkv=1, ps=64, max_splits=3)
    assert plan.info.max_chunks <= 3


@pytest.mark.parametrize("G,variant", [(1, 0), (2, 1), (3, 2), (8, 2), (9, 3), (16, 3),
                                       (17, 5), (32, 5)])
def test_variant_follows_group_size(G, variant):
    plan, _, _ = host_plan([64], Hq=G * 2, Hkv=2)
    assert plan.info.kernel_variant == variant
    # the mma.sync path for large groups: pairs of 16-row CTAs
    plan, _, _ = host_plan([64], Hq=G * 2, Hkv=2, tensor_path=1)
    assert plan.info.kernel_variant == (4 if G > 16 else variant)


BAD_DESC = {
    "batch0": dict(batch=0),
    "hq_not_multiple": dict(num_qo_heads=30),
    "head_dim": dict(head_dim=64),
    "page_size": dict(page_size=12),
    "group_64": dict(num_qo_heads=64, num_kv_heads=1),
    "layout": dict(layout=2),
    "num_pages0": dict(num_pages=0),
    "group_without_prefix": dict(share_group=4),
    "prefix_not_page_multiple": dict(shared_prefix_tokens=24, share_group=4),
    "prefix_group_of_one": dict(shared_prefix_tokens=32, share_group=1),
    "negative_prefix": dict(shared_prefix_tokens=-16, share_group=2),
    "negative_splits": dict(max_splits=-1),
    "tensor_path": dict(tensor_path=2),
    "pdl": dict(pdl=2),
    "negative_wait": dict(wait_timeout_ns=-5),
}


@pytest.mark.parametrize("name", sorted(BAD_DESC))
def test_bad_descriptors_are_rejected(name):
    desc = oxd.make_desc(2, 32, 8, 16, "NHD", 10, num_sms=152)
    mod = BAD_DESC[name]
    for k, v in mod.items():
        setattr(desc, k, v)
    expect = oxd.OXD_ERR_UNSUPPORTED if name in ("head_dim", "page_size", "group_64") \
        else oxd.OXD_ERR_INVALID_ARGUMENT
    indptr = np.array([0, 5, 10], np.int32)
    last = np.array([16, 3], np.int32)
    if name == "batch0":
        indptr, last = np.array([0], np.int32), np.zeros(0, np.int32)
    with pytest.raises(oxd.OxdError) as e:
        oxd.oxd_paged_decode_plan(desc, indptr, last)
    assert e.value.status == expect


@pytest.mark.parametrize("indptr,last", [
    ([0, 0, 5], [3, 3]),        # empty request
    ([0, 5, 4], [3, 3]),        # decreasing indptr
    ([0, 2, 5], [0, 3]),        # last_page_len 0
    ([0, 2, 5], [3, 17]),       # last_page_len > page_size
    ([-1, 2, 5], [3, 3]),       # negative start
])
def test_bad_block_tables_are_rejected(indptr, last):
    desc = oxd.make_desc(2, 32, 8, 16, "NHD", 10, num_sms=152)
    with pytest.raises(oxd.OxdError) as e:
        oxd.oxd_paged_decode_plan(desc, np.array(indptr, np.int32), np.array(last, np.int32))
    assert e.value.status == oxd.OXD_ERR_INVALID_ARGUMENT


def test_null_arguments_to_plan():
    L = oxd.lib()
    desc = oxd.make_desc(1, 8, 8, 16, "NHD", 4, num_sms=152)
    h, ws = ctypes.c_void_p(), ctypes.c_size_t()
    ind = np.array([0, 4], np.int32)
    last = np.array([16], np.int32)
    assert L.oxd_paged_decode_plan(None, ind.ctypes.data, last.ctypes.data, 0,
                                   ctypes.byref(h), ctypes.byref(ws)) == 1
    assert L.oxd_paged_decode_plan(ctypes.byref(desc), None, last.ctypes.data, 0,
                                   ctypes.byref(h), ctypes.byref(ws)) == 1
    assert h.value is None  # nothing written on error


# ------------------------------------------------------------------ run operand checks

def fake_operands(plan, B, Hq, num_pages, ps=16, Hkv=8):
    rows = B * Hq
    pool = num_pages * ps * Hkv * 128 * 2
    step = 1 << 36
    return dict(q=BASE, k_pages=BASE + step, v_pages=BASE + 2 * step, indptr=BASE + 3 * step,
                indices=BASE + 4 * step, last_page_len=BASE + 5 * step, sm_scale=0.088,
                out=BASE + 6 * step, lse=BASE + 7 * step, workspace=BASE + 8 * step,
                workspace_bytes=plan.workspace_bytes, stream=0), rows, pool


def run_status(plan, **ops):
    L = oxd.lib()
    return L.oxd_paged_decode_run(
        oxd._handle(plan), ops["q"], ops["k_pages"], ops["v_pages"], ops["indptr"],
        ops["indices"], ops["last_page_len"], ctypes.c_float(ops["sm_scale"]), ops["out"],
        ops["lse"], ops["workspace"], ops["workspace_bytes"], ops["stream"])


@pytest.mark.parametrize("case,expect", [
    ("q_misaligned", oxd.OXD_ERR_ALIGNMENT),
    ("k_misaligned", oxd.OXD_ERR_ALIGNMENT),
    ("out_misaligned", oxd.OXD_ERR_ALIGNMENT),
    ("lse_misaligned", oxd.OXD_ERR_ALIGNMENT),
    ("ws_misaligned", oxd.OXD_ERR_ALIGNMENT),
    ("indices_misaligned", oxd.OXD_ERR_ALIGNMENT),
    ("ws_small", oxd.OXD_ERR_WORKSPACE_TOO_SMALL),
    ("out_is_q", oxd.OXD_ERR_ALIAS),
    ("out_in_kpool", oxd.OXD_ERR_ALIAS),
    ("lse_in_out", oxd.OXD_ERR_ALIAS),
    ("ws_over_indices", oxd.OXD_ERR_ALIAS),
    ("ws_over_out", oxd.OXD_ERR_ALIAS),
    ("null_q", oxd.OXD_ERR_INVALID_ARGUMENT),
    ("null_ws", oxd.OXD_ERR_INVALID_ARGUMENT),
    ("nan_scale", oxd.OXD_ERR_INVALID_ARGUMENT),
    ("inf_scale", oxd.OXD_ERR_INVALID_ARGUMENT),
])
def test_run_rejects_bad_operands_before_enqueue(case, expect):
    plan, indptr, _ = host_plan([300, 50], Hq=32, Hkv=8)
    ops, rows, pool = fake_operands(plan, 2, 32, int(indptr[-1]))
    if case == "q_misaligned":
        ops["q"] += 8
    elif case == "k_misaligned":
        ops["k_pages"] += 2
    elif case == "out_misaligned":
        ops["out"] += 4
    elif case == "lse_misaligned":
        ops["lse"] += 2
    elif case == "ws_misaligned":
        ops["workspace"] += 128
    elif case == "indices_misaligned":
        ops["indices"] += 1
    elif case == "ws_small":
        ops["workspace_bytes"] -= 256
    elif case == "out_is_q":
        ops["out"] = ops["q"]
    elif case == "out_in_kpool":
        ops["out"] = ops["k_pages"] + pool - 256
    elif case == "lse_in_out":
        ops["lse"] = ops["out"] + rows * 256 - 64
    elif case == "ws_over_indices":
        ops["workspace"] = ops["indices"] - 256
    elif case == "ws_over_out":
        ops["workspace"] = ops["out"]
    elif case == "null_q":
        ops["q"] = None
    elif case == "null_ws":
        ops["workspace"] = None
    elif case == "nan_scale":
        ops["sm_scale"] = math.nan
    elif case == "inf_scale":
        ops["sm_scale"] = math.inf
    assert run_status(plan, **ops) == expect


def test_adjacent_buffers_are_not_aliases():
    # out ends exactly where lse starts: touching is not overlapping. The
    # call then passes every host check and only fails at the device step.
    plan, indptr, _ = host_plan([40], Hq=8, Hkv=8)
    ops, rows, pool = fake_operands(plan, 1, 8, int(indptr[-1]))
    ops["lse"] = ops["out"] + rows * 256
    assert run_status(plan, **ops) not in (oxd.OXD_ERR_ALIAS, oxd.OXD_ERR_ALIGNMENT,
                                           oxd.OXD_ERR_INVALID_ARGUMENT)


def test_destroyed_plan_is_refused():
    plan, indptr, _ = host_plan([40], Hq=8, Hkv=8)
    ops, _, _ = fake_operands(plan, 1, 8, int(indptr[-1]))
    h = plan.handle
    plan.destroy()
    assert oxd.lib().oxd_plan_destroy(h) == oxd.OXD_ERR_PLAN_MISMATCH
    ops["workspace_bytes"] = 1 << 20
    L = oxd.lib()
    st = L.oxd_paged_decode_run(h, ops["q"], ops["k_pages"], ops["v_pages"], ops["indptr"],
                                ops["indices"], ops["last_page_len"], ctypes.c_float(1.0),
                                ops["out"], ops["lse"], ops["workspace"], 1 << 20, 0)
    assert st == oxd.OXD_ERR_PLAN_MISMATCH
    info = oxd.PlanInfo()
    assert L.oxd_plan_get_info(h, ctypes.byref(info)) == oxd.OXD_ERR_PLAN_MISMATCH


def test_bind_workspace_checks_arguments_before_any_cuda_call():
    plan, _, _ = host_plan([300, 50], Hq=32, Hkv=8)
    L = oxd.lib()
    ws = BASE
    big = plan.workspace_bytes
    assert L.oxd_plan_bind_workspace(plan.handle, None, big, None) == \
        oxd.OXD_ERR_INVALID_ARGUMENT
    assert L.oxd_plan_bind_workspace(plan.handle, ws + 16, big, None) == oxd.OXD_ERR_ALIGNMENT
    assert L.oxd_plan_bind_workspace(plan.handle, ws, big - 1, None) == \
        oxd.OXD_ERR_WORKSPACE_TOO_SMALL
    # a plan made for no device (num_sms given) cannot be bound to device memory
    assert L.oxd_plan_bind_workspace(plan.handle, ws, big, None) == oxd.OXD_ERR_PLAN_MISMATCH
    h = plan.handle
    plan.destroy()
    assert L.oxd_plan_bind_workspace(h, ws, big, None) == oxd.OXD_ERR_PLAN_MISMATCH


def test_timing_events_must_come_in_pairs():
    plan, _, _ = host_plan([40], Hq=8, Hkv=8)
    L = oxd.lib()
    assert L.oxd_plan_set_timing_events(plan.handle, 0x1000, None) == 1
    assert L.oxd_plan_set_timing_events(plan.handle, None, None) == 0


@pytest.mark.parametrize("case,expect", [
    ("ok_shape_bad_D", oxd.OXD_ERR_INVALID_ARGUMENT),
    ("zero_N", oxd.OXD_ERR_INVALID_ARGUMENT),
    ("v_misaligned", oxd.OXD_ERR_ALIGNMENT),
    ("out_misaligned", oxd.OXD_ERR_ALIGNMENT),
    ("out_over_v", oxd.OXD_ERR_ALIAS),
    ("s_out_over_s", oxd.OXD_ERR_ALIAS),
    ("s_out_over_out", oxd.OXD_ERR_ALIAS),
])
def test_merge_rejects_bad_operands(case, expect):
    N, S, H, D = 3, 4, 8, 128
    v, s, o, so = BASE, BASE + (1 << 36), BASE + (2 << 36), BASE + (3 << 36)
    if case == "ok_shape_bad_D":
        D = 126
    elif case == "zero_N":
        N = 0
    elif case == "v_misaligned":
        v += 4
    elif case == "out_misaligned":
        o += 2
    elif case == "out_over_v":
        o = v + 64
    elif case == "s_out_over_s":
        so = s
    elif case == "s_out_over_out":
        so = o + 16
    st = oxd.lib().oxd_merge_states(v, s, N, S, H, D, o, so, None)
    assert st == expect


# ------------------------------------------------------------------ rope + append

def _append_args(T=4, B=2, Hq=8, Hkv=2, num_pages=16):
    """Fake, far-apart device addresses for every operand of oxd_rope_append."""
    names = ["q", "k", "v", "token_request", "positions", "indptr", "indices",
             "page_refcount", "q_out", "k_pages", "v_pages", "workspace"]
    return {n: BASE + (i + 1) * (1 << 36) for i, n in enumerate(names)}


def _append_status(desc, a, ws_bytes=256):
    L = oxd.lib()
    return L.oxd_rope_append(ctypes.byref(desc), a["q"], a["k"], a["v"], a["token_request"],
                             a["positions"], a["indptr"], a["indices"], a["page_refcount"],
                             a["q_out"], a["k_pages"], a["v_pages"], a["workspace"], ws_bytes,
                             None)


@pytest.mark.parametrize("case,expect", [
    ("no_tokens", oxd.OXD_ERR_INVALID_ARGUMENT),
    ("theta_one", oxd.OXD_ERR_INVALID_ARGUMENT),
    ("theta_nan", oxd.OXD_ERR_INVALID_ARGUMENT),
    ("reserved", oxd.OXD_ERR_INVALID_ARGUMENT),
    ("no_indices", oxd.OXD_ERR_INVALID_ARGUMENT),
    ("indices_over_pool", oxd.OXD_ERR_ALIAS),
    ("head_dim", oxd.OXD_ERR_UNSUPPORTED),
    ("page_size", oxd.OXD_ERR_UNSUPPORTED),
    ("q_misaligned", oxd.OXD_ERR_ALIGNMENT),
    ("workspace_misaligned", oxd.OXD_ERR_ALIGNMENT),
    ("workspace_small", oxd.OXD_ERR_WORKSPACE_TOO_SMALL),
    ("q_out_over_k", oxd.OXD_ERR_ALIAS),
    ("q_out_inside_q", oxd.OXD_ERR_ALIAS),
    ("pool_over_refcount", oxd.OXD_ERR_ALIAS),
    ("k_pool_is_v_pool", oxd.OXD_ERR_ALIAS),
    ("null_indices", oxd.OXD_ERR_INVALID_ARGUMENT),
])
def test_rope_append_rejects_bad_operands(case, expect):
    desc = oxd.make_rope_append_desc(4, 2, 8, 2, 16, "NHD", 16, 8)
    a = _append_args()
    ws_bytes = 256
    if case == "no_tokens":
        desc.num_tokens = 0
    elif case == "theta_one":
        desc.rope_theta = 1.0
    elif case == "theta_nan":
        desc.rope_theta = float("nan")
    elif case == "reserved":
        desc.reserved[0] = 1
    elif case == "no_indices":
        desc.num_indices = 0
    elif case == "head_dim":
        desc.head_dim = 64
    elif case == "page_size":
        desc.page_size = 12
    elif case == "q_misaligned":
        a["q"] += 8
    elif case == "workspace_misaligned":
        a["workspace"] += 16
    elif case == "workspace_small":
        ws_bytes = 255
    elif case == "q_out_over_k":
        a["q_out"] = a["k"]
    elif case == "q_out_inside_q":
        a["q_out"] = a["q"] + 256
    elif case == "pool_over_refcount":
        a["k_pages"] = a["page_refcount"]
    elif case == "k_pool_is_v_pool":
        a["v_pages"] = a["k_pages"]
    elif case == "null_indices":
        a["indices"] = None
    elif case == "indices_over_pool":
        a["k_pages"] = a["indices"]
    assert _append_status(desc, a, ws_bytes) == expect


def test_rope_append_accepts_in_place_query():
    # q_out == q passes every host check (the call then fails only for want
    # of a device on this machine)
    desc = oxd.make_rope_append_desc(4, 2, 8, 2, 16, "HND", 16, 8)
    a = _append_args()
    a["q_out"] = a["q"]
    assert _append_status(desc, a) not in (oxd.OXD_ERR_ALIAS, oxd.OXD_ERR_ALIGNMENT,
                                           oxd.OXD_ERR_INVALID_ARGUMENT)


# ------------------------------------------------------------------ causal prefill

def prefill_plan(q_lens, kv_lens, Hq=32, Hkv=8, ps=16, num_sms=152, **kw):
    kv = np.asarray(kv_lens, np.int64)
    pages = (kv + ps - 1) // ps
    indptr = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
    last = (kv - (pages - 1) * ps).astype(np.int32)
    qo = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    desc = oxd.make_prefill_desc(len(kv), Hq, Hkv, ps, kw.pop("layout", "NHD"),
                                 kw.pop("num_pages", int(pages.sum())), num_sms=num_sms, **kw)
    return oxd.oxd_paged_prefill_plan(desc, qo, indptr, last), qo, indptr, last


def test_prefill_plan_tiles_and_pieces():
    # the pages' shape: 32 + 64 query tokens, GQA4, 8 KV heads. 256-row tiles
    # would give 2 x 8 + 8 x 8 = 80 stages of 128 tokens, fewer than 152 SMs:
    # the planner picks 128-row tiles (32 tokens) on the narrow kernel.
    plan, *_ = prefill_plan((32, 64), (256, 1024))
    i = plan.info
    assert i.tile_rows == 128 and i.ctas_per_sm == 2
    assert i.tile_tokens == 32 and i.num_tiles == (1 + 2) * 8
    assert i.total_q_tokens == 96 and i.total_kv_tokens == 1280
    assert i.causal_pairs == 32 * 224 + 32 * 33 // 2 + 64 * 960 + 64 * 65 // 2
    assert i.num_units > i.num_tiles and i.launches_per_run == 2  # split to fill the GPU
    assert i.num_merge_rows == i.num_split_tiles * 32 * 4 or i.num_split_tiles < i.num_tiles
    one, *_ = prefill_plan((32, 64), (256, 1024), max_splits=1)
    assert one.info.num_units == 24 and one.info.launches_per_run == 1
    capped, *_ = prefill_plan((32, 64), (256, 1024), max_splits=2)
    assert capped.info.max_pieces == 2
    # the same shape on 256-row tiles (64 tokens, two halves), asked for
    wide, *_ = prefill_plan((32, 64), (256, 1024), tile_rows=256)
    w = wide.info
    assert w.tile_rows == 256 and w.ctas_per_sm == 1
    assert w.tile_tokens == 64 and w.num_tiles == (1 + 1) * 8
    # every tile split: one merged row per (query token, query head)
    assert w.num_split_tiles == w.num_tiles and w.num_merge_rows == (32 + 64) * 32
    one, *_ = prefill_plan((32, 64), (256, 1024), max_splits=1, tile_rows=256)
    assert one.info.num_units == 16 and one.info.launches_per_run == 1
    # enough tiles to fill the GPU: 256-row tiles, no split
    big, *_ = prefill_plan((2048,) * 8, [4096] * 8)
    assert big.info.tile_rows == 256
    assert big.info.num_split_tiles == 0 and big.info.num_units == 8 * 32 * 8


def test_prefill_tile_size_choice():
    # 256-row tiles once their 128-token stages reach the SM count, unless asked
    # otherwise; 152 SMs, GQA4 with 8 KV heads: one 64-token tile of a request
    # with 2 * 128 * k cached tokens gives 8 * 2k stages
    small, *_ = prefill_plan((64,), (128 * 18,))     # 8 x 18 = 144 stages
    assert small.info.tile_rows == 128
    large, *_ = prefill_plan((64,), (128 * 19,))     # 8 x 19 = 152 stages
    assert large.info.tile_rows == 256
    fewer, *_ = prefill_plan((64,), (128 * 19,), num_sms=153)
    assert fewer.info.tile_rows == 128
    forced, *_ = prefill_plan((64,), (128 * 19,), tile_rows=128)
    assert forced.info.tile_rows == 128 and forced.info.tile_tokens == 32


@pytest.mark.parametrize("rows,G,T", [(256, 1, 256), (256, 2, 128), (256, 3, 85), (256, 8, 32),
                                      (256, 32, 8), (256, 128, 2), (128, 1, 128), (128, 2, 64),
                                      (128, 3, 42), (128, 8, 16), (128, 32, 4), (128, 128, 1)])
def test_prefill_tile_tokens_follow_group(rows, G, T):
    plan, *_ = prefill_plan((T * 2 + 1,), (1000,), Hq=G, Hkv=1, tile_rows=rows)
    assert plan.info.tile_rows == rows
    assert plan.info.tile_tokens == T and plan.info.num_tiles == 3


@pytest.mark.parametrize("name", ["q_above_kv", "qo_start", "qo_decreasing", "no_query",
                                  "group_too_big", "page_size", "head_dim", "negative_wait",
                                  "heads_not_divisible", "tile_rows", "reserved"])
def test_prefill_bad_plans_are_rejected(name):
    q_lens, kv_lens, kw = (4, 4), (10, 10), {}
    expect = oxd.OXD_ERR_INVALID_ARGUMENT
    if name == "q_above_kv":
        q_lens = (4, 11)
    elif name == "no_query":
        q_lens = (0, 0)
    elif name == "group_too_big":
        kw = dict(Hq=256, Hkv=1)
        expect = oxd.OXD_ERR_UNSUPPORTED
    elif name == "heads_not_divisible":
        kw = dict(Hq=12, Hkv=8)
    kv = np.asarray(kv_lens)
    pages = (kv + 15) // 16
    indptr = np.concatenate([[0], np.cumsum(pages)]).astype(np.int32)
    last = (kv - (pages - 1) * 16).astype(np.int32)
    qo = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    desc = oxd.make_prefill_desc(2, kw.get("Hq", 8), kw.get("Hkv", 2), 16, "NHD", 4, num_sms=152)
    if name == "qo_start":
        qo = qo + 1
    elif name == "qo_decreasing":
        qo = np.array([0, 5, 4], np.int32)
    elif name == "page_size":
        desc.page_size = 12
        expect = oxd.OXD_ERR_UNSUPPORTED
    elif name == "head_dim":
        desc.head_dim = 64
        expect = oxd.OXD_ERR_UNSUPPORTED
    elif name == "negative_wait":
        desc.wait_timeout_ns = -1
    elif name == "tile_rows":
        desc.tile_rows = 64
    elif name == "reserved":
        desc.reserved = 1
    with pytest.raises(oxd.OxdError) as e:
        oxd.oxd_paged_prefill_plan(desc, qo, indptr, last)
    assert e.value.status == expect


def _prefill_status(plan, B, Hq, Hkv, num_pages, nq, ps=16, **over):
    step = 1 << 36
    ops = dict(q=BASE, k=BASE + step, v=BASE + 2 * step, qo=BASE + 3 * step,
               indptr=BASE + 4 * step, indices=BASE + 5 * step, last=BASE + 6 * step,
               scale=0.088, out=BASE + 7 * step, lse=BASE + 8 * step, ws=BASE + 9 * step,
               ws_bytes=plan.workspace_bytes)
    ops.update(over)
    return oxd.lib().oxd_paged_prefill_run(
        oxd._handle(plan), ops["q"], ops["k"], ops["v"], ops["qo"], ops["indptr"],
        ops["indices"], ops["last"], ctypes.c_float(ops["scale"]), ops["out"], ops["lse"],
        ops["ws"], ops["ws_bytes"], None)


@pytest.mark.parametrize("case,expect", [
    ("q_misaligned", oxd.OXD_ERR_ALIGNMENT),
    ("out_misaligned", oxd.OXD_ERR_ALIGNMENT),
    ("ws_misaligned", oxd.OXD_ERR_ALIGNMENT),
    ("qo_misaligned", oxd.OXD_ERR_ALIGNMENT),
    ("ws_small", oxd.OXD_ERR_WORKSPACE_TOO_SMALL),
    ("out_is_q", oxd.OXD_ERR_ALIAS),
    ("out_in_vpool", oxd.OXD_ERR_ALIAS),
    ("lse_in_out", oxd.OXD_ERR_ALIAS),
    ("ws_over_qo", oxd.OXD_ERR_ALIAS),
    ("null_indices", oxd.OXD_ERR_INVALID_ARGUMENT),
    ("nan_scale", oxd.OXD_ERR_INVALID_ARGUMENT),
    ("host_only_plan", oxd.OXD_ERR_PLAN_MISMATCH),
])
def test_prefill_run_rejects_bad_operands_before_enqueue(case, expect):
    plan, qo, *_ = prefill_plan((20, 5), (100, 40), Hq=8, Hkv=2)
    step = 1 << 36
    over = {
        "q_misaligned": dict(q=BASE + 8), "out_misaligned": dict(out=BASE + 7 * step + 4),
        "ws_misaligned": dict(ws=BASE + 9 * step + 128), "qo_misaligned": dict(qo=BASE + 3 * step + 2),
        "ws_small": dict(ws_bytes=plan.workspace_bytes - 256), "out_is_q": dict(out=BASE),
        "out_in_vpool": dict(out=BASE + 2 * step + 4096), "lse_in_out": dict(lse=BASE + 7 * step + 256),
        "ws_over_qo": dict(ws=BASE + 3 * step - 256), "null_indices": dict(indices=0),
        "nan_scale": dict(scale=float("nan")), "host_only_plan": {},
    }[case]
    assert _prefill_status(plan, 2, 8, 2, 9, 25, **over) == expect


def test_prefill_plan_lifetime():
    plan, *_ = prefill_plan((3,), (3,))
    h = plan.handle
    ws = (ctypes.c_uint8 * 512)()
    # a host-only plan cannot be bound (checked before any CUDA call)
    assert oxd.lib().oxd_prefill_plan_bind_workspace(h, BASE, plan.workspace_bytes, None) == \
        oxd.OXD_ERR_PLAN_MISMATCH
    assert oxd.lib().oxd_prefill_plan_set_timing_events(h, BASE, None) == \
        oxd.OXD_ERR_INVALID_ARGUMENT
    plan.destroy()
    assert oxd.lib().oxd_prefill_plan_destroy(h) == oxd.OXD_ERR_PLAN_MISMATCH
    info = oxd.PrefillPlanInfo()
    assert oxd.lib().oxd_prefill_plan_get_info(h, ctypes.byref(info)) == oxd.OXD_ERR_PLAN_MISMATCH
    del ws


# ------------------------------------------------------------------ cascade decode planning

def test_cascade_plan_counts_groups_and_shared_tokens():
    # 3 groups of 4; group 1 has two requests no longer than the prefix, group
    # 2 has only one longer request (decoded whole)
    lengths = [300, 500, 129, 1000,  100, 128, 700, 900,  64, 50, 2000, 120]
    plan, _, _ = host_plan(lengths, Hq=32, Hkv=8, ps=16, shared_prefix_tokens=128,
                           share_group=4)
    i = plan.info
    assert i.cascade_requests == 4 + 2
    assert i.cascade_units == (1 + 1) * 8          # one chunk per sharing group, x 8 KV heads
    assert i.shared_kv_tokens == (4 - 1) * 128 + (2 - 1) * 128
    assert i.launches_per_run == 3
    plain, _, _ = host_plan(lengths, Hq=32, Hkv=8, ps=16)
    assert plain.info.cascade_units == 0 and plain.info.shared_kv_tokens == 0


def test_cascade_groups_wider_than_a_tile_are_chunked():
    # prefix tiles hold 128 rows (the narrow kernel): G = 8 -> 16 requests per
    # tile; a group of 40 needs three chunks
    plan, _, _ = host_plan([5000] * 40, Hq=64, Hkv=8, ps=16, shared_prefix_tokens=1024,
                           share_group=40)
    assert plan.info.cascade_units == 3 * 8 and plan.info.cascade_requests == 40
    assert plan.info.shared_kv_tokens == (40 - 3) * 1024


# ------------------------------------------------------------------ encoding limits
# A work unit packs the request index in 19 bits and the KV head in the 12 bits
# above it (plus one bit for the row half), and page indices are int32: the
# planner accepts everything up to those limits and refuses the first value past.

def _one_page_each(B):
    return np.arange(B + 1, dtype=np.int32), np.ones(B, np.int32)


def test_largest_batch_is_planned():
    B = (1 << 19) - 1
    indptr, last = _one_page_each(B)
    desc = oxd.make_desc(B, 1, 1, 16, "NHD", B, num_sms=152)
    plan = oxd.oxd_paged_decode_plan(desc, indptr, last)
    info = plan.info
    assert info.total_kv_tokens == B
    assert info.num_split_requests == 0


def test_batch_past_the_unit_encoding_is_refused():
    B = 1 << 19
    indptr, last = _one_page_each(B)
    desc = oxd.make_desc(B, 1, 1, 16, "NHD", B, num_sms=152)
    with pytest.raises(oxd.OxdError) as e:
        oxd.oxd_paged_decode_plan(desc, indptr, last)
    assert e.value.status == oxd.OXD_ERR_UNSUPPORTED


@pytest.mark.parametrize("hkv,ok", [((1 << 12) - 1, True), (1 << 12, False)])
def test_kv_head_count_limit(hkv, ok):
    indptr, last = np.array([0, 2], np.int32), np.array([5], np.int32)
    desc = oxd.make_desc(1, hkv, hkv, 16, "NHD", 4, num_sms=152)
    if ok:
        plan = oxd.oxd_paged_decode_plan(desc, indptr, last)
        assert plan.info.total_kv_tokens == 21
    else:
        with pytest.raises(oxd.OxdError) as e:
            oxd.oxd_paged_decode_plan(desc, indptr, last)
        assert e.value.status == oxd.OXD_ERR_UNSUPPORTED


@pytest.mark.parametrize("num_pages,ok", [((1 << 31) - 1, True), (1 << 31, False)])
def test_pool_size_limit(num_pages, ok):
    indptr, last = np.array([0, 3], np.int32), np.array([16], np.int32)
    desc = oxd.make_desc(1, 8, 8, 16, "NHD", num_pages, num_sms=152)
    if ok:
        assert oxd.oxd_paged_decode_plan(desc, indptr, last).info.total_kv_tokens == 48
    else:
        with pytest.raises(oxd.OxdError) as e:
            oxd.oxd_paged_decode_plan(desc, indptr, last)
        assert e.value.status == oxd.OXD_ERR_UNSUPPORTED
