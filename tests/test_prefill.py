"""Paged causal prefill through the C ABI against the f64 oracle (GPU).

Each case compares every output row (small cases) or sampled rows (the full
workloads, in the launch configuration the benchmark times) with the oracle:
|out - ref| <= 1.5e-2 + 1e-2 |ref|, |lse - ref| <= 1e-3. The cases cover
both tile sizes (256 rows in two halves of 128 on the two-half kernel, 128 rows
on the narrow kernel, and the planner's own pick), group sizes that fill a tile
exactly and ones that leave rows idle, the halves partly filled and a token's
heads straddling them,
scores that jump or drop by large amounts between 128-token stages and
at a column in each quarter of a stage (in some rows of a warp and not in
others, and past the F32 range),
zero and negative scales, NHD and HND pages of every page size, query counts
of zero, one, a tile, a
tile plus one and the whole cache, split and unsplit tiles, a bound workspace
(bitwise equal to unbound runs) and a CUDA-graph replay, repeated runs of one
plan (bitwise identical, status OK every time), and the device status for bad
page indices and tables that differ from the plan's.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_attn_gb300 as oxd
import workloads as W
from gpu_helpers import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oxd.build()
    oracle.build()


class Prefill:
    """A case on the device with its plan, tables, outputs and workspace."""

    def __init__(self, case: W.PrefillCase, max_splits=0, bind=False, tile_rows=0):
        t = case.tables
        self.case = case
        self.desc = oxd.make_prefill_desc(case.batch, case.num_qo_heads, case.num_kv_heads,
                                          case.page_size, case.layout, t.num_pages,
                                          max_splits=max_splits, tile_rows=tile_rows)
        self.plan = oxd.oxd_paged_prefill_plan(self.desc, case.qo_indptr, t.indptr,
                                               t.last_page_len)
        if tile_rows:
            assert self.plan.info.tile_rows == tile_rows
        dev = case.q.device
        self.qo = torch.as_tensor(case.qo_indptr, device=dev)
        self.indptr = torch.as_tensor(t.indptr, device=dev)
        self.indices = torch.as_tensor(t.indices, device=dev)
        self.last = torch.as_tensor(t.last_page_len, device=dev)
        self.out = torch.full_like(case.q, float("nan"))
        self.lse = torch.full(case.q.shape[:2], float("nan"), device=dev)
        self.ws = torch.empty(max(self.plan.workspace_bytes, 256), dtype=torch.uint8, device=dev)
        if bind:
            oxd.oxd_prefill_plan_bind_workspace(self.plan, self.ws)

    def run(self, out=None, lse=None, stream=None):
        c = self.case
        oxd.oxd_paged_prefill_run(self.plan, c.q, c.k, c.v, self.qo, self.indptr, self.indices,
                                  self.last, c.sm_scale, self.out if out is None else out,
                                  self.lse if lse is None else lse, self.ws, stream=stream)

    def status(self):
        return oxd.oxd_read_device_status(self.ws)


def oracle_rows(case: W.PrefillCase, rows=None):
    t = case.tables
    return oracle.paged_prefill(W.bf16_bits(case.q), W.bf16_bits(case.k), W.bf16_bits(case.v),
                                case.qo_indptr, t.indptr, t.indices, t.last_page_len,
                                num_kv_heads=case.num_kv_heads, page_size=case.page_size,
                                layout=0 if case.layout == "NHD" else 1, sm_scale=case.sm_scale,
                                rows=rows)


def check_all(run: Prefill, what):
    torch.cuda.synchronize()
    assert run.status() == oxd.OXD_DEVICE_OK, what
    ref_o, ref_l = oracle_rows(run.case)
    return assert_parity(run.out, ref_o, run.lse, ref_l, what)


@pytest.mark.parametrize("rows", [128, 256])
@pytest.mark.parametrize("G,Hkv", [(1, 4), (2, 4), (4, 8), (8, 2), (32, 1), (3, 2), (128, 1)])
def test_group_sizes(rows, G, Hkv):
    # tile_tokens = rows // G: 256, 128, 64, 32, 8, 85 (one row idle), 2 on 256-row
    # tiles; 128, 64, 32, 16, 4, 42 (two rows idle), 1 on 128-row tiles
    case = W.prefill_case((70, 1, 33), (300, 64, 33), G * Hkv, Hkv, 16, "NHD", seed=G,
                          device="cuda")
    run = Prefill(case, tile_rows=rows)
    run.run()
    check_all(run, f"G={G} rows {rows}")


@pytest.mark.parametrize("G,Hkv,q_lens,kv_lens,max_splits", [
    (1, 2, (200, 129), (300, 129), 1),      # both halves, the second partly filled
    (1, 2, (256,), (4096,), 64),            # last pieces wholly past the first half's rows
    (3, 2, (85, 43, 44), (900, 43, 500), 0),  # a token's heads straddle the halves
    (4, 8, (64, 40), (5000, 41), 0),        # a GQA4 tile: 32 tokens a half
    (128, 1, (2, 1, 3), (600, 1, 3), 0),    # one token a half
])
def test_tile_halves(G, Hkv, q_lens, kv_lens, max_splits):
    # A tile is 256 rows in two halves of 128 MMA rows; each half streams the
    # piece's stages up to its own last position and writes its own rows.
    case = W.prefill_case(q_lens, kv_lens, G * Hkv, Hkv, 16, "NHD", seed=G + len(q_lens),
                          device="cuda")
    run = Prefill(case, max_splits=max_splits, tile_rows=256)
    if max_splits == 64:
        assert run.plan.info.max_pieces > 8
    run.run()
    check_all(run, f"G={G} halves {q_lens}/{kv_lens}")


@pytest.mark.parametrize("rows", [128, 256])
@pytest.mark.parametrize("G,Hkv,layout", [(1, 32, "NHD"), (4, 16, "HND"), (8, 16, "NHD")])
def test_many_kv_heads(rows, G, Hkv, layout):
    # more KV heads than the workloads' eight: tiles of every KV head, pages
    # at large head strides
    case = W.prefill_case((40, 1, 130), (300, 64, 700), G * Hkv, Hkv, 16, layout, seed=Hkv,
                          device="cuda")
    run = Prefill(case, tile_rows=rows)
    run.run()
    check_all(run, f"G={G} Hkv={Hkv} {layout} rows {rows}")


@pytest.mark.parametrize("rows", [128, 256])
@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("ps", [8, 16, 32, 64])
def test_layouts_and_page_sizes(rows, layout, ps):
    case = W.prefill_case((5, 40, 64), (5, 77, 200), 16, 4, ps, layout, seed=ps, device="cuda")
    run = Prefill(case, tile_rows=rows)
    run.run()
    check_all(run, f"{layout} ps{ps} rows {rows}")


@pytest.mark.parametrize("q_lens,kv_lens", [
    ((0, 31, 32, 33), (10, 31, 500, 33)),       # no query token, whole-cache prefills
    ((1, 1, 1), (1, 1000, 65)),                 # decode-like rows
    ((64, 96), (64, 2000)),                     # two tiles over a long cache
])
@pytest.mark.parametrize("rows", [128, 256])
def test_query_counts(q_lens, kv_lens, rows):
    case = W.prefill_case(q_lens, kv_lens, 32, 8, 16, "NHD", seed=len(q_lens), device="cuda")
    run = Prefill(case, tile_rows=rows)
    run.run()
    check_all(run, f"q {q_lens} kv {kv_lens} rows {rows}")


@pytest.mark.parametrize("rows", [128, 256])
@pytest.mark.parametrize("max_splits", [1, 2, 5, 0])
def test_split_and_unsplit_tiles(rows, max_splits):
    case = W.prefill_case((32, 64, 7), (2048, 1024, 3000), 32, 8, 16, "HND", seed=11,
                          device="cuda")
    run = Prefill(case, max_splits=max_splits, tile_rows=rows)
    info = run.plan.info
    if max_splits == 1:
        assert info.num_split_tiles == 0 and info.launches_per_run == 1
    elif max_splits > 1:
        assert 1 < info.max_pieces <= max_splits
    run.run()
    check_all(run, f"max_splits {max_splits}")


@pytest.mark.parametrize("rows", [0, 256])
def test_pages_prefill_shape_and_scores_growing_along_the_cache(rows):
    # the pages' paged-prefill shape (128-row tiles when the planner picks), once
    # plain and once with keys that grow along the cache (the running maximum is
    # raised stage after stage)
    cfg = W.PREFILL_CONFIGS["prefill_gqa4_q32+64_kv256+1024_ps16_nhd"]
    case = W.make_prefill_case(cfg, device="cuda")
    run = Prefill(case, tile_rows=rows)
    assert run.plan.info.tile_rows == (rows or 128)
    run.run()
    check_all(run, cfg.name)
    t = case.tables
    for b in range(case.batch):
        L = int(t.lengths[b])
        ramp = torch.linspace(0.0, 3.0, L, device="cuda")
        for j in range(0, L, case.page_size):
            page = int(t.indices[t.indptr[b] + j // case.page_size])
            n = min(case.page_size, L - j)
            case.k[page, :n] = (case.k[page, :n].float() + ramp[j:j + n, None, None]).to(
                torch.bfloat16)
    run.run()
    check_all(run, "growing scores")


def _set_key_rows(case, b, positions, value):
    """Key rows of request b at the given cache positions, every KV head, set to
    the constant `value` (NHD pages)."""
    t = case.tables
    for pos in positions:
        page = int(t.indices[t.indptr[b] + pos // case.page_size])
        case.k[page, pos % case.page_size] = value


@pytest.mark.parametrize("rows", [128, 256])
@pytest.mark.parametrize("jump", [6.0, 3.0])
def test_scores_jumping_and_dropping_between_stages(rows, jump):
    # q = 1 in every column. Request 0: small keys, then a few keys of `jump`
    # in every column from stage 2 on (scores 128 jump / sqrt(128) above the
    # first stage's: 98 in log2 units for 6.0, far past the one-pass bound of
    # 2^64, so those stages fall back to two passes; 49 for 3.0, accepted with
    # the reference lagging). Request 1: the large keys in its first stage,
    # small ones after (terms of later stages near 2^-98 of the first).
    case = W.prefill_case((300, 200), (1000, 900), 8, 2, 16, "NHD", seed=17, device="cuda")
    case.q.fill_(1.0)
    case.k.mul_(0.05)
    _set_key_rows(case, 0, (300, 301, 640, 999), jump)
    _set_key_rows(case, 1, (5, 70), jump)
    run = Prefill(case, tile_rows=rows)
    run.run()
    check_all(run, f"key jump {jump} rows {rows}")


@pytest.mark.parametrize("rows", [128, 256])
@pytest.mark.parametrize("col", [0, 33, 70, 127])
def test_one_pass_refused_at_each_quarter_of_a_stage(rows, col):
    # Query heads alternate q = +1 and q = -1 in every column, so neighbouring
    # rows of a warp see opposite scores. Request 0's key at position 128 + col
    # (column `col` of its second stage, seen whole by every row) is 6.0 in
    # every column: +98 in log2 units above the first stage for the q = +1 rows
    # (past the one-pass bound of 2^64, so that stage takes two passes), -98
    # for the others; a second key of 16.0 at column 100 of the fourth
    # stage lifts the q = +1 rows by 164 more (a term past the F32 range in
    # one pass). Request 1 has the jump in its first stage only.
    case = W.prefill_case((300, 200), (1000, 900), 8, 2, 16, "NHD", seed=19, device="cuda")
    case.q.fill_(1.0)
    case.q[:, 1::2] = -1.0
    case.k.mul_(0.05)
    _set_key_rows(case, 0, (128 + col,), 6.0)
    _set_key_rows(case, 0, (384 + 100,), 16.0)
    _set_key_rows(case, 1, (col,), 6.0)
    run = Prefill(case, tile_rows=rows)
    run.run()
    check_all(run, f"refused chunk at column {col} rows {rows}")


@pytest.mark.parametrize("rows", [128, 256])
@pytest.mark.parametrize("shape", ["pages", "single_half", "split_hnd"])
def test_repeated_runs_are_bitwise_identical(rows, shape):
    # Sixty runs of one plan: every run's device status is OK and its out and
    # lse equal the first run's bit for bit (a race between the warps of a
    # tile, or a barrier phase taken a phase late, would show as a differing
    # or timed-out run).
    if shape == "pages":
        case = W.make_prefill_case(W.PREFILL_CONFIGS["prefill_gqa4_q32+64_kv256+1024_ps16_nhd"],
                                   device="cuda")
    elif shape == "single_half":
        case = W.prefill_case((16,) * 20, (2048,) * 20, 64, 8, 16, "NHD", seed=29, device="cuda")
    else:
        case = W.prefill_case((32, 64, 7), (2048, 1024, 3000), 32, 8, 16, "HND", seed=11,
                              device="cuda")
    run = Prefill(case, tile_rows=rows)
    first = None
    for i in range(60):
        run.out.fill_(float("nan"))
        run.run()
        torch.cuda.synchronize()
        assert run.status() == oxd.OXD_DEVICE_OK, f"run {i}"
        if first is None:
            first = (run.out.clone(), run.lse.clone())
        else:
            assert torch.equal(run.out, first[0]) and torch.equal(run.lse, first[1]), f"run {i}"
    ref_o, ref_l = oracle_rows(case)
    assert_parity(run.out, ref_o, run.lse, ref_l, f"{shape} rows {rows}")


@pytest.mark.parametrize("rows", [128, 256])
@pytest.mark.parametrize("scale", [0.0, -0.09])
def test_zero_and_negative_scales(rows, scale):
    # Any finite sm_scale: 0 weighs every visible cached token the same, a
    # negative one reverses the scores' order; the one-pass stages (taken
    # only for a positive scale) and the masked ones must agree with the oracle.
    case = W.prefill_case((70, 130, 5), (700, 1300, 400), 16, 4, 16, "NHD", seed=3,
                          device="cuda", sm_scale=scale)
    run = Prefill(case, tile_rows=rows)
    run.run()
    check_all(run, f"scale {scale} rows {rows}")


def test_single_half_tiles_many_runs():
    # Tiles of at most 128 rows run with two score buffers in one half. 160
    # such tiles of 64 stages each, run 12 times, the device status read after
    # every run (a barrier phase read one phase late would stall a run until
    # its wait limit and show here as OXD_DEVICE_WAIT_TIMEOUT); sampled rows of
    # the last run against the oracle.
    case = W.prefill_case((16,) * 20, (8192,) * 20, 64, 8, 16, "NHD", seed=23, device="cuda")
    run = Prefill(case, max_splits=1, tile_rows=256)
    assert run.plan.info.tile_tokens == 32 and run.plan.info.num_units == 160
    for i in range(12):
        run.run()
        torch.cuda.synchronize()
        assert run.status() == oxd.OXD_DEVICE_OK, f"run {i}"
    rng = np.random.default_rng(3)
    rows = [(int(tk), int(h)) for tk in rng.integers(0, 320, 24) for h in rng.integers(0, 64, 2)]
    ref_o, ref_l = oracle_rows(case, rows)
    ti = torch.as_tensor([r[0] for r in rows], device="cuda")
    hi = torch.as_tensor([r[1] for r in rows], device="cuda")
    assert_parity(run.out[ti, hi], ref_o, run.lse[ti, hi], ref_l, "single-half tiles")


@pytest.mark.parametrize("name", W.PREFILL_ORDER)
def test_full_workloads_sampled_rows(name):
    cfg = W.PREFILL_CONFIGS[name]
    case = W.make_prefill_case(cfg, device="cuda")
    run = Prefill(case, bind=True)
    run.run()
    torch.cuda.synchronize()
    assert run.status() == oxd.OXD_DEVICE_OK
    assert torch.isfinite(run.out.float()).all() and torch.isfinite(run.lse).all()
    rng = np.random.default_rng(5)
    nq = case.num_q_tokens
    # first and last query token of every request, plus random ones
    toks = set()
    for b in range(case.batch):
        q0, q1 = int(case.qo_indptr[b]), int(case.qo_indptr[b + 1])
        if q1 > q0:
            toks.update({q0, q1 - 1})
    toks.update(int(x) for x in rng.integers(0, nq, 24))
    rows = [(tk, int(h)) for tk in sorted(toks) for h in rng.integers(0, case.num_qo_heads, 3)]
    ref_o, ref_l = oracle_rows(case, rows)
    ti = torch.as_tensor([r[0] for r in rows], device="cuda")
    hi = torch.as_tensor([r[1] for r in rows], device="cuda")
    assert_parity(run.out[ti, hi], ref_o, run.lse[ti, hi], ref_l, name)


@pytest.mark.parametrize("rows", [128, 256])
def test_bound_workspace_matches_unbound_and_graph_replays(rows):
    case = W.prefill_case((40, 9), (900, 300), 32, 8, 16, "NHD", seed=21, device="cuda")
    plain = Prefill(case, tile_rows=rows)
    plain.run()
    bound = Prefill(case, bind=True, tile_rows=rows)
    bound.run()
    torch.cuda.synchronize()
    assert torch.equal(plain.out.view(torch.int16), bound.out.view(torch.int16))
    assert torch.equal(plain.lse.view(torch.int32), bound.lse.view(torch.int32))
    assert bound.plan.info.launches_per_run == 2  # this case splits
    graph = torch.cuda.CUDAGraph()
    out2 = torch.empty_like(bound.out)
    lse2 = torch.empty_like(bound.lse)
    with torch.cuda.graph(graph):
        bound.run(out2, lse2, stream=torch.cuda.current_stream())
    gen = torch.Generator(device="cuda").manual_seed(3)
    case.q.copy_(torch.randn(case.q.shape, generator=gen, device="cuda").to(torch.bfloat16))
    graph.replay()
    torch.cuda.synchronize()
    assert bound.status() == oxd.OXD_DEVICE_OK
    ref_o, ref_l = oracle_rows(case)
    assert_parity(out2, ref_o, lse2, ref_l, "graph replay")


@pytest.mark.parametrize("rows", [128, 256])
def test_guard_bands_untouched(rows):
    case = W.prefill_case((20, 3), (100, 50), 8, 2, 16, "NHD", seed=22, device="cuda")
    run = Prefill(case, tile_rows=rows)
    n = case.q.numel()
    big_out = torch.full((n + 2048,), -7.0, dtype=torch.bfloat16, device="cuda")
    out = big_out[1024:1024 + n].view(case.q.shape)
    m = case.q.shape[0] * case.q.shape[1]
    big_lse = torch.full((m + 128,), -7.0, device="cuda")
    lse = big_lse[64:64 + m].view(case.q.shape[:2])
    run.run(out, lse)
    torch.cuda.synchronize()
    assert (big_out[:1024] == -7.0).all() and (big_out[1024 + n:] == -7.0).all()
    assert (big_lse[:64] == -7.0).all() and (big_lse[64 + m:] == -7.0).all()
    run.out, run.lse = out, lse
    check_all(run, "guarded")


@pytest.mark.parametrize("rows", [128, 256])
def test_bad_page_and_changed_tables_are_reported(rows):
    case = W.prefill_case((16, 16), (200, 100), 8, 2, 16, "NHD", seed=23, device="cuda")
    run = Prefill(case, tile_rows=rows)
    saved = run.indices.clone()
    run.indices[3] = case.tables.num_pages + 5  # outside the pool: read as page 0
    run.run()
    torch.cuda.synchronize()
    assert run.status() == oxd.OXD_DEVICE_BAD_PAGE
    assert torch.isfinite(run.out.float()).all()
    run.indices.copy_(saved)
    run.last[1] = int(run.last[1]) - 1 if int(run.last[1]) > 1 else 2
    run.run()
    torch.cuda.synchronize()
    assert run.status() == oxd.OXD_DEVICE_PLAN_MISMATCH
    run.last.copy_(torch.as_tensor(case.tables.last_page_len, device="cuda"))
    run.run()
    check_all(run, "tables restored")
