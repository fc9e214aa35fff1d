"""Pipeline waits that run out: typed status, no fault, a clean next run (GPU).

Every wait inside the kernels is bounded ("Oxide Infer" README, "Providers":
typed device-status failures). A plan made with a wait limit of a few
nanoseconds (``wait_timeout_ns``) makes the first wait that is not already
satisfied give up: the CTA records OXD_DEVICE_WAIT_TIMEOUT, its warps leave
their loops, it waits for the copies (and tensor-core operations) it has
already issued, releases its tensor memory and returns. Nothing here faults,
traps or waits without a limit: the give-up path is the bounded one.

For every kernel family (CUDA-core decode, the 8- and 16-row mma.sync
decode, paired 16-row CTAs, the tcgen05 decode, clusters that merge in their
first CTA, the cascade's prefix tiles and the paged prefill) each case checks:
  * the status word reads OXD_DEVICE_WAIT_TIMEOUT and no CUDA error is raised;
  * no byte outside out, lse and the workspace changed (guard bands);
  * the next run with the default limit, on the same buffers, reads
    OXD_DEVICE_OK and matches the f64 oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_decode_attn_gb300 as oxd
import workloads as W
from gpu_helpers import DeviceTables, assert_parity, oracle_ref, plan_case

pytestmark = pytest.mark.gpu

SHORT_NS = 1


@pytest.fixture(scope="module", autouse=True)
def setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oxd.build()
    oracle.build()


class Guarded:
    """One device buffer holding out, lse and the workspace, each between
    4 KiB guard bands of 0xA5."""

    PAD = 4096

    def __init__(self, out_bytes, lse_bytes, ws_bytes):
        up = lambda x: (x + 255) // 256 * 256  # noqa: E731
        self.o0 = self.PAD
        self.l0 = up(self.o0 + out_bytes + self.PAD)
        self.w0 = up(self.l0 + lse_bytes + self.PAD)
        self.total = up(self.w0 + ws_bytes + self.PAD)
        self.sizes = (out_bytes, lse_bytes, ws_bytes)
        self.buf = torch.full((self.total,), 0xA5, dtype=torch.uint8, device="cuda")
        self.base = self.buf.data_ptr()

    def out(self, like):
        return self.buf[self.o0:self.o0 + self.sizes[0]].view(torch.bfloat16).view_as(like)

    def lse(self, shape):
        return self.buf[self.l0:self.l0 + self.sizes[1]].view(torch.float32).view(shape)

    @property
    def ws(self):
        return self.base + self.w0

    def assert_bands_intact(self, what):
        torch.cuda.synchronize()
        host = self.buf.cpu().numpy()
        mask = np.ones(self.total, bool)
        mask[self.o0:self.o0 + self.sizes[0]] = False
        mask[self.l0:self.l0 + self.sizes[1]] = False
        mask[self.w0:self.w0 + self.sizes[2]] = False
        assert (host[mask] == 0xA5).all(), f"{what}: a byte outside the outputs changed"


def _decode_case(lengths, G, Hkv, layout="NHD", ps=16, seed=0, **kw):
    return W.custom_case(lengths, num_qo_heads=G * Hkv, num_kv_heads=Hkv, page_size=ps,
                         layout=layout, seed=seed, device="cuda", **kw)


def _timeout_then_recover(case, what, **plan_kw):
    short = plan_case(case, wait_timeout_ns=SHORT_NS, **plan_kw)
    normal = plan_case(case, **plan_kw)
    assert short.workspace_bytes == normal.workspace_bytes
    g = Guarded(case.q.numel() * 2, case.batch * case.num_qo_heads * 4, normal.workspace_bytes)
    out = g.out(case.q)
    lse = g.lse((case.batch, case.num_qo_heads))
    tables = DeviceTables(case)

    def run(plan):
        oxd.oxd_paged_decode_run(plan, case.q, case.k, case.v, tables.indptr, tables.indices,
                                 tables.last, case.sm_scale, out, lse, g.ws,
                                 normal.workspace_bytes)

    run(short)
    torch.cuda.synchronize()  # raises if the kernels faulted
    code = oxd.oxd_read_device_status(g.ws)
    assert code == oxd.OXD_DEVICE_WAIT_TIMEOUT, \
        f"{what}: status {oxd.oxd_device_status_string(code)}"
    g.assert_bands_intact(what + ", timed-out run")
    run(normal)
    torch.cuda.synchronize()
    assert oxd.oxd_read_device_status(g.ws) == oxd.OXD_DEVICE_OK, what + ", next run"
    g.assert_bands_intact(what + ", next run")
    ref_o, ref_l = oracle_ref(case)
    assert_parity(out, ref_o, lse, ref_l, what + ", next run")
    return short.info


@pytest.mark.parametrize("G,Hkv,tensor_path,variant", [
    (1, 8, 0, 0),    # CUDA cores, G = 1
    (2, 4, 0, 1),    # CUDA cores, G = 2
    (4, 8, 0, 2),    # mma.sync, 8-row tiles
    (16, 2, 0, 3),   # mma.sync, 16-row tiles
    (32, 1, 1, 4),   # mma.sync, pairs of 16-row CTAs
    (32, 1, 0, 5),   # tcgen05, scores and output in tensor memory
])
@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_decode_wait_timeout_is_reported_and_recovered(G, Hkv, tensor_path, variant, layout):
    case = _decode_case([3000, 700, 1500, 64, 2048], G, Hkv, layout, seed=90 + G)
    info = _timeout_then_recover(case, f"decode G{G} {layout}", tensor_path=tensor_path)
    assert info.kernel_variant == variant


@pytest.mark.parametrize("G,Hkv", [(1, 8), (4, 8)])
def test_cluster_decode_wait_timeout_is_reported_and_recovered(G, Hkv):
    case = _decode_case([512, 200, 1000], G, Hkv, seed=95 + G, extra_pages=2)
    info = _timeout_then_recover(case, f"cluster decode G{G}")
    assert info.cluster_size >= 2


@pytest.mark.parametrize("G,Hkv", [(4, 8), (32, 1)])
def test_cascade_wait_timeout_is_reported_and_recovered(G, Hkv):
    lengths = [700, 129, 3000, 256, 1500, 400, 2000, 900]
    case = _decode_case(lengths, G, Hkv, seed=97 + G, shared_prefix_tokens=128, share_group=4)
    info = _timeout_then_recover(case, f"cascade G{G}", shared_prefix_tokens=128, share_group=4)
    assert info.cascade_units > 0


@pytest.mark.parametrize("rows", [128, 256])
@pytest.mark.parametrize("max_splits", [1, 0])
def test_prefill_wait_timeout_is_reported_and_recovered(max_splits, rows):
    case = W.make_prefill_case(W.PrefillConfig(
        name="timeout", q_lens=(64, 300, 1), kv_lens=(1024, 2000, 700), num_qo_heads=32,
        num_kv_heads=8, page_size=16, layout="NHD", seed=99), device="cuda")
    t = case.tables
    plans = [oxd.oxd_paged_prefill_plan(
        oxd.make_prefill_desc(case.batch, case.num_qo_heads, case.num_kv_heads, case.page_size,
                              case.layout, t.num_pages, max_splits=max_splits,
                              wait_timeout_ns=ns, tile_rows=rows), case.qo_indptr, t.indptr,
        t.last_page_len)
        for ns in (SHORT_NS, 0)]
    ws_bytes = max(plans[1].workspace_bytes, 256)
    g = Guarded(case.q.numel() * 2, case.q.shape[0] * case.q.shape[1] * 4, ws_bytes)
    out = g.out(case.q)
    lse = g.lse(case.q.shape[:2])
    dev = case.q.device
    qo = torch.as_tensor(case.qo_indptr, device=dev)
    indptr = torch.as_tensor(t.indptr, device=dev)
    indices = torch.as_tensor(t.indices, device=dev)
    last = torch.as_tensor(t.last_page_len, device=dev)
    for i, plan in enumerate(plans):
        oxd.oxd_paged_prefill_run(plan, case.q, case.k, case.v, qo, indptr, indices, last,
                                  case.sm_scale, out, lse, g.ws, ws_bytes)
        torch.cuda.synchronize()
        code = oxd.oxd_read_device_status(g.ws)
        assert code == (oxd.OXD_DEVICE_WAIT_TIMEOUT if i == 0 else oxd.OXD_DEVICE_OK), \
            oxd.oxd_device_status_string(code)
        g.assert_bands_intact(f"prefill run {i}")
    ref_o, ref_l = oracle.paged_prefill(
        W.bf16_bits(case.q), W.bf16_bits(case.k), W.bf16_bits(case.v), case.qo_indptr,
        t.indptr, t.indices, t.last_page_len, num_kv_heads=case.num_kv_heads,
        page_size=case.page_size, layout=0, sm_scale=case.sm_scale)
    assert_parity(out, ref_o, lse, ref_l, "prefill after a timed-out run")
