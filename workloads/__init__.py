"""Seeded synthetic inputs for paged-KV decode attention.

This module is the only thing the CUDA path and the oracle share: it draws
block tables (CSR ``indptr``/``indices``/``last_page_len``) and bf16 q/K/V
values from seeded generators. It holds none of the attention arithmetic.

Recipe (stated once, used everywhere):

* KV lengths are drawn with ``numpy.random.default_rng(seed)`` from the
  distribution of the workload; pages per request ``P_b = ceil(L_b / ps)``;
  ``last_page_len_b = L_b - (P_b - 1) * ps`` (so it is ``ps``, not 0, when
  ``ps`` divides ``L_b``).
* Physical pages: every logical page gets its own physical page, except the
  shared-prefix pages of a sharing group (the first ``prefix/ps`` pages of each
  request in a group of ``share_group`` consecutive requests map to the same
  physical pages). The pool holds exactly the pages in use, and physical ids
  are a seeded random permutation of the pool, so neighbouring logical pages
  are scattered.
* Values: q, K and V are ``sigma * N(0, 1)`` drawn with ``torch.randn`` from a
  ``torch.Generator`` seeded with ``seed`` on the target device, rounded once
  to bf16 (round to nearest even). Unused slots of partially filled last pages
  hold random values too, as stale cache entries would.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

LAYOUTS = ("NHD", "HND")


@dataclass(frozen=True)
class DecodeConfig:
    """One decode workload: shapes, length distribution, layout and value scale."""

    name: str
    batch: int
    num_qo_heads: int
    num_kv_heads: int
    page_size: int
    layout: str
    lengths: tuple  # ("const", L) | ("uniform", lo, hi) | ("lognormal", median, sigma, lo, hi)
    sigma: float = 1.0
    head_dim: int = 128
    shared_prefix_tokens: int = 0
    share_group: int = 1
    want_lse: bool = True
    seed: int = 0

    @property
    def group_size(self) -> int:
        return self.num_qo_heads // self.num_kv_heads

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


# The five workloads of the decode benchmark. Seeds are 20261202 + position.
CONFIGS = {
    c.name: c
    for c in [
        DecodeConfig("mha8_b1_l512_ps16_nhd", batch=1, num_qo_heads=8, num_kv_heads=8,
                     page_size=16, layout="NHD", lengths=("const", 512), seed=20261203),
        DecodeConfig("gqa4_b32_u512to4096_ps16_nhd", batch=32, num_qo_heads=32, num_kv_heads=8,
                     page_size=16, layout="NHD", lengths=("uniform", 512, 4096),
                     seed=20261204),
        DecodeConfig("gqa4_b128_lognorm2048_ps16_hnd", batch=128, num_qo_heads=32,
                     num_kv_heads=8, page_size=16, layout="HND",
                     lengths=("lognormal", 2048, 1.0, 128, 8192), seed=20261205),
        DecodeConfig("mqa32_b16_l32768_ps64_nhd", batch=16, num_qo_heads=32, num_kv_heads=1,
                     page_size=64, layout="NHD", lengths=("const", 32768), seed=20261206),
        DecodeConfig("gqa8_b256_u128to16384_prefix1024x8_ps16_nhd", batch=256, num_qo_heads=64,
                     num_kv_heads=8, page_size=16, layout="NHD",
                     lengths=("uniform", 128, 16384), sigma=1.5, shared_prefix_tokens=1024,
                     share_group=8, seed=20261207),
    ]
}
CONFIG_ORDER = list(CONFIGS)


@dataclass
class BlockTables:
    """CSR block tables plus the facts tests need about them."""

    lengths: np.ndarray        # int64 [B]
    indptr: np.ndarray         # int32 [B+1]
    indices: np.ndarray        # int32 [nnz]
    last_page_len: np.ndarray  # int32 [B]
    num_pages: int             # pool capacity (pages in use)
    page_size: int
    shared_pages: int = 0      # physical pages referenced by more than one request
    extra: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.lengths.shape[0])


def draw_lengths(spec: tuple, batch: int, rng: np.random.Generator) -> np.ndarray:
    kind = spec[0]
    if kind == "const":
        return np.full(batch, int(spec[1]), np.int64)
    if kind == "uniform":
        lo, hi = int(spec[1]), int(spec[2])
        return rng.integers(lo, hi + 1, size=batch, dtype=np.int64)
    if kind == "lognormal":
        median, sig, lo, hi = spec[1], spec[2], spec[3], spec[4]
        x = np.exp(rng.normal(math.log(median), sig, size=batch))
        return np.clip(np.rint(x), lo, hi).astype(np.int64)
    if kind == "list":
        return np.asarray(spec[1], np.int64)
    raise ValueError(f"unknown length spec {spec!r}")


def build_block_tables(lengths, page_size: int, rng: np.random.Generator,
                       shared_prefix_tokens: int = 0, share_group: int = 1,
                       permute: bool = True) -> BlockTables:
    """Assign physical pages to each request's logical pages (see module doc)."""
    lengths = np.asarray(lengths, np.int64)
    if (lengths < 1).any():
        raise ValueError("every request needs at least one token")
    B = lengths.shape[0]
    pages = (lengths + page_size - 1) // page_size
    shared_n = shared_prefix_tokens // page_size if share_group > 1 else 0
    logical_to_phys = []
    next_id = 0
    group_prefix = {}
    for b in range(B):
        ids = []
        g = b // share_group if shared_n else None
        if shared_n:
            if g not in group_prefix:
                group_prefix[g] = list(range(next_id, next_id + shared_n))
                next_id += shared_n
            ids.extend(group_prefix[g][: min(int(pages[b]), shared_n)])
        rest = int(pages[b]) - len(ids)
        ids.extend(range(next_id, next_id + rest))
        next_id += rest
        logical_to_phys.append(ids)
    # Pool = pages in use; drop shared ids that no request of the group reaches.
    used = sorted({i for ids in logical_to_phys for i in ids})
    compact = {old: new for new, old in enumerate(used)}
    num_pages = len(used)
    perm = rng.permutation(num_pages) if permute else np.arange(num_pages)
    indices = np.asarray([perm[compact[i]] for ids in logical_to_phys for i in ids], np.int32)
    indptr = np.zeros(B + 1, np.int64)
    indptr[1:] = np.cumsum(pages)
    last = lengths - (pages - 1) * page_size
    counts = np.bincount(indices, minlength=num_pages)
    return BlockTables(lengths=lengths, indptr=indptr.astype(np.int32), indices=indices,
                       last_page_len=last.astype(np.int32), num_pages=num_pages,
                       page_size=page_size, shared_pages=int((counts > 1).sum()))


def make_tables(cfg: DecodeConfig, batch: int | None = None) -> BlockTables:
    """Block tables of a workload (optionally only its first ``batch`` requests)."""
    rng = np.random.default_rng(cfg.seed)
    lengths = draw_lengths(cfg.lengths, cfg.batch, rng)
    if batch is not None:
        lengths = lengths[:batch]
    return build_block_tables(lengths, cfg.page_size, rng, cfg.shared_prefix_tokens,
                              cfg.share_group)


def pool_shape(layout: str, num_pages: int, page_size: int, num_kv_heads: int, head_dim: int):
    if layout == "NHD":
        return (num_pages, page_size, num_kv_heads, head_dim)
    if layout == "HND":
        return (num_pages, num_kv_heads, page_size, head_dim)
    raise ValueError(layout)


def make_values(batch, num_qo_heads, num_kv_heads, head_dim, num_pages, page_size, layout,
                seed, sigma=1.0, device="cpu", chunk_elems=1 << 28):
    """q [B, Hq, D] and K/V pools as bf16 torch tensors on ``device``."""
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))

    def draw(shape):
        out = torch.empty(shape, dtype=torch.bfloat16, device=device)
        flat = out.view(-1)
        for s in range(0, flat.numel(), chunk_elems):
            n = min(chunk_elems, flat.numel() - s)
            x = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
            flat[s:s + n] = (x * sigma).to(torch.bfloat16)
        return out

    q = draw((batch, num_qo_heads, head_dim))
    shape = pool_shape(layout, num_pages, page_size, num_kv_heads, head_dim)
    k = draw(shape)
    v = draw(shape)
    return q, k, v


@dataclass
class Case:
    """A complete decode problem: config-like shape facts, tables and tensors."""

    batch: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    layout: str
    sm_scale: float
    tables: BlockTables
    q: object
    k: object
    v: object
    want_lse: bool = True
    name: str = "case"

    @property
    def group_size(self):
        return self.num_qo_heads // self.num_kv_heads

    def kv_bytes(self) -> int:
        """Logical KV bytes one decode step reads: sum_b L_b * Hkv * D * 2 (K,V) * 2 B."""
        return int(self.tables.lengths.sum()) * self.num_kv_heads * self.head_dim * 4

    def unique_kv_bytes(self) -> int:
        """KV bytes of distinct (page, token) slots read, counting shared pages once."""
        used = {}
        ind = self.tables.indices
        ptr = self.tables.indptr
        for b in range(self.batch):
            p0, p1 = int(ptr[b]), int(ptr[b + 1])
            for j, page in enumerate(ind[p0:p1]):
                n = self.page_size if p0 + j < p1 - 1 else int(self.tables.last_page_len[b])
                used[int(page)] = max(used.get(int(page), 0), n)
        return sum(used.values()) * self.num_kv_heads * self.head_dim * 4


def make_case(cfg: DecodeConfig, device="cpu", batch: int | None = None) -> Case:
    t = make_tables(cfg, batch)
    q, k, v = make_values(t.batch, cfg.num_qo_heads, cfg.num_kv_heads, cfg.head_dim,
                          t.num_pages, cfg.page_size, cfg.layout, cfg.seed, cfg.sigma, device)
    return Case(t.batch, cfg.num_qo_heads, cfg.num_kv_heads, cfg.head_dim, cfg.page_size,
                cfg.layout, cfg.sm_scale, t, q, k, v, cfg.want_lse, cfg.name)


def custom_case(lengths, num_qo_heads, num_kv_heads, page_size, layout="NHD", head_dim=128,
                seed=1, sigma=1.0, device="cpu", sm_scale=None, shared_prefix_tokens=0,
                share_group=1, permute=True, extra_pages=0) -> Case:
    """A hand-shaped case for tests (``extra_pages`` unused pages pad the pool)."""
    rng = np.random.default_rng(seed)
    t = build_block_tables(lengths, page_size, rng, shared_prefix_tokens, share_group, permute)
    t.num_pages += int(extra_pages)
    q, k, v = make_values(t.batch, num_qo_heads, num_kv_heads, head_dim, t.num_pages, page_size,
                          layout, seed, sigma, device)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(head_dim)
    return Case(t.batch, num_qo_heads, num_kv_heads, head_dim, page_size, layout, sm_scale, t,
                q, k, v, True, "custom")


def bf16_bits(t) -> np.ndarray:
    """Host uint16 view of a bf16 torch tensor (copies to host if needed)."""
    import torch

    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


# ------------------------------------------------------------------ causal prefill

@dataclass(frozen=True)
class PrefillConfig:
    """A paged causal prefill workload: request b has q_lens[b] new query
    tokens, the last of its kv_lens[b] cached tokens (the cache already holds
    the new tokens' K and V)."""

    name: str
    q_lens: tuple
    kv_lens: tuple
    num_qo_heads: int
    num_kv_heads: int
    page_size: int = 16
    layout: str = "NHD"
    head_dim: int = 128
    seed: int = 1
    sigma: float = 1.0

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


PREFILL_CONFIGS = {
    # the pages' paged-prefill shape: two requests, 32 and 64 new tokens over
    # 256 and 1024 cached tokens, GQA group of four, D = 128
    "prefill_gqa4_q32+64_kv256+1024_ps16_nhd": PrefillConfig(
        "prefill_gqa4_q32+64_kv256+1024_ps16_nhd", (32, 64), (256, 1024), 32, 8, seed=20261301),
    # a long chunked prefill: eight requests, 2048 new tokens each over 2048
    # to 16384 cached tokens
    "prefill_gqa4_b8_q2048_kv2048to16384_ps16_nhd": PrefillConfig(
        "prefill_gqa4_b8_q2048_kv2048to16384_ps16_nhd", (2048,) * 8,
        (2048, 4096, 6144, 8192, 10240, 12288, 14336, 16384), 32, 8, seed=20261302),
}
PREFILL_ORDER = list(PREFILL_CONFIGS)


@dataclass
class PrefillCase:
    """A complete causal prefill problem. q is [Nq, Hq, D]; qo_indptr [B+1]."""

    batch: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    layout: str
    sm_scale: float
    tables: BlockTables
    qo_indptr: np.ndarray
    q: object
    k: object
    v: object
    name: str = "prefill"

    @property
    def group_size(self):
        return self.num_qo_heads // self.num_kv_heads

    @property
    def num_q_tokens(self) -> int:
        return int(self.qo_indptr[-1])

    def causal_pairs(self) -> int:
        """(query token, cached token) pairs attended, per query head."""
        n = 0
        for b in range(self.batch):
            ql = int(self.qo_indptr[b + 1] - self.qo_indptr[b])
            L = int(self.tables.lengths[b])
            n += ql * (L - ql) + ql * (ql + 1) // 2
        return n

    def flops(self) -> int:
        """Multiply-adds of QK^T and PV counted as 2 flops each: 4 D per pair per head."""
        return 4 * self.head_dim * self.num_qo_heads * self.causal_pairs()


def prefill_case(q_lens, kv_lens, num_qo_heads, num_kv_heads, page_size, layout="NHD",
                 head_dim=128, seed=1, sigma=1.0, device="cpu", sm_scale=None,
                 permute=True, name="prefill") -> PrefillCase:
    """Block tables over kv_lens (recipe above), q [sum q_lens, Hq, D], pools."""
    if len(q_lens) != len(kv_lens) or any(q > L for q, L in zip(q_lens, kv_lens)):
        raise ValueError("each request needs q_len <= kv_len")
    rng = np.random.default_rng(seed)
    t = build_block_tables(list(kv_lens), page_size, rng, 0, 1, permute)
    qo = np.zeros(len(q_lens) + 1, np.int32)
    qo[1:] = np.cumsum(np.asarray(q_lens, np.int64))
    q, k, v = make_values(int(qo[-1]), num_qo_heads, num_kv_heads, head_dim, t.num_pages,
                          page_size, layout, seed, sigma, device)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(head_dim)
    return PrefillCase(len(q_lens), num_qo_heads, num_kv_heads, head_dim, page_size, layout,
                       sm_scale, t, qo, q, k, v, name)


def make_prefill_case(cfg: PrefillConfig, device="cpu") -> PrefillCase:
    return prefill_case(cfg.q_lens, cfg.kv_lens, cfg.num_qo_heads, cfg.num_kv_heads,
                        cfg.page_size, cfg.layout, cfg.head_dim, cfg.seed, cfg.sigma, device,
                        cfg.sm_scale, name=cfg.name)
