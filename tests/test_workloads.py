"""The seeded input recipe produces the workloads' stated shapes and structure."""
import numpy as np
import pytest
import torch

import workloads as W


def _check_csr(t: W.BlockTables):
    assert t.indptr[0] == 0 and (np.diff(t.indptr) >= 1).all()
    assert t.indptr[-1] == t.indices.shape[0]
    assert ((t.last_page_len >= 1) & (t.last_page_len <= t.page_size)).all()
    pages = np.diff(t.indptr)
    assert np.array_equal((pages - 1) * t.page_size + t.last_page_len, t.lengths)
    assert t.indices.min() >= 0 and t.indices.max() < t.num_pages
    assert np.unique(t.indices).shape[0] == t.num_pages  # the pool is exactly the pages in use


@pytest.mark.parametrize("name", W.CONFIG_ORDER)
def test_tables_follow_the_recipe(name):
    cfg = W.CONFIGS[name]
    t = W.make_tables(cfg)
    _check_csr(t)
    kind = cfg.lengths[0]
    if kind == "const":
        assert (t.lengths == cfg.lengths[1]).all()
    elif kind == "uniform":
        assert t.lengths.min() >= cfg.lengths[1] and t.lengths.max() <= cfg.lengths[2]
    elif kind == "lognormal":
        assert t.lengths.min() >= cfg.lengths[3] and t.lengths.max() <= cfg.lengths[4]
        assert 1200 < np.median(t.lengths) < 3400
    if cfg.shared_prefix_tokens:
        n = cfg.shared_prefix_tokens // cfg.page_size
        for g in range(cfg.batch // cfg.share_group):
            rows = [t.indices[t.indptr[b]:t.indptr[b] + min(n, t.indptr[b + 1] - t.indptr[b])]
                    for b in range(g * cfg.share_group, (g + 1) * cfg.share_group)]
            longest = max(rows, key=len)
            for r in rows:
                assert np.array_equal(r, longest[:len(r)])
        assert t.shared_pages > 0
    else:
        assert t.shared_pages == 0
    # physical order is scattered, not the logical order
    assert not np.array_equal(t.indices, np.arange(t.indices.shape[0]))


def test_same_seed_same_inputs_and_sigma():
    cfg = W.CONFIGS["mha8_b1_l512_ps16_nhd"]
    a = W.make_case(cfg)
    b = W.make_case(cfg)
    assert torch.equal(a.k, b.k) and torch.equal(a.q, b.q)
    assert np.array_equal(a.tables.indices, b.tables.indices)
    assert 0.95 < float(a.k.float().std()) < 1.05
    assert a.k.shape == (32, 16, 8, 128) and a.q.shape == (1, 8, 128)
    assert a.kv_bytes() == 512 * 8 * 128 * 4 == a.unique_kv_bytes()


def test_shared_prefix_bytes_counted_once():
    case = W.custom_case([64, 64, 100], num_qo_heads=2, num_kv_heads=1, page_size=16,
                         shared_prefix_tokens=32, share_group=3, seed=2)
    assert case.kv_bytes() == 228 * 128 * 4
    assert case.unique_kv_bytes() == (228 - 2 * 32) * 128 * 4
