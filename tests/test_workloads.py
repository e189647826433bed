"""Checks of the seeded generator: structure, determinism, segment layout."""
import numpy as np
import pytest

import workloads as W


def test_deterministic():
    a = W.make("llama8b", small=True)
    b = W.make("llama8b", small=True)
    assert np.array_equal(a.pool, b.pool) and np.array_equal(a.block_table, b.block_table)
    c = W.make("llama8b", seed=9, small=True)
    assert not np.array_equal(a.q, c.q)


def test_tiny_fp32_pool_reading():
    p = W.make("tiny_fp32")
    assert p.dtype == W.F32 and p.num_q_heads == 4 and p.num_kv_heads == 4 and p.head_dim == 64
    assert p.num_req == 16 and p.num_groups == 2
    assert (p.prefix_len == 256).all()
    assert p.suffix_len.min() >= 1 and p.suffix_len.max() <= 64
    needed = 2 * 16 + sum(-(-int(s) // 16) for s in p.suffix_len)
    assert p.num_pool_blocks == max(64, -(-needed // 64) * 64)
    assert p.scale == pytest.approx(1 / 8)


def test_segments_and_blocks_unique():
    p = W.make("two_level", small=True)
    B = p.block_size
    owner = {}
    for r in range(p.num_req):
        col = 0
        for g in p.chain(r):
            n = -(-int(p.prefix_len[g]) // B)
            for c in range(col, col + n):
                assert owner.setdefault(int(p.block_table[r, c]), ("g", g)) == ("g", g)
            col += n
        n = -(-int(p.suffix_len[r]) // B)
        for c in range(col, col + n):
            assert owner.setdefault(int(p.block_table[r, c]), ("r", r)) == ("r", r)
        assert (p.block_table[r, col + n:] == -1).all()


def test_poison_layout():
    p = W.make("tiny_fp32")
    used = set(int(b) for b in p.block_table.ravel() if b >= 0)
    for b in range(p.num_pool_blocks):
        assert np.isnan(p.pool[b]).all() == (b not in used)


def test_flat_variant_shares_blocks():
    a = W.make("two_level", small=True)
    f = W.make("two_level_flat", small=True)
    assert np.array_equal(a.block_table, f.block_table) and f.group_parent is None
    for r in range(a.num_req):
        total = sum(int(a.prefix_len[g]) for g in a.chain(r))
        assert int(f.prefix_len[f.group_of_req[r]]) == total


def test_skewed_shape():
    p = W.make("skewed", small=True)
    assert (p.group_of_req == -1).sum() == round(0.1 * p.num_req)
    counts = np.bincount(p.group_of_req[p.group_of_req >= 0])
    assert (counts > 0).all()


def test_bf16_rounding_is_rne():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e-3], np.float32)
    bits = W.f32_to_bf16_bits(x)
    import torch
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bits, ref)
