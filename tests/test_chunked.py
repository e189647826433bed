"""Prefill chunks in the decode launch (include/psattn_chunked.h).

CPU: the expansion is exact.  The oracle's decode attention over the expanded
batch equals its chunked (causal) attention over the original batch bit for
bit, because each expanded row lists the same tokens in the same order.  The
expanded tables also satisfy what the planner requires.  GPU: the fused
decode over the expanded batch matches the chunked oracle within the bf16
bounds.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import workloads as W
import shared_prefix_kv_gb300 as ps
from shared_prefix_kv_gb300 import chunked as C


def shape_of(p):
    return ps.make_shape(p.num_req, p.num_groups, p.num_q_heads, p.num_kv_heads, p.head_dim,
                         p.block_size, p.max_blocks_per_req, p.num_pool_blocks, p.dtype, p.scale)


def expanded(p, q_len, q, level_tokens):
    sh, bt, gor, gpar, plen, slen = C.expand(shape_of(p), p.block_table, p.group_of_req,
                                             p.group_parent, p.prefix_len, p.suffix_len, q_len,
                                             level_tokens)
    assert sh.num_req == int(np.sum(q_len)) == q.shape[0]
    return dataclasses.replace(p, name=p.name + "_expanded", q=q, block_table=bt,
                               group_of_req=gor, group_parent=gpar, prefix_len=plen,
                               suffix_len=slen)


def two_level_chunked(seed):
    """The small two-level batch with chunks on a few requests (multi-level
    groups under the new levels, chunk starts on and off block boundaries)."""
    p = W.make("two_level", small=True, seed=seed)
    rng = np.random.default_rng(seed)
    ql = np.ones(p.num_req, np.int32)
    pick = rng.choice(p.num_req, size=4, replace=False)
    for r in pick:
        s = int(p.suffix_len[r])
        if s >= 2:
            ql[r] = int(rng.integers(2, s + 1))
    return p, ql, W.chunk_queries(p, ql)


def tiny_fp32_chunked():
    """The tiny fp32 batch (d 64, GQA 1) with chunks: every third request's
    whole suffix, and half the suffix of the next ones."""
    p = W.make("tiny_fp32")
    ql = np.ones(p.num_req, np.int32)
    for r in range(0, p.num_req, 3):
        if p.suffix_len[r] >= 2:
            ql[r] = int(p.suffix_len[r])
    for r in range(1, p.num_req, 3):
        if p.suffix_len[r] >= 4:
            ql[r] = int(p.suffix_len[r]) // 2
    return p, ql, W.chunk_queries(p, ql)


CASES = ([("chunked", s) for s in range(6, 16)] +
         [("two_level", s) for s in (4, 9, 11, 13, 15, 17)])


def make_case(kind, seed):
    return W.make_chunked(seed=seed, small=True) if kind == "chunked" else two_level_chunked(seed)


@pytest.mark.parametrize("level_tokens", [0, 16, 128])
@pytest.mark.parametrize("kind,seed", CASES)
def test_expansion_is_exact_under_the_oracle(kind, seed, level_tokens):
    p, ql, q = make_case(kind, seed)
    p2 = expanded(p, ql, q, level_tokens)
    o2, l2 = oracle.attention(p2)
    o1, l1 = oracle.attention_chunked(p, ql, q)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("level_tokens", [0, 16])
def test_expansion_is_exact_fp32(level_tokens):
    p, ql, q = tiny_fp32_chunked()
    p2 = expanded(p, ql, q, level_tokens)
    o2, l2 = oracle.attention(p2)
    o1, l1 = oracle.attention_chunked(p, ql, q)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("level_tokens", [0, 16, 128])
def test_expanded_tables(level_tokens):
    p, ql, q = W.make_chunked(seed=6, small=True)
    p2 = expanded(p, ql, q, level_tokens)
    NG = p.num_groups
    # new levels: whole blocks (multiples of level_tokens for the causal ones),
    # parents before children
    assert (p2.prefix_len[NG:] % p.block_size == 0).all() and (p2.prefix_len[NG:] > 0).all()
    assert all(p2.group_parent[g] < g for g in range(NG, p2.num_groups))
    assert np.array_equal(p2.prefix_len[:NG], p.prefix_len)
    # each row keeps its request's block-table row and sees n_tok - n + i + 1 tokens
    row = 0
    for r in range(p.num_req):
        n_tok = len(oracle.gather_kv(p, r, 0)[0])
        for i in range(int(ql[r])):
            assert np.array_equal(p2.block_table[row], p.block_table[r])
            assert len(oracle.gather_kv(p2, row, 0)[0]) == n_tok - int(ql[r]) + i + 1
            if ql[r] == 1:
                assert p2.group_of_req[row] == p.group_of_req[r]
            row += 1
    # the planner accepts the expanded batch; its shared levels de-duplicate
    plan = ps.Plan(shape_of(p2), p2.block_table, p2.group_of_req, p2.group_parent,
                   p2.prefix_len, p2.suffix_len, host_only_sms=152)
    info = plan.info()
    assert info["unique_kv_bytes"] > 0
    plan.close()


def test_decode_only_batch_is_unchanged():
    p = W.make("skewed", small=True)
    ones = np.ones(p.num_req, np.int32)
    p2 = expanded(p, ones, p.q, 128)
    assert p2.num_groups == p.num_groups
    for f in ("block_table", "group_of_req", "suffix_len", "prefix_len"):
        assert np.array_equal(getattr(p2, f), getattr(p, f))


def test_chunk_is_whole_suffix_and_level_boundaries():
    # one ungrouped request whose suffix is exactly its chunk of 64 queries:
    # no earlier level; with 16-token levels, query i has (i + 1) // 16 levels
    # and an own suffix of (i + 1) % 16 tokens
    st = W.Structure(group_parent=None, prefix_len=[], group_of_req=[-1], suffix_len=[64])
    p = W.materialize("one", st, dtype=W.BF16, Hq=8, Hkv=2, d=128, seed=1)
    ql = np.array([64], np.int32)
    p2 = expanded(p, ql, W.chunk_queries(p, ql), 16)
    assert p2.num_groups == 4 and (p2.prefix_len == 16).all()
    assert p2.group_parent.tolist() == [-1, 0, 1, 2]
    for i in range(64):
        m = (i + 1) // 16
        assert p2.suffix_len[i] == (i + 1) % 16
        assert p2.group_of_req[i] == (m - 1 if m else -1)


def test_invalid_arguments():
    p, ql, _ = W.make_chunked(seed=6, small=True)
    r = int(np.argmax(ql))
    bad = ql.copy()
    bad[r] = p.suffix_len[r] + 1
    for args in ((bad, 128), (ql, 24), (ql, -16), (np.zeros_like(ql), 128)):
        with pytest.raises(ps.PsattnError):
            C.expand(shape_of(p), p.block_table, p.group_of_req, p.group_parent, p.prefix_len,
                     p.suffix_len, *args)


# ------------------------------------------------------------------- GPU

def _gpu_check(p, ql, q, level_tokens):
    from workloads.device import DeviceProblem, tolerances
    p2 = expanded(p, ql, q, level_tokens)
    d = DeviceProblem(p2)
    with d.plan() as pl:
        d.decode(pl)
        out, lse = d.result()
        rc, dev_flags = pl.status()
        assert rc == 0 and dev_flags == 0, (rc, dev_flags)
    o_ref, l_ref = oracle.attention_chunked(p, ql, q)
    t_out, t_lse = tolerances(p)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    eo, el = np.abs(out - o_ref).max(), np.abs(lse - l_ref).max()
    assert eo <= t_out and el <= t_lse, (eo, el)
    return eo, el


@pytest.mark.gpu
@pytest.mark.parametrize("level_tokens", [0, 128])
@pytest.mark.parametrize("kind,seed", CASES)
def test_gpu_chunked_parity(kind, seed, level_tokens):
    pytest.importorskip("torch")
    p, ql, q = make_case(kind, seed)
    _gpu_check(p, ql, q, level_tokens)


@pytest.mark.gpu
@pytest.mark.parametrize("level_tokens", [0, 16])
def test_gpu_chunked_fp32_and_simt(level_tokens):
    """The CUDA-core path (fp32, d 64, GQA 1) under the same expansion: fp32
    bounds (1e-4)."""
    pytest.importorskip("torch")
    p, ql, q = tiny_fp32_chunked()
    eo, el = _gpu_check(p, ql, q, level_tokens)
    assert eo <= 1e-4 and el <= 1e-4


@pytest.mark.gpu
def test_gpu_chunked_full_size_sampled():
    """The full mixed batch (7 prefill chunks of 256-512 queries beside 256
    decode requests): every prefill query row and a sample of decode rows."""
    pytest.importorskip("torch")
    from workloads.device import DeviceProblem, tolerances
    p, ql, q = W.make_chunked(seed=6)
    p2 = expanded(p, ql, q, 128)
    d = DeviceProblem(p2)
    with d.plan() as pl:
        d.decode(pl)
        out, lse = d.result()
        rc, dev_flags = pl.status()
        assert rc == 0 and dev_flags == 0, (rc, dev_flags)
    starts = np.r_[0, np.cumsum(ql)[:-1]]
    pre = [r for r in range(p.num_req) if ql[r] > 1]
    dec = [r for r in range(p.num_req) if ql[r] == 1][::16]
    # the oracle over just those requests: a sub-batch with the same tables
    sub = sorted(pre + dec)
    ps_sub = dataclasses.replace(p, block_table=p.block_table[sub],
                                 group_of_req=p.group_of_req[sub], suffix_len=p.suffix_len[sub])
    q_sub = np.concatenate([q[starts[r]:starts[r] + ql[r]] for r in sub])
    o_ref, l_ref = oracle.attention_chunked(ps_sub, ql[sub], q_sub)
    rows = np.concatenate([np.arange(starts[r], starts[r] + ql[r]) for r in sub])
    t_out, t_lse = tolerances(p)
    assert np.isfinite(out[rows]).all()
    assert np.abs(out[rows] - o_ref).max() <= t_out
    assert np.abs(lse[rows] - l_ref).max() <= t_lse


# ------------------------------------------------------------ ragged form

def expanded_ragged(p, q_len, q):
    sh, bt, gor, gpar, plen, slen, leaf = C.expand_ragged(
        shape_of(p), p.block_table, p.group_of_req, p.group_parent, p.prefix_len, p.suffix_len,
        q_len)
    p2 = dataclasses.replace(p, name=p.name + "_ragged", q=q, block_table=bt, group_of_req=gor,
                             group_parent=gpar, prefix_len=plen, suffix_len=slen)
    return p2, leaf


def test_ragged_tables():
    p, ql, q = W.make_chunked(seed=6, small=True)
    p2, leaf = expanded_ragged(p, ql, q)
    row = 0
    for r in range(p.num_req):
        n = int(ql[r])
        n_tok = len(oracle.gather_kv(p, r, 0)[0])
        for i in range(n):
            assert np.array_equal(p2.block_table[row], p.block_table[r])
            if n == 1:
                assert leaf[row] == -1 and p2.suffix_len[row] == p.suffix_len[r]
            else:
                g = int(p2.group_of_req[row])
                assert p2.suffix_len[row] == 0 and 1 <= leaf[row] <= p2.prefix_len[g]
                # the row sees the chain above its ragged level plus leaf_len tokens
                chain = p2.chain(row)
                seen = sum(int(p2.prefix_len[c]) for c in chain[:-1]) + int(leaf[row])
                assert seen == n_tok - n + i + 1
            row += 1
    with ps.Plan(shape_of(p2), p2.block_table, p2.group_of_req, p2.group_parent, p2.prefix_len,
                 p2.suffix_len, host_only_sms=152, leaf_len=leaf) as pl:
        assert pl.info()["dense_items"] > 0


def test_ragged_plan_reads_the_level_once():
    from tests.test_plan import tables, item_span
    p, ql, q = W.make_chunked(seed=7, small=True)
    p2, leaf = expanded_ragged(p, ql, q)
    with ps.Plan(shape_of(p2), p2.block_table, p2.group_of_req, p2.group_parent, p2.prefix_len,
                 p2.suffix_len, host_only_sms=152, leaf_len=leaf) as pl:
        t = tables(pl)
        ragged = set(int(p2.group_of_req[k]) for k in range(p2.num_req) if leaf[k] >= 0)
        G = p.num_q_heads // p.num_kv_heads
        per = 4 * (32 // G)
        for g in ragged:
            # members in row order; a tile of `per` members reads the level up to
            # the farthest token one of them sees (the rest of the triangle is skipped)
            lims = [int(leaf[k]) for k in range(p2.num_req) if p2.group_of_req[k] == g]
            want = sum(min(int(p2.prefix_len[g]), max(lims[i:i + per]))
                       for i in range(0, len(lims), per))
            assert want < int(p2.prefix_len[g]) * -(-len(lims) // per)
            for h in range(p.num_kv_heads):
                tok = sum(item_span(t, it, p2)[1] - item_span(t, it, p2)[0] for it in t["d"]
                          if it[2] == g and it[1] == h)
                assert tok == want
                assert all(it[0] == 3 for it in t["d"] if it[2] == g)


def test_ragged_invalid():
    p, ql, q = W.make_chunked(seed=6, small=True)
    p2, leaf = expanded_ragged(p, ql, q)
    k = int(np.argmax(leaf))
    bad = leaf.copy()
    bad[k] = int(p2.prefix_len[p2.group_of_req[k]]) + 1
    with pytest.raises(ps.PsattnError):
        ps.Plan(shape_of(p2), p2.block_table, p2.group_of_req, p2.group_parent, p2.prefix_len,
                p2.suffix_len, host_only_sms=152, leaf_len=bad)
    with pytest.raises(ps.PsattnError):  # ragged levels need the bf16 d 128 path
        ps.Plan(shape_of(p2), p2.block_table, p2.group_of_req, p2.group_parent, p2.prefix_len,
                p2.suffix_len, flags=ps.SIMT, host_only_sms=152, leaf_len=leaf)


def _gpu_check_ragged(p, ql, q, flags=0):
    from workloads.device import DeviceProblem, tolerances
    p2, leaf = expanded_ragged(p, ql, q)
    d = DeviceProblem(p2)
    with ps.Plan(shape_of(p2), p2.block_table, p2.group_of_req, p2.group_parent, p2.prefix_len,
                 p2.suffix_len, flags=flags, leaf_len=leaf) as pl:
        d.decode(pl)
        out, lse = d.result()
        rc, dev_flags = pl.status()
        assert rc == 0 and dev_flags == 0, (rc, dev_flags)
    o_ref, l_ref = oracle.attention_chunked(p, ql, q)
    t_out, t_lse = tolerances(p)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    eo, el = np.abs(out - o_ref).max(), np.abs(lse - l_ref).max()
    assert eo <= t_out and el <= t_lse, (eo, el)


@pytest.mark.gpu
@pytest.mark.parametrize("flags", ["0", "NO_TENSOR_PREFIX", "NO_DEDUP"])
@pytest.mark.parametrize("kind,seed", CASES)
def test_gpu_ragged_parity(kind, seed, flags):
    """The causal part of each chunk as one ragged level: tensor-core tiles
    with per-row limits (and, with tensor tiles off or de-duplication off,
    the mma.sync items with per-row limits)."""
    pytest.importorskip("torch")
    p, ql, q = make_case(kind, seed)
    _gpu_check_ragged(p, ql, q, 0 if flags == "0" else getattr(ps, flags))


@pytest.mark.gpu
def test_gpu_ragged_full_size_sampled():
    pytest.importorskip("torch")
    from workloads.device import DeviceProblem, tolerances
    p, ql, q = W.make_chunked(seed=6)
    p2, leaf = expanded_ragged(p, ql, q)
    d = DeviceProblem(p2)
    with ps.Plan(shape_of(p2), p2.block_table, p2.group_of_req, p2.group_parent, p2.prefix_len,
                 p2.suffix_len, leaf_len=leaf) as pl:
        d.decode(pl)
        out, lse = d.result()
        rc, dev_flags = pl.status()
        assert rc == 0 and dev_flags == 0, (rc, dev_flags)
    starts = np.r_[0, np.cumsum(ql)[:-1]]
    pre = [r for r in range(p.num_req) if ql[r] > 1]
    dec = [r for r in range(p.num_req) if ql[r] == 1][::16]
    sub = sorted(pre + dec)
    ps_sub = dataclasses.replace(p, block_table=p.block_table[sub],
                                 group_of_req=p.group_of_req[sub], suffix_len=p.suffix_len[sub])
    q_sub = np.concatenate([q[starts[r]:starts[r] + ql[r]] for r in sub])
    o_ref, l_ref = oracle.attention_chunked(ps_sub, ql[sub], q_sub)
    rows = np.concatenate([np.arange(starts[r], starts[r] + ql[r]) for r in sub])
    t_out, t_lse = tolerances(p)
    assert np.isfinite(out[rows]).all()
    assert np.abs(out[rows] - o_ref).max() <= t_out
    assert np.abs(lse[rows] - l_ref).max() <= t_lse


@pytest.mark.gpu
def test_gpu_ragged_long_chunk_split_into_chunks():
    """A 300-query chunk that is its request's whole suffix (1200 rows at GQA
    4) beside a few decode requests: the ragged level is split into chunks, so
    the tiles of the first queries have a chunk they see nothing of (items of
    zero tokens that still deliver their empty partials)."""
    pytest.importorskip("torch")
    st = W.Structure(group_parent=None, prefix_len=[96], group_of_req=[0, 0, -1, 0],
                     suffix_len=[300, 40, 33, 9])
    p = W.materialize("long_chunk", st, dtype=W.BF16, Hq=32, Hkv=8, d=128, seed=3,
                      shuffle_requests=False)
    ql = np.array([300, 1, 1, 1], np.int32)
    q = W.chunk_queries(p, ql)
    p2, leaf = expanded_ragged(p, ql, q)
    with ps.Plan(shape_of(p2), p2.block_table, p2.group_of_req, p2.group_parent, p2.prefix_len,
                 p2.suffix_len, host_only_sms=152, leaf_len=leaf) as pl:
        from tests.test_plan import tables
        t = tables(pl)
        assert (t["d"][:, 0] == 3).any() and (t["d"][:, 7] == 0).any()  # zero-token items
    _gpu_check_ragged(p, ql, q)
