"""Parity of the fused CUDA decode (through the C ABI) with the CPU oracle.

Element-wise on every output at sizes the oracle finishes in seconds (several
tiles, ragged tails, NaN-poisoned unused slots), and on sampled requests at
the full workload sizes in the benchmark's launch configuration.  Bounds:
max abs error 1e-4 for fp32 inputs; 1e-2 on outputs and 1e-3 on LSE for bf16
inputs (outputs compared after the kernel's bf16 rounding).
"""
import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _lib():
    import shared_prefix_kv_gb300 as ps  # fails loudly when the library is not built
    return ps


def _check(p, out, lse, requests=None):
    from workloads.device import tolerances
    o_ref, l_ref = oracle.attention(p, requests)
    if requests is not None:
        out, lse = out[requests], lse[requests]
    t_out, t_lse = tolerances(p)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    eo = np.abs(out - o_ref).max()
    el = np.abs(lse - l_ref).max()
    assert eo <= t_out, f"{p.name}: max |out - oracle| = {eo:.3g} > {t_out}"
    assert el <= t_lse, f"{p.name}: max |lse - oracle| = {el:.3g} > {t_lse}"
    return eo, el


def _run(p, flags=0, launches=1):
    from workloads.device import DeviceProblem
    d = DeviceProblem(p)
    with d.plan(flags) as pl:
        for _ in range(launches):
            d.decode(pl)
        out, lse = d.result()
        rc, dev_flags = pl.status()
        assert rc == 0 and dev_flags == 0, (rc, dev_flags)
    return out, lse


SMALL = ["tiny_fp32", "llama8b", "long_prefix", "skewed", "two_level", "two_level_flat"]


@pytest.mark.parametrize("name", SMALL)
def test_parity_small(name):
    _lib()
    p = W.make(name, small=name != "tiny_fp32")
    _check(p, *_run(p))


@pytest.mark.parametrize("name", ["llama8b", "skewed", "two_level"])
@pytest.mark.parametrize("flag", ["NO_DEDUP", "SIMT", "NO_TENSOR_PREFIX"])
def test_parity_flags(name, flag):
    ps = _lib()
    p = W.make(name, small=True)
    _check(p, *_run(p, getattr(ps, flag)))


def test_parity_flatten_flag():
    ps = _lib()
    p = W.make("two_level", small=True)
    _check(p, *_run(p, ps.FLATTEN))


@pytest.mark.parametrize("seed", [100, 101, 102])
def test_parity_more_seeds(seed):
    _lib()
    for name in ("llama8b", "skewed"):
        p = W.make(name, seed=seed, small=True)
        _check(p, *_run(p))


def test_repeated_launches_reset_counters():
    _lib()
    p = W.make("skewed", small=True)
    out, lse = _run(p, launches=4)
    _check(p, out, lse)


def _custom(Hq, Hkv, d, dtype, groups, parent, members, suffix, seed=0):
    st = W.Structure(group_parent=parent, prefix_len=groups, group_of_req=members,
                     suffix_len=suffix)
    return W.materialize("custom", st, dtype=dtype, Hq=Hq, Hkv=Hkv, d=d, seed=seed)


def test_edge_prefix_only_single_token_ungrouped():
    _lib()
    # suffix 0 (prefix only), one-token requests, ungrouped requests, a prefix of
    # exactly one block, and one longer than a chunk
    p = _custom(32, 8, 128, W.BF16, groups=[16, 1, 333], parent=None,
                members=[0, 0, 1, 1, 2, 2, 2, -1, -1, 0],
                suffix=[0, 1, 0, 17, 16, 0, 1, 1, 64, 33])
    _check(p, *_run(p))


@pytest.mark.parametrize("Hq,Hkv", [(16, 2), (8, 4), (8, 8)])
def test_edge_gqa_ratios_mma(Hq, Hkv):
    _lib()
    p = _custom(Hq, Hkv, 128, W.BF16, groups=[50, 200], parent=None,
                members=[0, 1, 1, 0, -1, 1, 1, 1, 0], suffix=[3, 40, 0, 77, 5, 16, 9, 1, 130])
    _check(p, *_run(p))


@pytest.mark.parametrize("dtype,d", [(W.BF16, 64), (W.F32, 128), (W.F32, 64)])
def test_edge_simt_shapes(dtype, d):
    _lib()
    p = _custom(8, 2, d, dtype, groups=[70, 33], parent=None,
                members=[0, 0, 1, -1, 1, 0], suffix=[5, 0, 48, 3, 1, 100])
    _check(p, *_run(p))


def test_dense_running_max_regrow():
    """A dense prefix tile whose later K/V tiles score far above the first:
    the tensor-core softmax must move its running max mid-chunk (recompute P
    and rescale O in TMEM), for some rows and not others."""
    _lib()
    p = _custom(32, 8, 128, W.BF16, groups=[1000], parent=None,
                members=[0] * 12 + [-1], suffix=[3, 40, 0, 77, 5, 16, 9, 1, 130, 2, 2, 2, 50])
    rng = np.random.default_rng(5)
    cols = -(-1000 // 16)
    blocks = p.block_table[0, :cols]
    vals = W.bf16_bits_to_f32(p.pool[blocks])            # [cols][2][Hkv][16][d]
    scale = np.ones((cols, 1, 1, 1, 1), np.float32)
    scale[cols // 3:] = 4.0                               # K of the later tokens x4
    scale[2 * cols // 3:] = rng.uniform(0.5, 6.0, size=(cols - 2 * cols // 3, 1, 1, 1, 1))
    vals[:, 0:1] *= scale
    # the scaled scores make attention peaky (|out| ~ |v|): V is scaled down so
    # that the bf16 rounding of the output stays well inside the 1e-2 bound
    vals[:, 1:2] *= 0.25
    p.pool[blocks] = W.f32_to_bf16_bits(vals)
    _check(p, *_run(p))


def test_edge_dense_prefix_only_members():
    """Members of a tensor-core group whose only partial is the prefix (no
    suffix): the dense item's own partial is the whole output."""
    _lib()
    p = _custom(32, 8, 128, W.BF16, groups=[200, 1000], parent=None,
                members=[0] * 10 + [1] * 9 + [-1],
                suffix=[0, 0, 0, 5, 0, 17, 0, 0, 33, 0] + [0, 2, 0, 0, 0, 40, 0, 0, 1] + [7])
    _check(p, *_run(p))


def test_edge_three_level_chain():
    _lib()
    p = _custom(32, 8, 128, W.BF16, groups=[48, 20, 7, 100], parent=[-1, 0, 1, 0],
                members=[2, 2, 1, 3, 3, 0, 2, -1], suffix=[4, 0, 9, 31, 2, 1, 50, 8])
    _check(p, *_run(p))


def long_context_problem():
    """Long contexts: a 131072-token prefix shared by 8 requests and a
    65539-token one (not a whole number of blocks) shared by 6, suffixes from
    0 to 8192 tokens, one ungrouped request with a 100000-token suffix and one
    with 3.  Llama-3-8B attention shape, bf16; about 1.3 GB of pool."""
    return _custom(32, 8, 128, W.BF16, groups=[131072, 65539], parent=None,
                   members=[0] * 8 + [1] * 6 + [-1, -1],
                   suffix=[8192, 1, 0, 300, 5000, 17, 2048, 64,
                           7, 4095, 0, 1000, 33, 6000, 100000, 3], seed=12)


def test_edge_long_context():
    """Split-k at its longest: the prefixes run as many tensor-core chunks
    (or, with tensor tiles off, many per-warp chunks), and the 100000-token
    suffix as many per-warp chunks.  Each (request, KV head) merges tens of
    partials.  Checked on every output, with each plan flag that changes the
    split."""
    ps = _lib()
    p = long_context_problem()
    o_ref, l_ref = oracle.attention(p)
    from workloads.device import tolerances
    t_out, t_lse = tolerances(p)
    for flag in (0, ps.NO_TENSOR_PREFIX, ps.NO_DEDUP):
        out, lse = _run(p, flag)
        assert np.isfinite(out).all() and np.isfinite(lse).all()
        eo, el = np.abs(out - o_ref).max(), np.abs(lse - l_ref).max()
        assert eo <= t_out and el <= t_lse, (flag, eo, el)


@pytest.mark.parametrize("case", ["two_children", "chain"])
@pytest.mark.parametrize("flag", ["default", "NO_FOLD"])
def test_parity_folded_levels(case, flag):
    """Parent levels read by their children's tensor-core items (the default
    plan of these batches) against the oracle, and the same batches with
    every level its own partial."""
    ps = _lib()
    from tests.test_plan import FOLD_CASES, fold_case
    (groups, parent, members), _, _ = FOLD_CASES[case]
    p = fold_case(groups, parent, members)
    _check(p, *_run(p, 0 if flag == "default" else getattr(ps, flag)))


def test_edge_empty_batch():
    ps = _lib()
    from workloads.device import shape_of
    sh = ps.make_shape(0, 0, 32, 8, 128, 16, 1, 64, ps.BF16, 0.088)
    with ps.Plan(sh, np.zeros((0, 1), np.int32), np.zeros(0, np.int32), None, None,
                 np.zeros(0, np.int32)) as pl:
        x = torch.zeros(16, device="cuda", dtype=torch.bfloat16)
        pl.decode(x, x, x, x, x, x, x, None)
        assert pl.status() == (0, 0)


def test_suffix_grows_across_blocks_without_replanning():
    """A decode loop keeps its plan while every request's suffix grows by
    1-40 tokens, crossing block boundaries: the new blocks go into spare
    block-table columns (unused, -1, when the plan was built), and the kernel
    reads lengths and block ids from the device tables of each launch."""
    _lib()
    import dataclasses
    from workloads.device import DeviceProblem
    p = W.make("llama8b", small=True, poison=False)
    spare = 4  # 40 tokens need at most 3 more blocks
    R, maxb = p.block_table.shape
    bt = np.full((R, maxb + spare), -1, np.int32)
    bt[:, :maxb] = p.block_table
    nb0 = p.num_pool_blocks
    growth = np.random.default_rng(8).integers(1, 41, size=R)
    # enough new pool blocks for every request's new suffix blocks
    new_blocks = [-(-(int(s) + int(g)) // 16) - -(-int(s) // 16)
                  for s, g in zip(p.suffix_len, growth)]
    extra = sum(new_blocks)
    pool = np.concatenate([p.pool, np.zeros((extra,) + p.pool.shape[1:], p.pool.dtype)])
    rng = np.random.default_rng(9)
    pool[nb0:] = W.f32_to_bf16_bits(rng.standard_normal(pool[nb0:].shape, dtype=np.float32))
    p = dataclasses.replace(p, block_table=bt, pool=pool)
    d = DeviceProblem(p)
    with d.plan() as pl:
        # step 1: the planned batch
        d.decode(pl)
        out0, lse0 = d.result()
        assert pl.status() == (0, 0)
        _check(p, out0, lse0)
        # step 2: the same plan after the suffixes grew
        grown_bt = bt.copy()
        grown_len = p.suffix_len.copy()
        nxt = nb0
        for r in range(R):
            used = int(np.count_nonzero(bt[r] >= 0))
            for k in range(new_blocks[r]):
                grown_bt[r, used + k] = nxt
                nxt += 1
            s0 = int(p.suffix_len[r])
            grown_len[r] = s0 + int(growth[r])
            # the tokens past the old end inside the old last block get new values
            if s0 % 16:
                blk = bt[r, used - 1]
                pool[blk, :, :, s0 % 16:, :] = W.f32_to_bf16_bits(
                    rng.standard_normal((2, p.num_kv_heads, 16 - s0 % 16, p.head_dim),
                                        dtype=np.float32))
        assert nxt == pool.shape[0]
        p2 = dataclasses.replace(p, block_table=grown_bt, suffix_len=grown_len, pool=pool)
        d2 = DeviceProblem(p2)
        d2.decode(pl)
        out, lse = d2.result()
        assert pl.status() == (0, 0)
    _check(p2, out, lse)


def test_suffix_grows_without_replanning():
    _lib()
    from workloads.device import DeviceProblem
    p = W.make("llama8b", small=True)
    d = DeviceProblem(p)
    with d.plan() as pl:
        # grow every request whose last suffix block has a free slot by one token
        grown = p.suffix_len.copy()
        rng = np.random.default_rng(3)
        for r in range(p.num_req):
            s = int(p.suffix_len[r])
            if s % 16:
                col = int(np.count_nonzero(p.block_table[r] >= 0)) - 1
                blk = p.block_table[r, col]
                p.pool[blk, :, :, s % 16, :] = W.f32_to_bf16_bits(
                    rng.standard_normal((2, p.num_kv_heads, p.head_dim)))
                grown[r] = s + 1
        p.suffix_len = grown
        d2 = DeviceProblem(p)
        d2.decode(pl)
        out, lse = d2.result()
        assert pl.status() == (0, 0)
    _check(p, out, lse)


def test_bounded_wait_gives_up_and_reports():
    """A kernel wait on an mbarrier that nothing completes (1 ms limit) gives
    up through the decode kernel's own bounded wait: error flag 16 comes back,
    no fault, and the context still runs a decode with a clean error word."""
    ps = _lib()
    rc, flags = ps.psattn_selftest_wait_timeout(1000)
    assert rc == ps.ERR_DEVICE and flags == 16, (rc, flags)
    p = W.make("llama8b", small=True)
    _check(p, *_run(p))


def test_device_error_word_on_bad_block_id():
    _lib()
    from workloads.device import DeviceProblem
    p = W.make("llama8b", small=True)
    d = DeviceProblem(p)
    with d.plan() as pl:
        bt = p.block_table.copy()
        bt[5, int(np.count_nonzero(bt[5] >= 0)) - 1] = p.num_pool_blocks + 1000
        d.bt.copy_(torch.from_numpy(bt))
        d.decode(pl)
        d.decode(pl)
        rc, flags = pl.status()
        assert rc == -7 and flags & 1
        # the error word, counters and tickets were reset by the status read
        # the plan still works once the table is fixed
        d.bt.copy_(torch.from_numpy(p.block_table))
        d.decode(pl)
        out, lse = d.result()
        assert pl.status() == (0, 0)
    _check(p, out, lse)


def test_device_error_word_on_group_mismatch():
    _lib()
    from workloads.device import DeviceProblem
    p = W.make("llama8b", small=True)
    d = DeviceProblem(p)
    with d.plan() as pl:
        g = p.group_of_req.copy()
        g[3] = (g[3] + 1) % p.num_groups
        d.gor.copy_(torch.from_numpy(g))
        d.decode(pl)
        rc, flags = pl.status()
        assert rc == -7 and flags & 2


# ------------------------------------------------- full sizes, sampled outputs

FULL = ["tiny_fp32", "llama8b", "long_prefix", "skewed", "two_level", "two_level_flat"]


def _sample(p, n=160):
    rng = np.random.default_rng(11)
    picks = set(rng.choice(p.num_req, size=min(n, p.num_req), replace=False).tolist())
    picks.add(int(np.argmax(p.suffix_len)))
    picks.add(int(np.argmin(p.suffix_len)))
    none = np.nonzero(p.group_of_req < 0)[0]
    if none.size:
        picks.add(int(none[0]))
    return sorted(picks)


@pytest.mark.parametrize("name,flag", [(n, "0") for n in FULL] + [("two_level", "NO_FOLD")])
def test_parity_full_size_sampled(name, flag):
    """Sampled requests of every full-size batch, in the benchmark's launch
    configuration.  The two-level batch also runs as the three-partial merge
    (NO_FOLD: level 1, the request's level-2 group and its suffix are each a
    partial of their own, merged in the same launch)."""
    ps = _lib()
    p = W.make(name)
    out, lse = _run(p, 0 if flag == "0" else getattr(ps, flag))
    _check(p, out, lse, _sample(p))
    assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_no_fold_plan_has_three_partials_per_request():
    """The NO_FOLD plan of the full-size two-level batch is the literal
    three-partial form: every request merges level 1, its level-2 group and
    its suffix chunks, and the dense items read level 1 and level 2
    separately."""
    ps = _lib()
    from workloads.device import shape_of
    p = W.make("two_level", poison=False)
    with ps.Plan(shape_of(p), p.block_table, p.group_of_req, p.group_parent, p.prefix_len,
                 p.suffix_len, flags=ps.NO_FOLD, host_only_sms=152) as pl:
        req = pl.export(ps.EXPORT_REQ).reshape(-1, 8)
        grp = pl.export(ps.EXPORT_GROUP).reshape(-1, 8)
    n_suffix_chunks = req[:, 4]
    assert (req[:, 1] == grp[0, 2] + grp[1, 2] + n_suffix_chunks).all()
    assert grp[0, 2] >= 1 and grp[1, 2] >= 1 and (n_suffix_chunks >= 1).all()
