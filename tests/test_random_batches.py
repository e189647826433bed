"""Random batch structures: the planner's coverage on the CPU, the fused
decode's parity with the oracle on the GPU.

Each case draws a random group forest (up to three levels, groups with 0 to
45 members, prefix lengths on and off block boundaries, zero-length levels
and suffixes) and materialises it with the seeded generator.  These cover
shapes the named workloads do not: tiny groups on the tensor-core path,
single-member groups, deep chains with empty levels, ungrouped requests.
"""
import numpy as np
import pytest

import oracle
import workloads as W
import shared_prefix_kv_gb300 as ps

from tests.test_plan import expected_segments, host_plan, item_members, item_span, tables


def random_structure(rng):
    n_roots = int(rng.integers(1, 4))
    parent, plen = [], []

    def add(par, depth):
        g = len(parent)
        parent.append(par)
        # levels with children end on a block boundary half the time
        plen.append(int(rng.choice([0, 16, 48, 100, 256, 333, 700])))
        if depth < 2:
            for _ in range(int(rng.integers(0, 3))):
                add(g, depth + 1)

    for _ in range(n_roots):
        add(-1, 0)
    gor, slen = [], []
    for g in range(len(parent)):
        for _ in range(int(rng.choice([0, 1, 2, 3, 7, 12, 45]))):
            gor.append(g)
            slen.append(int(rng.integers(0, 150)))
    for _ in range(int(rng.integers(0, 6))):  # ungrouped requests
        gor.append(-1)
        slen.append(int(rng.integers(1, 300)))
    # every request must attend to at least one token
    for i, g in enumerate(gor):
        chain_len, gg = 0, g
        while gg >= 0:
            chain_len += plen[gg]
            gg = parent[gg]
        if chain_len + slen[i] == 0:
            slen[i] = 1
    return W.Structure(group_parent=parent, prefix_len=plen, group_of_req=gor, suffix_len=slen)


def make_case(seed, dtype=W.BF16, d=128, Hq=32, Hkv=8):
    rng = np.random.default_rng(seed)
    st = random_structure(rng)
    return W.materialize(f"random{seed}", st, dtype=dtype, Hq=Hq, Hkv=Hkv, d=d, seed=seed)


@pytest.mark.parametrize("seed", range(30))
def test_random_plan_covers_every_token_once(seed):
    p = make_case(seed)
    for flags in (0, ps.NO_TENSOR_PREFIX):
        with host_plan(p, flags) as pl:
            t = tables(pl)
            cover = {}
            for it in np.concatenate([t["w"], t["d"]]):
                lo, hi = item_span(t, it, p)
                key = ("s", int(it[2])) if it[0] == 0 else ("g", int(it[2]))
                for r in item_members(t, it):
                    cover.setdefault((r, int(it[1]), key), []).append((lo, hi))
            for r, segs in expected_segments(p, add=t["add"]).items():
                for h in range(p.num_kv_heads):
                    for key, n in segs:
                        pos = 0
                        for lo, hi in sorted(cover.pop((r, h, key))):
                            assert lo == pos
                            pos = hi
                        assert pos == n
            assert not cover


@pytest.mark.gpu
@pytest.mark.parametrize("seed", range(150))
def test_random_batches_gpu_parity(seed):
    shapes = [dict(), dict(Hq=16, Hkv=8), dict(dtype=W.F32, d=64, Hq=8, Hkv=2)]
    _gpu_parity(make_case(1000 + seed, **shapes[seed % 3]))


# structures whose default plan folds a parent level into its children's
# tensor-core items
FOLDED_SEEDS = [4, 10, 23, 25]


def test_folded_seeds_fold():
    for seed in FOLDED_SEEDS:
        with host_plan(make_case(seed)) as pl:
            assert tables(pl)["add"].any(), seed


@pytest.mark.gpu
@pytest.mark.parametrize("seed", FOLDED_SEEDS)
def test_random_folded_batches_gpu_parity(seed):
    _gpu_parity(make_case(seed))


def _gpu_parity(p):
    pytest.importorskip("torch")
    from workloads.device import DeviceProblem, tolerances
    d = DeviceProblem(p)
    with d.plan() as pl:
        d.decode(pl)
        out, lse = d.result()
        rc, flags = pl.status()
        assert rc == 0 and flags == 0, (rc, flags)
    o_ref, l_ref = oracle.attention(p)
    t_out, t_lse = tolerances(p)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    assert np.abs(out - o_ref).max() <= t_out
    assert np.abs(lse - l_ref).max() <= t_lse
