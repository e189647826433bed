"""Grouping metadata built from token ids (include/psattn_forest.h) drives the
decode path: the planner reads each shared level once, and the fused kernel
matches the oracle on that grouping (multi-level and single-level)."""
import numpy as np
import pytest

import oracle
import workloads as W
from shared_prefix_kv_gb300 import forest as F
import shared_prefix_kv_gb300 as ps


def token_batch(seed, n_sys=3, n_shot=3, R=40, chunk=16):
    """system prompts (several chunks), few-shot blocks per system prompt,
    then each request's own tokens"""
    rng = np.random.default_rng(seed)
    sys_p = [list(rng.integers(0, 32000, int(rng.integers(2, 12)) * chunk)) for _ in range(n_sys)]
    shots = [[list(rng.integers(0, 32000, int(rng.integers(1, 6)) * chunk)) for _ in range(n_shot)]
             for _ in range(n_sys)]
    reqs = []
    for _ in range(R):
        s = int(rng.integers(0, n_sys))
        k = int(rng.integers(0, n_shot + 1))  # n_shot: no few-shot block
        own = list(rng.integers(0, 32000, int(rng.integers(1, 200))))
        reqs.append(sys_p[s] + (shots[s][k] if k < n_shot else []) + own)
    return reqs


def problem(res, seed, dtype=W.BF16):
    st = W.Structure(group_parent=None if res["group_parent"] is None else res["group_parent"].tolist(),
                     prefix_len=res["prefix_len"].tolist(), group_of_req=res["group_of_req"].tolist(),
                     suffix_len=res["suffix_len"].tolist())
    return W.materialize("forest", st, dtype=dtype, Hq=32, Hkv=8, d=128, seed=seed)


@pytest.mark.parametrize("single", [False, True])
def test_planner_reads_each_shared_level_once(single):
    reqs = token_batch(3)
    res = F.forest_group(reqs, chunk=16, single=single)
    p = problem(res, seed=3)
    sh = ps.make_shape(p.num_req, p.num_groups, p.num_q_heads, p.num_kv_heads, p.head_dim,
                       p.block_size, p.max_blocks_per_req, p.num_pool_blocks, p.dtype, p.scale)
    with ps.Plan(sh, p.block_table, p.group_of_req, p.group_parent, p.prefix_len, p.suffix_len,
                 host_only_sms=152) as pl:
        info = pl.info()
    used = set()
    for g in res["group_of_req"]:
        g = int(g)
        while g >= 0:
            used.add(g)
            g = -1 if res["group_parent"] is None else int(res["group_parent"][g])
    shared_tok = sum(int(res["prefix_len"][g]) for g in used)
    token_bytes = 2 * p.num_kv_heads * p.head_dim * 2
    assert info["unique_kv_bytes"] == (shared_tok + int(res["suffix_len"].sum())) * token_bytes
    total = sum(len(r) for r in reqs)
    assert total - (shared_tok + int(res["suffix_len"].sum())) == res["saved_tokens"]


@pytest.mark.gpu
@pytest.mark.parametrize("single", [False, True])
def test_decode_on_forest_groups(single):
    pytest.importorskip("torch")
    from workloads.device import DeviceProblem, tolerances
    reqs = token_batch(11, R=64)
    res = F.forest_group(reqs, chunk=16, single=single)
    p = problem(res, seed=11)
    d = DeviceProblem(p)
    with d.plan() as pl:
        d.decode(pl)
        out, lse = d.result()
        assert pl.status() == (0, 0)
    o_ref, l_ref = oracle.attention(p)
    t_out, t_lse = tolerances(p)
    assert np.abs(out - o_ref).max() <= t_out
    assert np.abs(lse - l_ref).max() <= t_lse


@pytest.mark.gpu
@pytest.mark.parametrize("single", [False, True])
def test_decode_on_cht_batches(single):
    """Feather's chunked-hash-tree batches, each grouped into prefix levels
    (psattn_cht_group) and run through the planner and the fused decode as a
    batch of its own, against the oracle."""
    pytest.importorskip("torch")
    from workloads.device import DeviceProblem, tolerances
    reqs = token_batch(13, R=72)
    res = F.cht_group(reqs, chunk=16, max_batch=24, max_new_chunks=4, single=single)
    assert res["num_batches"] >= 3
    for b in range(res["num_batches"]):
        req, gor, gpar, plen, slen = F.batch_grouping(res, b)
        part = {"group_of_req": gor, "group_parent": None if single else gpar,
                "prefix_len": plen, "suffix_len": slen}
        p = problem(part, seed=100 + b)
        d = DeviceProblem(p)
        with d.plan() as pl:
            d.decode(pl)
            out, lse = d.result()
            assert pl.status() == (0, 0)
        o_ref, l_ref = oracle.attention(p)
        t_out, t_lse = tolerances(p)
        assert np.abs(out - o_ref).max() <= t_out, b
        assert np.abs(lse - l_ref).max() <= t_lse, b
