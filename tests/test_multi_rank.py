"""Multi-rank path on CPU: two gloo ranks each take a shard of one batch (whole
prefix trees, balanced by bytes), compute it, and rank 0 reassembles the batch
and compares it with the single-process result.  No data moves between ranks
except the final gather the test does to check the answer."""
import dataclasses
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import workloads as W
from shared_prefix_kv_gb300 import shard


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _sub(p, reqs):
    bt, gor, gpar, plen, slen = shard.subproblem_arrays(reqs, p.block_table, p.group_of_req,
                                                        p.group_parent, p.prefix_len, p.suffix_len)
    return dataclasses.replace(p, q=np.ascontiguousarray(p.q[reqs]), block_table=bt,
                               group_of_req=gor, group_parent=gpar, prefix_len=plen,
                               suffix_len=slen)


def _worker(rank, world, port, name, out_path):
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    p = W.make(name, small=True)
    shards = shard.shard_requests(p.group_of_req, p.group_parent, p.prefix_len, p.suffix_len, world)
    mine = shards[rank]
    o, l = oracle.attention(_sub(p, mine), nthreads=2)
    got = [None] * world
    dist.all_gather_object(got, (mine.tolist(), o, l))
    if rank == 0:
        full_o = np.zeros((p.num_req, p.num_q_heads, p.head_dim))
        full_l = np.zeros((p.num_req, p.num_q_heads))
        seen = np.zeros(p.num_req, int)
        for reqs, oo, ll in got:
            full_o[reqs] = oo
            full_l[reqs] = ll
            seen[reqs] += 1
        np.savez(out_path, o=full_o, l=full_l, seen=seen)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("name", ["two_level", "skewed", "llama8b"])
def test_two_rank_shards_reassemble_exactly(name, tmp_path):
    import oracle
    out = str(tmp_path / "res.npz")
    mp.spawn(_worker, args=(2, _free_port(), name, out), nprocs=2, join=True)
    res = np.load(out)
    assert (res["seen"] == 1).all()
    p = W.make(name, small=True)
    o, l = oracle.attention(p, nthreads=2)
    np.testing.assert_array_equal(res["o"], o)
    np.testing.assert_array_equal(res["l"], l)


@pytest.mark.parametrize("name", ["two_level", "skewed", "long_prefix", "llama8b"])
@pytest.mark.parametrize("world", [2, 3, 8])
def test_shards_keep_trees_whole_and_balance(name, world):
    p = W.make(name, small=True)
    shards = shard.shard_requests(p.group_of_req, p.group_parent, p.prefix_len, p.suffix_len, world)
    allr = np.concatenate(shards)
    assert sorted(allr.tolist()) == list(range(p.num_req))
    unit, cost = shard.placement_units(p.group_of_req, p.group_parent, p.prefix_len,
                                       p.suffix_len, world)
    owner, leaf_owner = {}, {}
    for r, reqs in enumerate(shards):
        for q in reqs:
            assert owner.setdefault(int(unit[q]), r) == r  # a placement unit never splits
            g = int(p.group_of_req[q])
            if g >= 0:
                assert leaf_owner.setdefault(g, r) == r  # nor does a leaf group
    loads = [int(cost[np.unique(unit[s])].sum()) if len(s) else 0 for s in shards]
    # greedy LPT bound: no rank exceeds the average by more than the largest unit
    assert max(loads) <= sum(loads) / world + cost.max()
    assert shard.shard_requests(p.group_of_req, p.group_parent, p.prefix_len, p.suffix_len,
                                world)[0].tolist() == shards[0].tolist()


def test_shard_tables_plan_on_every_rank():
    import shared_prefix_kv_gb300 as ps
    p = W.make("two_level", small=True)
    shards = shard.shard_requests(p.group_of_req, p.group_parent, p.prefix_len, p.suffix_len, 2)
    assert all(len(r) for r in shards)  # the single shared root is split at its children
    for reqs in shards:
        s = _sub(p, reqs)
        sh = ps.make_shape(s.num_req, s.num_groups, s.num_q_heads, s.num_kv_heads, s.head_dim,
                           s.block_size, s.max_blocks_per_req, s.num_pool_blocks, s.dtype, s.scale)
        with ps.Plan(sh, s.block_table, s.group_of_req, s.group_parent, s.prefix_len, s.suffix_len,
                     host_only_sms=152) as pl:
            assert pl.info()["unique_kv_bytes"] > 0
