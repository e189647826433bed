"""Sharding a batch across GPUs by prefix-group trees.

Prefix groups are independent: a request's output depends only on its own
chain of prefix levels and its suffix.  A batch therefore splits across ranks
with no exchange of data at all.  The unit of placement is a prefix tree (a
root level, every level below it and every request that reads any of them),
which keeps each shared prefix read once.  A tree heavier than a rank's fair
share is split at its child subtrees instead; each part then re-reads the
levels above it on its own rank (one extra read of those levels per part),
which costs far less than exchanging partial results.  Requests with no
shared prefix are trees of their own.

``shard_requests`` assigns parts to ranks greedily, heaviest first, to the
currently lightest rank (longest-processing-time rule), by their K/V token
count (every level a part reads once, plus every suffix): the same quantity
the device reads per KV head.  Pure host code, deterministic.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np


def _roots(group_parent: Optional[np.ndarray], num_groups: int) -> np.ndarray:
    root = np.arange(num_groups)
    if group_parent is None:
        return root
    for g in range(num_groups):
        r, steps = g, 0
        while group_parent[r] >= 0:
            r = int(group_parent[r])
            steps += 1
            if steps > num_groups:
                raise ValueError("group_parent has a cycle")
        root[g] = r
    return root


def tree_costs(group_of_req: Sequence[int], group_parent: Optional[Sequence[int]],
               prefix_len: Sequence[int], suffix_len: Sequence[int]):
    """Returns (unit_of_req, unit_cost): every request's tree id and each
    tree's K/V token count.  Tree ids: roots first (by group id), then one per
    ungrouped request (by request id)."""
    gor = np.asarray(group_of_req, np.int64)
    plen = np.asarray(prefix_len, np.int64)
    slen = np.asarray(suffix_len, np.int64)
    gpar = None if group_parent is None else np.asarray(group_parent, np.int64)
    G = plen.shape[0]
    root = _roots(gpar, G)
    roots = sorted(set(root.tolist()))
    rid = {r: i for i, r in enumerate(roots)}
    used = np.zeros(G, bool)
    unit = np.empty(gor.shape[0], np.int64)
    n_units = len(roots)
    for i, g in enumerate(gor):
        if g < 0:
            unit[i] = n_units
            n_units += 1
        else:
            unit[i] = rid[int(root[g])]
            h = int(g)
            while h >= 0:
                used[h] = True
                h = int(gpar[h]) if gpar is not None else -1
    cost = np.zeros(n_units, np.int64)
    for g in range(G):
        if used[g]:
            cost[rid[int(root[g])]] += plen[g]
    np.add.at(cost, unit, slen)
    return unit, cost


def placement_units(group_of_req, group_parent, prefix_len, suffix_len, world: int):
    """Returns (unit_of_req, unit_cost): trees, with trees heavier than
    total / world split at child subtrees (recursively while that helps).  A
    part's cost counts the levels above it again (they are re-read)."""
    gor = np.asarray(group_of_req, np.int64)
    plen = np.asarray(prefix_len, np.int64)
    slen = np.asarray(suffix_len, np.int64)
    gpar = None if group_parent is None else np.asarray(group_parent, np.int64)
    G = plen.shape[0]
    children = [[] for _ in range(G)]
    if gpar is not None:
        for g in range(G):
            if gpar[g] >= 0:
                children[int(gpar[g])].append(g)
    direct = [[] for _ in range(G)]
    for i, g in enumerate(gor):
        if g >= 0:
            direct[int(g)].append(i)
    sub_reqs = [None] * G

    def reqs_of(g):
        if sub_reqs[g] is None:
            out = list(direct[g])
            for c in children[g]:
                out += reqs_of(c)
            sub_reqs[g] = out
        return sub_reqs[g]

    def used_levels(g):  # levels in subtree(g) that some request reads
        lv = 0
        for c in children[g]:
            lv += used_levels(c)
        return lv + (plen[g] if reqs_of(g) else 0)

    # parts: (kind, group, ancestor tokens); kind 0 = whole subtree, 1 = direct members only
    roots = [g for g in range(G) if gpar is None or gpar[g] < 0]
    parts = [(0, g, 0) for g in roots if reqs_of(g)]

    def cost(part):
        kind, g, anc = part
        if kind == 0:
            return anc + used_levels(g) + int(slen[reqs_of(g)].sum())
        return anc + int(plen[g]) + int(slen[direct[g]].sum())

    singles = [i for i, g in enumerate(gor) if g < 0]
    total = sum(cost(pt) for pt in parts) + int(slen[singles].sum())
    target = total / world
    for _ in range(4 * G + 4):
        splittable = [pt for pt in parts if pt[0] == 0 and children[pt[1]] and cost(pt) > target]
        if not splittable:
            break
        pt = max(splittable, key=lambda x: (cost(x), -x[1]))
        parts.remove(pt)
        _, g, anc = pt
        anc2 = anc + int(plen[g])
        parts += [(0, c, anc2) for c in children[g] if reqs_of(c)]
        if direct[g]:
            parts.append((1, g, anc))
    unit = np.empty(gor.shape[0], np.int64)
    costs = []
    for u, pt in enumerate(parts):
        unit[reqs_of(pt[1]) if pt[0] == 0 else direct[pt[1]]] = u
        costs.append(cost(pt))
    for i in singles:
        unit[i] = len(costs)
        costs.append(int(slen[i]))
    return unit, np.asarray(costs, np.int64)


def shard_requests(group_of_req, group_parent, prefix_len, suffix_len, world: int) -> List[np.ndarray]:
    """Request ids of each rank (sorted), whole placement units per rank,
    balanced by K/V token count."""
    if world < 1:
        raise ValueError("world must be >= 1")
    unit, cost = placement_units(group_of_req, group_parent, prefix_len, suffix_len, world)
    order = sorted(range(cost.shape[0]), key=lambda u: (-int(cost[u]), u))
    load = [0] * world
    rank_of_unit = np.empty(cost.shape[0], np.int64)
    for u in order:
        r = min(range(world), key=lambda k: (load[k], k))
        rank_of_unit[u] = r
        load[r] += int(cost[u])
    rank = rank_of_unit[unit]
    return [np.nonzero(rank == r)[0] for r in range(world)]


def subproblem_arrays(requests: np.ndarray, block_table, group_of_req, group_parent, prefix_len,
                      suffix_len):
    """Tables of the batch restricted to `requests` (ids into the full batch):
    (block_table, group_of_req, group_parent, prefix_len, suffix_len) with the
    groups those requests use renumbered in order.  The KV pool is unchanged."""
    req = np.asarray(requests, np.int64)
    gor = np.asarray(group_of_req, np.int64)[req]
    gpar = None if group_parent is None else np.asarray(group_parent, np.int64)
    keep = set()
    for g in gor:
        h = int(g)
        while h >= 0 and h not in keep:
            keep.add(h)
            h = int(gpar[h]) if gpar is not None else -1
    old = sorted(keep)
    new_id = {g: i for i, g in enumerate(old)}
    sub_gor = np.array([new_id[int(g)] if g >= 0 else -1 for g in gor], np.int32)
    sub_plen = np.asarray(prefix_len, np.int32)[old] if old else np.zeros(0, np.int32)
    sub_par = None
    if gpar is not None:
        sub_par = np.array([new_id[int(gpar[g])] if gpar[g] >= 0 else -1 for g in old], np.int32)
    return (np.ascontiguousarray(np.asarray(block_table)[req]), sub_gor, sub_par, sub_plen,
            np.asarray(suffix_len, np.int32)[req])
