"""Test helper: scatter dense per-segment K/V into a paged pool.

This is the inverse of the oracle's gather, written as a scatter so that a
wrong block, slot, head or level index on the gather side cannot cancel out.
"""
import math

import numpy as np

import workloads as W


def pack(levels, parent, members, suffixes, q, *, Hkv, B, dtype=W.F32, scale=None, seed=0,
         pad_blocks=3):
    """levels[g] = (K [Hkv][P_g][d], V) for prefix group g (P_g may be 0);
    parent[g] = parent group or -1 (None for single level);
    members[r] = leaf group of request r or -1;
    suffixes[r] = (K [Hkv][S_r][d], V);
    q = [R][Hq][d].  Values must be exactly representable in the storage dtype.
    Returns (Problem, dense) where dense[r] = (K [Hkv][n][d], V) concatenated
    root level first, then the suffix."""
    rng = np.random.default_rng(seed)
    R = len(suffixes)
    d = q.shape[2]
    nblk = lambda n: -(-n // B)
    G = len(levels)
    need = sum(nblk(l[0].shape[1]) for l in levels) + sum(nblk(s[0].shape[1]) for s in suffixes)
    nb = need + pad_blocks
    phys = rng.permutation(nb)
    store = np.float32 if dtype == W.F32 else np.uint16
    nan = np.float32(np.nan) if dtype == W.F32 else np.uint16(0x7FC0)
    pool = np.full((nb, 2, Hkv, B, d), nan, store)
    conv = (lambda a: a.astype(np.float32)) if dtype == W.F32 else W.f32_to_bf16_bits
    cur = 0

    def put(K, V):
        nonlocal cur
        n = K.shape[1]
        ids = []
        for j in range(nblk(n)):
            b = int(phys[cur]); cur += 1
            ids.append(b)
            lo, hi = j * B, min(n, (j + 1) * B)
            pool[b, 0, :, :hi - lo, :] = conv(K[:, lo:hi, :])
            pool[b, 1, :, :hi - lo, :] = conv(V[:, lo:hi, :])
        return ids

    gids = [put(*levels[g]) for g in range(G)]

    def chain(g):
        out = []
        while g >= 0:
            out.append(g)
            g = parent[g] if parent is not None else -1
        return out[::-1]

    rows, dense = [], []
    for r in range(R):
        cols, Ks, Vs = [], [], []
        for g in chain(members[r]):
            cols += gids[g]
            Ks.append(levels[g][0]); Vs.append(levels[g][1])
        cols += put(*suffixes[r])
        Ks.append(suffixes[r][0]); Vs.append(suffixes[r][1])
        rows.append(cols)
        dense.append((np.concatenate(Ks, axis=1), np.concatenate(Vs, axis=1)))
    maxb = max(1, max(len(c) for c in rows))
    bt = np.full((R, maxb), -1, np.int32)
    for r, c in enumerate(rows):
        bt[r, :len(c)] = c
    p = W.Problem(name="packed", dtype=dtype, num_q_heads=q.shape[1], num_kv_heads=Hkv,
                  head_dim=d, block_size=B, scale=(1.0 / math.sqrt(d)) if scale is None else scale,
                  q=conv(q), pool=pool, block_table=bt,
                  group_of_req=np.asarray(members, np.int32),
                  group_parent=None if parent is None else np.asarray(parent, np.int32),
                  prefix_len=np.asarray([l[0].shape[1] for l in levels], np.int32),
                  suffix_len=np.asarray([s[0].shape[1] for s in suffixes], np.int32))
    return p, dense


def single_request(K, V, q, B=4, scale=None, seed=0):
    """One request, no shared prefix: K, V [Hkv][n][d], q [Hq][d]."""
    p, _ = pack([], None, [-1], [(K, V)], q[None], Hkv=K.shape[0], B=B, scale=scale, seed=seed)
    return p
