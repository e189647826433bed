"""Seeded synthetic inputs for shared-prefix paged decode attention.

This module only draws inputs: group structure, lengths, physical block ids,
and the Q / K / V values.  It holds none of the attention arithmetic, so the
oracle and the CUDA path can both consume its output without sharing any of
the method's code.

Layout produced (the paged KV cache of the vLLM/PagedAttention pages, with
the head axis placed outside the 16-token axis so one (block, K|V, head) tile
is contiguous):

  pool         [num_pool_blocks][2][Hkv][B][d]   (index 0 = K, 1 = V)
  q            [R][Hq][d]
  block_table  int32 [R][max_blocks_per_req]     (-1 padded)
  group_of_req int32 [R]     leaf prefix group, -1 = no shared prefix
  group_parent int32 [num_groups] or None (single-level)
  prefix_len   int32 [num_groups]   tokens that level adds
  suffix_len   int32 [R]

Segment addressing: a request's block-table row lists its prefix chain root
level first, each level starting at a fresh block and occupying ceil(P/B)
blocks, then its ceil(S/B) suffix blocks.  Slots past the end of a segment
inside its last block are unused (NaN when ``poison`` is set), and so are the
pool blocks no segment owns.

bf16 values are stored as uint16 bit patterns (round-to-nearest-even from an
fp32 N(0,1) draw); fp32 values as float32.
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor
from typing import List, Optional

import numpy as np

F32, BF16 = 0, 1
_BF16_NAN = np.uint16(0x7FC0)
_FILL_CHUNK = 1 << 22  # elements per independently seeded value stream


@dataclasses.dataclass
class Problem:
    name: str
    dtype: int                    # F32 or BF16
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    scale: float
    q: np.ndarray                 # [R][Hq][d] float32 or uint16 (bf16 bits)
    pool: np.ndarray              # [nb][2][Hkv][B][d] float32 or uint16
    block_table: np.ndarray       # int32 [R][maxb]
    group_of_req: np.ndarray      # int32 [R]
    group_parent: Optional[np.ndarray]  # int32 [num_groups] or None
    prefix_len: np.ndarray        # int32 [num_groups]
    suffix_len: np.ndarray        # int32 [R]
    seed: int = 0

    @property
    def num_req(self) -> int:
        return int(self.suffix_len.shape[0])

    @property
    def num_groups(self) -> int:
        return int(self.prefix_len.shape[0])

    @property
    def num_pool_blocks(self) -> int:
        return int(self.pool.shape[0])

    @property
    def max_blocks_per_req(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == F32 else 2

    def chain(self, r: int) -> List[int]:
        """Prefix groups of request r, root level first."""
        g = int(self.group_of_req[r])
        out = []
        while g >= 0:
            out.append(g)
            g = int(self.group_parent[g]) if self.group_parent is not None else -1
        return out[::-1]


@dataclasses.dataclass
class Structure:
    """Group tree and lengths before any block or value is drawn."""
    group_parent: Optional[List[int]]
    prefix_len: List[int]
    group_of_req: List[int]   # logical request order
    suffix_len: List[int]


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16, returned as uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _fill_normal(out_flat: np.ndarray, dtype: int, seed: int, stream_tag: int) -> None:
    """Fill a flat array with N(0,1) values, in fixed-size chunks, each from its
    own PCG64 stream spawned from (seed, stream_tag): the result does not depend
    on the number of threads used."""
    n = out_flat.shape[0]
    nchunks = _ceil_div(n, _FILL_CHUNK)
    if nchunks == 0:
        return
    children = np.random.SeedSequence([seed, stream_tag]).spawn(nchunks)

    def work(i: int) -> None:
        lo, hi = i * _FILL_CHUNK, min(n, (i + 1) * _FILL_CHUNK)
        g = np.random.Generator(np.random.PCG64(children[i]))
        v = g.standard_normal(hi - lo, dtype=np.float32)
        if dtype == F32:
            out_flat[lo:hi] = v
        else:
            out_flat[lo:hi] = f32_to_bf16_bits(v)

    if nchunks == 1:
        work(0)
        return
    with ThreadPoolExecutor(max_workers=min(nchunks, os.cpu_count() or 1)) as ex:
        list(ex.map(work, range(nchunks)))


def materialize(name: str, st: Structure, *, dtype: int, Hq: int, Hkv: int, d: int,
                B: int = 16, seed: int = 0, min_pool_blocks: int = 0,
                shuffle_requests: bool = True, poison: bool = True) -> Problem:
    """Turn a drawn structure into a Problem.

    Draw order (all from one PCG64 stream seeded with ``seed`` after the
    structure draws of the caller, except the value fills which use their own
    spawned streams): 1) request order permutation, 2) physical block
    permutation of the pool.  Values: q from stream tag 1, pool from tag 2.
    """
    rng = np.random.Generator(np.random.PCG64([seed, 7]))
    G = len(st.prefix_len)
    R = len(st.suffix_len)
    parent = st.group_parent

    # request order: logical request i is stored at row perm[i]
    perm = rng.permutation(R) if shuffle_requests else np.arange(R)
    group_of_req = np.full(R, -1, np.int32)
    suffix_len = np.zeros(R, np.int32)
    for i in range(R):
        group_of_req[perm[i]] = st.group_of_req[i]
        suffix_len[perm[i]] = st.suffix_len[i]

    prefix_len = np.asarray(st.prefix_len, np.int32)
    gparent = None if parent is None else np.asarray(parent, np.int32)

    def chain(g: int) -> List[int]:
        out = []
        while g >= 0:
            out.append(g)
            g = int(gparent[g]) if gparent is not None else -1
        return out[::-1]

    gblocks = [_ceil_div(int(p), B) for p in prefix_len]
    needed = sum(gblocks) + sum(_ceil_div(int(s), B) for s in suffix_len)
    nb = max(min_pool_blocks, _ceil_div(max(needed, 1), 64) * 64)
    phys = rng.permutation(nb).astype(np.int32)

    # allocate: every group's blocks first (group id order), then suffixes (row order)
    cursor = 0
    group_phys = []
    for g in range(G):
        group_phys.append(phys[cursor:cursor + gblocks[g]])
        cursor += gblocks[g]
    rows = []
    for r in range(R):
        cols: List[int] = []
        for g in chain(int(group_of_req[r])):
            cols.extend(int(x) for x in group_phys[g])
        nsb = _ceil_div(int(suffix_len[r]), B)
        cols.extend(int(x) for x in phys[cursor:cursor + nsb])
        cursor += nsb
        rows.append(cols)
    maxb = max(1, max((len(c) for c in rows), default=0))
    bt = np.full((R, maxb), -1, np.int32)
    for r, cols in enumerate(rows):
        bt[r, :len(cols)] = cols

    store = np.float32 if dtype == F32 else np.uint16
    q = np.empty((R, Hq, d), store)
    _fill_normal(q.reshape(-1), dtype, seed, 1)
    pool = np.empty((nb, 2, Hkv, B, d), store)
    _fill_normal(pool.reshape(-1), dtype, seed, 2)

    if poison:
        nan = np.float32(np.nan) if dtype == F32 else _BF16_NAN
        used = np.zeros(nb, bool)
        used[phys[:needed]] = True
        pool[~used] = nan
        for g in range(G):
            tail = int(prefix_len[g]) % B
            if gblocks[g] and tail:
                pool[group_phys[g][-1], :, :, tail:, :] = nan
        for r in range(R):
            s = int(suffix_len[r])
            tail = s % B
            if s and tail:
                pool[bt[r, len(rows[r]) - 1], :, :, tail:, :] = nan

    return Problem(name=name, dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                   block_size=B, scale=1.0 / math.sqrt(d), q=q, pool=pool, block_table=bt,
                   group_of_req=group_of_req, group_parent=gparent, prefix_len=prefix_len,
                   suffix_len=suffix_len, seed=seed)


# ---------------------------------------------------------------------------
# The five workloads.  Integers "uniform in [a, b]" include both ends.
# ---------------------------------------------------------------------------

def _uniform_int(rng, lo, hi, n):
    return rng.integers(lo, hi + 1, size=n).tolist()


def _lognormal_len(rng, median, sigma, lo, hi, n):
    z = rng.standard_normal(n)
    v = np.rint(np.exp(math.log(median) + sigma * z))  # rint = round half to even
    return np.clip(v, lo, hi).astype(np.int64).tolist()


def struct_grouped(rng, n_groups: int, members: int, prefix, suffix) -> Structure:
    """n_groups single-level groups of `members` requests each.  `prefix` and
    `suffix` are an int or an inclusive (lo, hi) uniform range; prefix is drawn
    per group, suffix per request."""
    if isinstance(prefix, int):
        plen = [prefix] * n_groups
    else:
        plen = _uniform_int(rng, prefix[0], prefix[1], n_groups)
    R = n_groups * members
    if isinstance(suffix, int):
        slen = [suffix] * R
    else:
        slen = _uniform_int(rng, suffix[0], suffix[1], R)
    gor = [i // members for i in range(R)]
    return Structure(group_parent=None, prefix_len=plen, group_of_req=gor, suffix_len=slen)


def struct_skewed(rng, R: int = 1024, n_ranks: int = 128, zipf_s: float = 1.2,
                  frac_none: float = 0.1, p_med: float = 1500, p_sigma: float = 0.8,
                  p_lo: int = 64, p_hi: int = 8192, s_med: float = 200, s_sigma: float = 0.7,
                  s_lo: int = 1, s_hi: int = 2048) -> Structure:
    """Zipf(s) over `n_ranks` groups (finite support, p_k ~ k^-s), a fixed
    round(frac_none*R) requests with no prefix, lognormal lengths.  Groups
    that draw no member are dropped and the rest renumbered in rank order."""
    n_none = int(round(frac_none * R))
    none_rows = set(rng.permutation(R)[:n_none].tolist())
    k = np.arange(1, n_ranks + 1, dtype=np.float64)
    p = k ** (-zipf_s)
    p /= p.sum()
    ranks = rng.choice(n_ranks, size=R - n_none, p=p).tolist()
    plen_all = _lognormal_len(rng, p_med, p_sigma, p_lo, p_hi, n_ranks)
    slen = _lognormal_len(rng, s_med, s_sigma, s_lo, s_hi, R)
    used = sorted(set(ranks))
    remap = {rk: i for i, rk in enumerate(used)}
    gor, it = [], iter(ranks)
    for i in range(R):
        gor.append(-1 if i in none_rows else remap[next(it)])
    return Structure(group_parent=None, prefix_len=[plen_all[rk] for rk in used],
                     group_of_req=gor, suffix_len=slen)


def struct_two_level(rng, l1: int = 4096, l2: int = 1024, n_l2: int = 64, members: int = 64,
                     suffix=(32, 256)) -> Structure:
    """Group 0 is the root level shared by all; groups 1..n_l2 are its children."""
    R = n_l2 * members
    parent = [-1] + [0] * n_l2
    plen = [l1] + [l2] * n_l2
    slen = _uniform_int(rng, suffix[0], suffix[1], R)
    gor = [1 + i // members for i in range(R)]
    return Structure(group_parent=parent, prefix_len=plen, group_of_req=gor, suffix_len=slen)


def flatten_problem(p: Problem) -> Problem:
    """The same requests, pool and block tables with every prefix chain
    collapsed into one level per leaf group (prefix = the chain's total).
    Physical blocks of a shared root level stay shared, so the flattened
    problem reads them once per leaf group instead of once overall.  Valid
    when every non-leaf level is a whole number of blocks, which keeps the
    block-table rows unchanged."""
    assert p.group_parent is not None
    leaves = sorted(set(int(g) for g in p.group_of_req) - {-1})
    idx = {g: i for i, g in enumerate(leaves)}
    plen = []
    for g in leaves:
        t, h = 0, g
        while h >= 0:
            if h != g:
                assert int(p.prefix_len[h]) % p.block_size == 0
            t += int(p.prefix_len[h])
            h = int(p.group_parent[h])
        plen.append(t)
    gor = np.array([idx[int(g)] if g >= 0 else -1 for g in p.group_of_req], np.int32)
    return dataclasses.replace(p, name=p.name + "_flat", group_parent=None,
                               prefix_len=np.asarray(plen, np.int32), group_of_req=gor)


def chunk_queries(p: Problem, q_len, stream_tag: int = 3) -> np.ndarray:
    """q rows of a batch with prefill chunks: [sum q_len][Hq][d] in p's
    storage dtype, N(0,1) (rounded to bf16 for bf16 problems), from p's seed
    and a value stream of their own."""
    n = int(np.sum(q_len))
    store = np.float32 if p.dtype == F32 else np.uint16
    q = np.empty((n, p.num_q_heads, p.head_dim), store)
    _fill_normal(q.reshape(-1), p.dtype, p.seed, stream_tag)
    return q


def make_chunked(seed: int = 6, *, small: bool = False, poison: bool = True):
    """Prefill chunks mixed with decode requests, Llama-3-8B attention shape
    (bf16, 32/8 heads, d 128): the decode requests sit in groups under a shared
    prompt; each prefill request joins one of those groups or none, has drawn
    earlier distinct tokens, and a chunk of q_len new tokens at the end of its
    suffix.  Full size: 8 groups x 32 decode requests (prefix 2048, suffix
    uniform in [64, 512]) and 7 prefill requests (earlier tokens uniform in
    [0, 1024], chunks uniform in [256, 512]).  Returns (Problem, q_len int32
    [R], q [sum q_len][Hq][d])."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if small:
        ng, mem, prefix, dsuf, npre, early, chunk = 2, 8, 200, (1, 90), 3, (0, 70), (17, 100)
    else:
        ng, mem, prefix, dsuf, npre, early, chunk = 8, 32, 2048, (64, 512), 7, (0, 1024), (256, 512)
    gor = [i // mem for i in range(ng * mem)]
    slen = _uniform_int(rng, dsuf[0], dsuf[1], ng * mem)
    ql = [1] * (ng * mem)
    pre_g = rng.integers(-1, ng, size=npre).tolist()
    pre_e = _uniform_int(rng, early[0], early[1], npre)
    pre_c = _uniform_int(rng, chunk[0], chunk[1], npre)
    gor += pre_g
    slen += [e + c for e, c in zip(pre_e, pre_c)]
    ql += pre_c
    perm = rng.permutation(len(gor))
    st = Structure(group_parent=None, prefix_len=[prefix] * ng,
                   group_of_req=[gor[i] for i in perm], suffix_len=[slen[i] for i in perm])
    p = materialize("chunked", st, dtype=BF16, Hq=32, Hkv=8, d=128, seed=seed,
                    shuffle_requests=False, poison=poison)
    q_len = np.asarray([ql[i] for i in perm], np.int32)
    return p, q_len, chunk_queries(p, q_len)


CONFIG_NAMES = ("tiny_fp32", "llama8b", "long_prefix", "skewed", "two_level", "two_level_flat")


def make(name: str, seed: Optional[int] = None, *, small: bool = False, poison: bool = True,
         **override) -> Problem:
    """Build one of the named workloads.

    ``small=True`` keeps the structure (heads, head_dim, length distributions)
    but shrinks group and request counts so the CPU oracle finishes in
    seconds; it still spans several tiles and ragged tails.
    Default seeds: tiny_fp32 0, llama8b 1, long_prefix 2, skewed 3, two_level 4.
    """
    default_seed = {"tiny_fp32": 0, "llama8b": 1, "long_prefix": 2, "skewed": 3,
                    "two_level": 4, "two_level_flat": 4}
    seed = default_seed[name] if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed))
    kw = dict(seed=seed, poison=poison)
    if name == "tiny_fp32":
        st = struct_grouped(rng, override.get("n_groups", 2), override.get("members", 8),
                            override.get("prefix", 256), override.get("suffix", (1, 64)))
        return materialize(name, st, dtype=F32, Hq=4, Hkv=4, d=64, min_pool_blocks=64, **kw)
    if name == "llama8b":
        ng, mem = (3, 32) if small else (64, 32)
        st = struct_grouped(rng, override.get("n_groups", ng), override.get("members", mem),
                            override.get("prefix", 2048 if not small else 272),
                            override.get("suffix", (64, 512) if not small else (1, 100)))
        return materialize(name, st, dtype=BF16, Hq=32, Hkv=8, d=128, **kw)
    if name == "long_prefix":
        ng, mem = (8, 100) if not small else (2, 40)
        pr = (1024, 10240) if not small else (100, 700)
        st = struct_grouped(rng, override.get("n_groups", ng), override.get("members", mem),
                            override.get("prefix", pr), override.get("suffix", (16, 256)))
        return materialize(name, st, dtype=BF16, Hq=32, Hkv=8, d=128, **kw)
    if name == "skewed":
        if small:
            st = struct_skewed(rng, R=96, n_ranks=16, p_hi=1024, s_hi=700)
        else:
            st = struct_skewed(rng)
        return materialize(name, st, dtype=BF16, Hq=32, Hkv=8, d=128, **kw)
    if name in ("two_level", "two_level_flat"):
        if small:
            st = struct_two_level(rng, l1=256, l2=96, n_l2=3, members=12, suffix=(1, 80))
        else:
            st = struct_two_level(rng, n_l2=override.get("n_groups", 64))
        p = materialize("two_level", st, dtype=BF16, Hq=32, Hkv=8, d=128, **kw)
        return flatten_problem(p) if name == "two_level_flat" else p
    raise KeyError(name)
