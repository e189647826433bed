"""Seeded fuzz of the host-side C calls (no GPU): the planner and both
chunked-prefill expansions, on random valid batches with zero to two values
corrupted (block ids, group ids, parents, lengths, chunk sizes, pool size,
table width; extreme values included).  Also the grouping calls (prefix
forest, CHT batches) and the token-batching simulation, with extreme chunk
sizes, limits and lengths.

Every call must return a status: a crash of the library would end the test
process.  A batch left intact must expand and plan.  The exceptions are the
restrictions the headers state: FLATTEN needs whole-block non-leaf levels and
takes no ragged leaves, and the ragged form needs the bf16 d = 128 path.
"""
import numpy as np
import pytest

import workloads as W
import shared_prefix_kv_gb300 as ps
from shared_prefix_kv_gb300 import chunked as C
from shared_prefix_kv_gb300 import forest as F
from shared_prefix_kv_gb300 import sched as S

from tests.test_plan import shape_of
from tests.test_random_batches import random_structure

EXTREME = [-1, -2, 0, 1, 15, 16, 17, 2 ** 24, 2 ** 30, 2 ** 31 - 1, -2 ** 31]
SHAPES = [(W.BF16, 128, 32, 8), (W.F32, 64, 4, 4), (W.BF16, 64, 8, 2)]


def _corrupt(rng, sh, bt, gor, gpar, plen, slen, ql):
    n = int(rng.integers(0, 3))
    for _ in range(n):
        what, v = int(rng.integers(0, 8)), int(rng.choice(EXTREME))
        if what == 0 and bt.size:
            bt.flat[rng.integers(0, bt.size)] = v
        elif what == 1 and gor.size:
            gor[rng.integers(0, gor.size)] = v
        elif what == 2 and slen.size:
            slen[rng.integers(0, slen.size)] = v
        elif what == 3 and plen.size:
            plen[rng.integers(0, plen.size)] = v
        elif what == 4 and gpar is not None and gpar.size:
            gpar[rng.integers(0, gpar.size)] = v
        elif what == 5 and ql.size:
            ql[rng.integers(0, ql.size)] = v
        elif what == 6:
            sh.num_pool_blocks = max(0, sh.num_pool_blocks + int(rng.integers(-3, 3)))
        elif what == 7:
            sh.max_blocks_per_req = max(0, sh.max_blocks_per_req - int(rng.integers(0, 3)))
    return n


@pytest.mark.parametrize("block", range(4))
def test_host_calls_return_a_status(block):
    for it in range(block * 60, (block + 1) * 60):
        rng = np.random.default_rng([2024, it])
        st = random_structure(rng)
        dtype, d, Hq, Hkv = SHAPES[it % 3]
        p = W.materialize("fuzz", st, dtype=dtype, Hq=Hq, Hkv=Hkv, d=d, seed=it, poison=False)
        sh = shape_of(p)
        bt, gor, slen = p.block_table.copy(), p.group_of_req.copy(), p.suffix_len.copy()
        plen = p.prefix_len.copy()
        gpar = None if p.group_parent is None else p.group_parent.copy()
        ql = np.ones(p.num_req, np.int32)
        for r in range(p.num_req):
            if slen[r] >= 2 and rng.random() < 0.3:
                ql[r] = int(rng.integers(2, slen[r] + 1))
        ncor = _corrupt(rng, sh, bt, gor, gpar, plen, slen, ql)
        bt = np.ascontiguousarray(bt[:, :sh.max_blocks_per_req]) if sh.max_blocks_per_req else \
            np.zeros((bt.shape[0], 0), np.int32)
        flags = int(rng.choice([0, 0, ps.NO_DEDUP, ps.FLATTEN, ps.NO_TENSOR_PREFIX, ps.SIMT,
                                ps.NO_FOLD]))
        mma_path = dtype == W.BF16 and d == 128 and not flags & ps.SIMT
        clean = ncor == 0

        try:
            h = ps.psattn_plan_host(sh, bt, gor, gpar, plen, slen, flags, 152)
            for which in range(6):
                ps.psattn_plan_export(h, which)
            ps.psattn_plan_destroy(h)
        except ps.PsattnError as e:
            assert not clean or e.status == ps.ERR_UNSUPPORTED, (it, e.status)

        for form in ("levels", "ragged"):
            try:
                if form == "levels":
                    out = C.expand(sh, bt, gor, gpar, plen, slen, ql, 256)
                else:
                    out = C.expand_ragged(sh, bt, gor, gpar, plen, slen, ql)
            except ps.PsattnError as e:
                assert not clean, (it, form, e.status)
                continue
            sh2, bt2, gor2, gpar2, plen2, slen2 = out[:6]
            try:
                if form == "levels":
                    h = ps.psattn_plan_host(sh2, bt2, gor2, gpar2, plen2, slen2, flags, 152)
                else:
                    h = ps.psattn_plan_host_ragged(sh2, bt2, gor2, gpar2, plen2, slen2, out[6],
                                                   flags, 152)
                ps.psattn_plan_destroy(h)
            except ps.PsattnError as e:
                allowed = flags & ps.FLATTEN or (form == "ragged" and not mma_path) or \
                    (e.status == ps.ERR_UNSUPPORTED and not mma_path and flags & ps.SIMT)
                assert not clean or allowed, (it, form, e.status, flags)


def test_grouping_and_scheduling_calls_return_a_status():
    ext = [-1, 0, 1, 2, 16, 17, 2 ** 30, 2 ** 31 - 1, -2 ** 31]
    outcomes = set()
    for it in range(300):
        rng = np.random.default_rng([2025, it])
        roots = [rng.integers(0, 50, size=int(rng.integers(0, 80))).tolist() for _ in range(3)]
        reqs = [roots[rng.integers(0, 3)][:int(rng.integers(0, 80))] +
                rng.integers(0, 50, size=int(rng.integers(0, 40))).tolist()
                for _ in range(int(rng.integers(0, 25)))]
        chunk = int(rng.choice([16, 8, 1, 32] + ext))
        try:
            g = F.forest_group(reqs, chunk=chunk, single=bool(rng.random() < 0.5))
            outcomes.add("forest ok")
            assert len(g["group_of_req"]) == len(reqs)
        except ps.PsattnError as e:
            assert e.status == ps.ERR_INVALID_ARG and chunk < 1, (it, chunk, e.status)
        try:
            F.cht_batches(reqs, chunk=chunk, max_batch=int(rng.choice([1, 4, 64] + ext)),
                          max_new_chunks=int(rng.choice([0, 1, 5] + ext)))
            outcomes.add("cht ok")
        except ps.PsattnError as e:
            assert e.status == ps.ERR_INVALID_ARG, (it, e.status)
        try:
            c = F.cht_group(reqs, chunk=chunk, max_batch=int(rng.choice([1, 4, 64] + ext)),
                            max_new_chunks=int(rng.choice([0, 1, 5] + ext)),
                            single=bool(rng.random() < 0.5))
            outcomes.add("cht group ok")
            assert len(c["group_of_req"]) == len(reqs)
            assert c["batch_group_offset"][-1] == len(c["prefix_len"])
        except ps.PsattnError as e:
            assert e.status == ps.ERR_INVALID_ARG, (it, e.status)
        R, NG = len(reqs), int(rng.integers(0, 6))
        gp = rng.integers(0, 300, size=NG)
        gor = rng.integers(-1, NG, size=R) if NG else -np.ones(R, np.int64)
        dl, ol = rng.integers(0, 200, size=R), rng.integers(1, 50, size=R)
        for arr in (gp, gor, dl, ol):
            if arr.size and rng.random() < 0.3:
                arr[rng.integers(0, arr.size)] = int(rng.choice(ext))
        try:
            S.token_batches(gp, gor, dl, ol, n_chunk=int(rng.choice([64, 512] + ext)),
                            m_threshold=int(rng.choice([-1, 1000, 100000] + ext)),
                            max_requests=int(rng.choice([0, 4, 256] + ext)),
                            reorder=bool(rng.random() < 0.5))
            outcomes.add("sched ok")
        except ps.PsattnError as e:
            assert e.status == ps.ERR_INVALID_ARG, (it, e.status)
    assert outcomes == {"forest ok", "cht ok", "cht group ok", "sched ok"}
