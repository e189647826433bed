"""Bit-exact checks of the host planner (no GPU): every (request, KV head,
token) is covered by exactly one partial, prefixes are read once per group,
partial indices are a permutation, the tables are deterministic, and every
malformed input is rejected with its status before any device work."""
import os
import re
from collections import defaultdict

import numpy as np
import pytest

import workloads as W
import shared_prefix_kv_gb300 as ps

ROOT_HEADER = __import__("os").path.join(__import__("os").path.dirname(__file__), "..",
                                         "include", "psattn.h")


def shape_of(p):
    return ps.make_shape(p.num_req, p.num_groups, p.num_q_heads, p.num_kv_heads, p.head_dim,
                         p.block_size, p.max_blocks_per_req, p.num_pool_blocks, p.dtype, p.scale)


def host_plan(p, flags=0, sms=152, gpar="auto"):
    gp = p.group_parent if gpar == "auto" else gpar
    return ps.Plan(shape_of(p), p.block_table, p.group_of_req, gp, p.prefix_len, p.suffix_len,
                   flags=flags, host_only_sms=sms)


def tables(pl):
    return dict(w=pl.export(ps.EXPORT_WARP_ITEMS).reshape(-1, 8),
                d=pl.export(ps.EXPORT_DENSE_ITEMS).reshape(-1, 8),
                req=pl.export(ps.EXPORT_REQ).reshape(-1, 8),
                grp=pl.export(ps.EXPORT_GROUP).reshape(-1, 8),
                mem=pl.export(ps.EXPORT_MEMBERS),
                add=pl.export(ps.EXPORT_LEN_ADD))


def item_span(t, it, p):
    """Token range of an item, the way the kernel derives it from the tables."""
    kind, kvh, seg, chunk = it[:4]
    if kind == 0:
        r = t["req"][seg]
        ln, ch, n = int(p.suffix_len[seg]), r[3], r[4]
    else:
        g = t["grp"][seg]
        ln, ch, n = int(p.prefix_len[seg]) + int(t["add"][seg]), g[1], g[2]
    lo = chunk * ch
    hi = ln if chunk == n - 1 else min(ln, lo + ch)
    if kind == 3:  # tensor-core item on a ragged level: its span stops at its cost
        hi = min(hi, lo + int(it[7]))
    return lo, max(lo, hi)


def item_members(t, it):
    kind, _, seg, _, mem_off, nmem = it[:6]
    if kind == 0:
        return [int(seg)]
    return [int(x) for x in t["mem"][mem_off:mem_off + nmem]]


def expected_segments(p, flatten=False, add=None):
    """(request -> list of (segment key, length)) from the problem itself.
    add: the plan's len_add table.  A level that leads its children's items
    (folded) shows there as its length added to the next level down, which
    then spans both; the walk below takes from each level's add exactly the
    levels above it, so a wrong add fails the assertion."""
    out = {}
    for r in range(p.num_req):
        ch = p.chain(r)
        segs = []
        if flatten and ch:
            segs.append((("g", ch[-1]), sum(int(p.prefix_len[g]) for g in ch)))
        elif add is None:
            segs += [(("g", g), int(p.prefix_len[g])) for g in ch]
        else:
            i = len(ch) - 1
            while i >= 0:
                g, need, j = ch[i], int(add[ch[i]]), i - 1
                while need > 0:
                    assert j >= 0, "len_add longer than the chain above"
                    need -= int(p.prefix_len[ch[j]])
                    j -= 1
                assert need == 0, "len_add does not end on a level boundary"
                segs.insert(0, (("g", g), int(p.prefix_len[g]) + int(add[g])))
                i = j
        segs.append((("s", r), int(p.suffix_len[r])))
        out[r] = [(k, n) for k, n in segs if n > 0]
    return out


CASES = ["tiny_fp32", "llama8b", "long_prefix", "skewed", "two_level", "two_level_flat"]


@pytest.mark.parametrize("flags", [0, ps.NO_DEDUP, ps.SIMT])
@pytest.mark.parametrize("name", CASES)
def test_coverage_exact(name, flags):
    p = W.make(name, small=True)
    with host_plan(p, flags) as pl:
        t = tables(pl)
        Hkv = p.num_kv_heads
        cover = defaultdict(list)   # (r, h, segkey) -> [(lo, hi)]
        slots = defaultdict(list)   # (r, h) -> [slot_j]
        for it in np.concatenate([t["w"], t["d"]]):
            lo, hi = item_span(t, it, p)
            key = ("s", int(it[2])) if it[0] == 0 else ("g", int(it[2]))
            for r in item_members(t, it):
                cover[(r, int(it[1]), key)].append((lo, hi))
                slots[(r, int(it[1]))].append(int(it[6]))
        segs = expected_segments(p, add=t["add"])
        for r in range(p.num_req):
            nparts = int(t["req"][r][1])
            for h in range(Hkv):
                assert sorted(slots[(r, h)]) == list(range(nparts))
                for key, n in segs[r]:
                    spans = sorted(cover.pop((r, h, key)))
                    pos = 0
                    for lo, hi in spans:
                        assert lo == pos
                        pos = hi
                    assert pos == n
        assert not cover, f"items on segments a request does not own: {list(cover)[:3]}"


@pytest.mark.parametrize("name", ["llama8b", "two_level", "skewed"])
def test_prefix_read_once_per_group(name):
    """Each prefix token of a group is read once per (group, KV head) by every
    item that serves a set of its members: 128/G members per tensor-core tile,
    8/G per warp item, 1 with de-duplication off."""
    p = W.make(name, small=True)
    G = p.num_q_heads // p.num_kv_heads
    for flags in (0, ps.NO_TENSOR_PREFIX, ps.NO_DEDUP):
        with host_plan(p, flags) as pl:
            t = tables(pl)
            reads = defaultdict(int)
            for it in np.concatenate([t["w"], t["d"]]):
                if it[0] in (1, 2):
                    lo, hi = item_span(t, it, p)
                    reads[(int(it[2]), int(it[1]))] += hi - lo
            for g in range(p.num_groups):
                nmem, dense = int(t["grp"][g][5]), int(t["grp"][g][7])
                if nmem == 0:
                    continue
                per_item = 1 if flags == ps.NO_DEDUP else (128 // G if dense else 8 // G)
                if flags:
                    assert not dense
                else:
                    assert dense == (nmem * G >= 8)
                want = int(p.prefix_len[g]) * -(-nmem // per_item)
                for h in range(p.num_kv_heads):
                    assert reads[(g, h)] == want


def test_group_tables_match_block_table():
    p = W.make("two_level", small=True)
    with host_plan(p) as pl:
        t = tables(pl)
        B = p.block_size
        for r in range(p.num_req):
            col = 0
            for g in p.chain(r):
                gi = t["grp"][g]
                assert gi[0] == col
                members = t["mem"][gi[4]:gi[4] + gi[5]]
                assert r in members and gi[3] in members
                n = -(-int(p.prefix_len[g]) // B)
                assert np.array_equal(p.block_table[gi[3], col:col + n], p.block_table[r, col:col + n])
                col += n
            assert t["req"][r][2] == col
            assert t["req"][r][5] == p.group_of_req[r]


def test_deterministic_and_sorted():
    p = W.make("skewed", small=True)
    with host_plan(p) as a, host_plan(p) as b:
        ta, tb = tables(a), tables(b)
        for k in ta:
            assert np.array_equal(ta[k], tb[k])
        cost = ta["w"][:, 7]
        assert (np.diff(cost) <= 0).all()


def fold_case(groups, parent, members, Hq=32, Hkv=8, dtype=W.BF16, d=128, seed=0):
    rng = np.random.default_rng(seed)
    st = W.Structure(group_parent=parent, prefix_len=groups, group_of_req=members,
                     suffix_len=[int(x) for x in rng.integers(0, 60, len(members))])
    return W.materialize("fold", st, dtype=dtype, Hq=Hq, Hkv=Hkv, d=d, seed=seed)


FOLD_CASES = {
    # case: ((prefix_len, group_parent, group_of_req), len_add wanted, folded levels)
    # parent 256 tokens, two children of 32 members: 2 tiles either way -> folds
    "two_children": (([256, 100, 37], [-1, 0, 0], [1] * 32 + [2] * 32), {1: 256, 2: 256}, {0}),
    # root -> mid -> two leaves of 20 members: both upper levels fold
    "chain": (([128, 64, 50, 0], [-1, 0, 1, 1], [2] * 20 + [3] * 20), {2: 192, 3: 192},
              {0, 1}),
    # one request of the parent's own (4 rows, no tile of its own): no fold
    "direct_member": (([256, 100, 37], [-1, 0, 0], [1] * 32 + [2] * 32 + [0]), {}, set()),
    # eight requests of the parent's own fill a third tile: 1 + 1 + 1 <= 3 -> folds,
    # the parent keeps items for those eight
    "direct_tile": (([256, 100, 37], [-1, 0, 0], [1] * 32 + [2] * 32 + [0] * 8),
                    {1: 256, 2: 256}, {0}),
    # children of 30 and 34 members and 40 requests of the parent's own need
    # 1 + 2 + 2 tiles where the parent alone needs 4: no fold
    "direct_extra_tile": (([256, 100, 37], [-1, 0, 0], [1] * 30 + [2] * 34 + [0] * 40), {},
                          set()),
    # a child of one member (4 rows, no tensor-core tile): no fold
    "small_child": (([256, 100, 37], [-1, 0, 0], [1] * 32 + [2]), {}, set()),
    # a parent that ends inside a block: no fold
    "ragged_parent": (([250, 100, 37], [-1, 0, 0], [1] * 32 + [2] * 32), {}, set()),
    # three children of 12 members need 3 tiles where the parent needs 2: no fold
    "more_tiles": (([256, 64, 64, 64], [-1, 0, 0, 0], [1] * 12 + [2] * 12 + [3] * 12), {},
                   set()),
}


@pytest.mark.parametrize("case", sorted(FOLD_CASES))
def test_fold_rules(case):
    (groups, parent, members), want, folded = FOLD_CASES[case]
    p = fold_case(groups, parent, members)
    with host_plan(p) as pl, host_plan(p, ps.NO_FOLD) as nf:
        t, tn = tables(pl), tables(nf)
        assert {g: int(a) for g, a in enumerate(t["add"]) if a} == want
        assert not tn["add"].any()
        # a folded level keeps items only for its own requests; its children's
        # items span it
        for it in np.concatenate([t["w"], t["d"]]):
            if it[0] != 0 and int(it[2]) in folded:
                assert all(p.group_of_req[r] == it[2] for r in item_members(t, it))
        assert folded <= {int(it[2]) for it in tn["d"]}
        # the roofline counts a folded level once; the tiles read it per child
        assert pl.info()["unique_kv_bytes"] == nf.info()["unique_kv_bytes"]


@pytest.mark.parametrize("flag", ["NO_DEDUP", "NO_TENSOR_PREFIX", "SIMT", "FLATTEN"])
def test_fold_only_on_tensor_path(flag):
    (groups, parent, members), _, _ = FOLD_CASES["two_children"]
    p = fold_case(groups, parent, members)
    with host_plan(p, getattr(ps, flag)) as pl:
        t = tables(pl)
        if flag == "FLATTEN":  # every leaf takes its whole chain instead
            assert sorted(int(a) for a in t["add"] if a) == [256, 256]
        else:
            assert not t["add"].any()
    q = fold_case(groups, parent, members, dtype=W.F32, d=64, Hq=8, Hkv=2)
    with host_plan(q) as pl:
        assert not tables(pl)["add"].any()


def test_fold_matches_flatten_on_two_level():
    """On the two-level workload every first level folds: the default plan
    runs the same items as FLATTEN and counts the first level once."""
    p = W.make("two_level")
    with host_plan(p) as a, host_plan(p, ps.FLATTEN) as f, host_plan(p, ps.NO_FOLD) as n:
        ta, tf = tables(a), tables(f)
        for k in ("w", "d", "req", "add"):
            assert np.array_equal(ta[k], tf[k]), k
        assert a.info()["unique_kv_bytes"] == n.info()["unique_kv_bytes"]
        assert a.info()["unique_kv_bytes"] < f.info()["unique_kv_bytes"]


def test_flatten_flag_equals_flattened_input():
    a = W.make("two_level", small=True)
    f = W.make("two_level_flat", small=True)
    with host_plan(a, ps.FLATTEN) as pa, host_plan(f) as pf:
        ia, ib = pa.info(), pf.info()
        for k in ("warp_items", "partial_slots", "unique_kv_bytes", "planned_kv_bytes"):
            assert ia[k] == ib[k], k
        ta = tables(pa)
        tf = tables(pf)
        # the same (kind, kv head, chunk, member set, token span) multiset
        def keyset(t, p):
            return sorted((int(i[0]), int(i[1]), int(i[3]), tuple(sorted(item_members(t, i))),
                           item_span(t, i, p)) for i in t["w"])
        assert keyset(ta, a) == keyset(tf, f)


def test_byte_accounting():
    p = W.make("llama8b", small=True)
    tb = 2 * p.num_kv_heads * p.head_dim * 2
    uniq = (int(p.prefix_len.sum()) + int(p.suffix_len.sum())) * tb
    with host_plan(p) as pl, host_plan(p, ps.NO_DEDUP) as nd:
        assert pl.info()["unique_kv_bytes"] == uniq
        chain_tok = sum(int(p.prefix_len[p.group_of_req[r]]) for r in range(p.num_req))
        assert nd.info()["planned_kv_bytes"] == (chain_tok + int(p.suffix_len.sum())) * tb


def test_plan_independent_of_call_order():
    p = W.make("long_prefix", small=True)
    with host_plan(p, sms=148) as a:
        ta = tables(a)
    with host_plan(p, sms=152) as b, host_plan(p, sms=148) as c:
        tc = tables(c)
    for k in ta:
        assert np.array_equal(ta[k], tc[k])


# ----------------------------------------------------------------- errors

def _err(p, flags=0, **kw):
    shape = kw.pop("shape", shape_of(p))
    args = dict(block_table=p.block_table, group_of_req=p.group_of_req,
                group_parent=p.group_parent, prefix_len=p.prefix_len, suffix_len=p.suffix_len)
    args.update(kw)
    with pytest.raises(ps.PsattnError) as e:
        ps.psattn_plan_host(shape, args["block_table"], args["group_of_req"],
                            args["group_parent"], args["prefix_len"], args["suffix_len"],
                            flags, 152)
    return e.value.status


def test_error_block_oob():
    p = W.make("tiny_fp32")
    bt = p.block_table.copy()
    last = int((bt[5] >= 0).sum()) - 1
    bt[5, last] = p.num_pool_blocks + 7
    assert _err(p, block_table=bt) == ps.ERR_BLOCK_OOB
    bt[5, last] = -3
    assert _err(p, block_table=bt) == ps.ERR_BLOCK_OOB


def test_error_group_mismatch_and_no_dedup_accepts():
    p = W.make("tiny_fp32")
    bt = p.block_table.copy()
    r = int(np.nonzero(p.group_of_req == 1)[0][2])
    bt[r, 3] = bt[r, -1] if bt[r, -1] >= 0 else int(p.block_table.max())
    assert _err(p, block_table=bt) == ps.ERR_GROUP_MISMATCH
    h = ps.psattn_plan_host(shape_of(p), bt, p.group_of_req, None, p.prefix_len, p.suffix_len,
                            ps.NO_DEDUP, 152)
    ps.psattn_plan_destroy(h)


def test_error_lengths_and_empty():
    p = W.make("tiny_fp32")
    s = p.suffix_len.copy(); s[0] = -1
    assert _err(p, suffix_len=s) == ps.ERR_INVALID_ARG
    pl = p.prefix_len.copy(); pl[1] = -5
    assert _err(p, prefix_len=pl) == ps.ERR_INVALID_ARG
    gor = p.group_of_req.copy(); gor[4] = -1
    s = p.suffix_len.copy(); s[4] = 0
    assert _err(p, group_of_req=gor, suffix_len=s) == ps.ERR_EMPTY_REQUEST
    gor = p.group_of_req.copy(); gor[2] = p.num_groups
    assert _err(p, group_of_req=gor) == ps.ERR_INVALID_ARG


def test_error_table_too_narrow():
    p = W.make("tiny_fp32")
    sh = shape_of(p)
    sh.max_blocks_per_req = p.max_blocks_per_req - 1
    bt = np.ascontiguousarray(p.block_table[:, :-1])
    assert _err(p, shape=sh, block_table=bt) == ps.ERR_INVALID_ARG


def test_error_cycle():
    p = W.make("two_level", small=True)
    gp = p.group_parent.copy()
    gp[0] = 2   # root now points into a child: cycle
    assert _err(p, group_parent=gp) == ps.ERR_GROUP_CYCLE
    gp = p.group_parent.copy(); gp[1] = 99
    assert _err(p, group_parent=gp) == ps.ERR_GROUP_CYCLE


def test_error_unsupported():
    p = W.make("llama8b", small=True)
    for field, val in [("block_size", 32), ("head_dim", 96), ("dtype", 7)]:
        sh = shape_of(p)
        setattr(sh, field, val)
        assert _err(p, shape=sh) == ps.ERR_UNSUPPORTED
    sh = shape_of(p); sh.num_q_heads = 12  # G = 1.5
    assert _err(p, shape=sh) == ps.ERR_INVALID_ARG
    sh = shape_of(p); sh.num_kv_heads = 2  # G = 16
    assert _err(p, shape=sh) == ps.ERR_UNSUPPORTED


def test_flatten_needs_whole_blocks():
    p = W.make("two_level", small=True)
    pl = p.prefix_len.copy(); pl[0] = 250   # root level not a whole number of blocks
    assert _err(p, ps.FLATTEN, prefix_len=pl) in (ps.ERR_UNSUPPORTED, ps.ERR_GROUP_MISMATCH)


def test_empty_batch_plans():
    sh = ps.make_shape(0, 0, 32, 8, 128, 16, 1, 64, ps.BF16, 0.088)
    h = ps.psattn_plan_host(sh, np.zeros((0, 1), np.int32), np.zeros(0, np.int32), None,
                            None, np.zeros(0, np.int32), 0, 152)
    info = ps.psattn_plan_info_get(h)
    assert info["warp_items"] == 0 and info["partial_slots"] == 0
    ps.psattn_plan_destroy(h)


def test_status_strings():
    for s in range(0, -10, -1):
        assert ps.psattn_status_string(s) != "unknown status"


def test_abi_exports_every_declared_symbol():
    from shared_prefix_kv_gb300 import chunked, forest, sched
    inc = os.path.dirname(ROOT_HEADER)
    text = "".join(open(os.path.join(inc, h)).read() for h in sorted(os.listdir(inc))
                   if h.endswith(".h"))
    declared = set(re.findall(r"^\s*(?:int|int64_t|void|const char\*)\s+(psattn_\w+)\s*\(",
                              text, flags=re.M))
    assert declared >= set(ps.EXPORTED_SYMBOLS) | set(forest.EXPORTED_SYMBOLS) | set(sched.EXPORTED_SYMBOLS) \
        | set(chunked.EXPORTED_SYMBOLS)
    for name in declared:
        assert hasattr(ps._lib, name), name


def test_binding_constants_match_header():
    """The binding's flags, status codes and dtypes carry the header's values."""
    text = open(ROOT_HEADER).read()
    defines = dict(re.findall(r"^#define PSATTN_(\w+)\s+(\d+)u\b", text, flags=re.M))
    enums = dict(re.findall(r"^\s*PSATTN_(\w+)\s*=\s*(-?\d+)", text, flags=re.M))
    enums.update(re.findall(r"\bPSATTN_(F32|BF16)\s*=\s*(\d+)", text))
    flags = {k: int(v) for k, v in defines.items() if k != "NOALLOC_SCRATCH_BYTES"}
    assert {"NO_DEDUP", "FLATTEN", "NO_TENSOR_PREFIX", "SIMT", "NO_FOLD"} <= set(flags)
    for k, v in flags.items():
        assert getattr(ps, k) == v, k
    assert len(enums) >= 12
    for k, v in enums.items():
        assert getattr(ps, k) == int(v), k


@pytest.mark.parametrize("name,warps", [("llama8b", 4), ("long_prefix", 4), ("skewed", 4),
                                        ("two_level", 4), ("tiny_fp32", 0)])
def test_item_warps_beside_tensor_core_items(name, warps):
    """Four per-warp item warps per CTA run beside the tensor-core items (the
    other eight warps run those items); 0 without tensor-core items."""
    from workloads.device import shape_of
    p = W.make(name, poison=False)
    with ps.Plan(shape_of(p), p.block_table, p.group_of_req, p.group_parent, p.prefix_len,
                 p.suffix_len, host_only_sms=152) as pl:
        assert pl.info()["dense_item_warps"] == warps
