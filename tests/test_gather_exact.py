"""Byte-exact check of the paged gather, through the fused decode kernel.

Every used K slot of the pool is overwritten with a random +-1 code, and each
query (request or prefill row, q head) is B times the K code of one token its
row sees (B = 64, a power of two, so q is exact in bf16).  Its scaled score,
scale * B * d, then beats every other token's by more than 110 natural-log
units.  Every other softmax weight is below 2^-158 and flushes to 0 in fp32.
The attention output is therefore the chosen token's V row itself, and
LSE = scale * B * d.  This holds for any split of the token list into
partials: a partial that does not hold the token has max m_i far below the
merged max, so its merge weight e^(m_i - m*) is 0 too.

So the kernel's bf16 output must equal that V row bit for bit, whatever path
the plan takes: tensor-core tiles, mma.sync or CUDA-core per-warp items,
split-k chunks, folded levels, ragged per-row limits, or de-duplication off.
Unlike the parity tests, this checks every output of the full-size batches,
with no sampling and no tolerance.  The parity tests cannot see a single
dropped or duplicated token in a long context: it moves the output by about
1/n.  The fp32 path divides the same fp32 weight out of O and l, so its
output may differ from V by one rounding (rtol 1e-6).

What it detects: a row whose selected token is not read, or is read twice,
or is read from the wrong slot, and any read of a NaN-poisoned slot (NaN
reaches the row's output).  A misread block that no row selected from stays
invisible, since its tokens score far below the selected one.  So the
selections aim at the places where indexing goes wrong: besides uniform
picks, the first and last token of every segment (each prefix level and the
suffix), and each prefill row's causal boundary (the last token it sees).
A wrong level offset, block column, slot or chunk boundary shifts those
tokens in every request and is caught.  Attention does not depend on the
order of the tokens a row reads, so the set of tokens is what is checked.

The expected rows come from the oracle's gather (pinned against a dense
scatter in the oracle tests).  The CPU test checks the one-hot construction
itself: the oracle's attention over it gives the chosen V rows.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import workloads as W

BOOST = 64.0          # q = BOOST * code: exact in bf16 (a power of two times +-1)
MIN_MARGIN = 110.0    # natural-log units between the chosen score and any other
_BF16_ONE, _BF16_MINUS_ONE, _BF16_NAN = np.uint16(0x3F80), np.uint16(0xBF80), np.uint16(0x7FC0)


def _code_pool(p, seed):
    """Overwrite every used K slot of p.pool (in place) with a random +-1 code;
    unused (NaN-poisoned) slots stay NaN.  Block ranges one at a time to bound
    host memory on the full-size pools."""
    rng = np.random.default_rng([seed, 17])
    nb = p.pool.shape[0]
    step = 2048
    for b0 in range(0, nb, step):
        k = p.pool[b0:b0 + step, 0]
        bits = np.unpackbits(rng.integers(0, 256, size=(k.size + 7) // 8, dtype=np.uint8))
        neg = bits[:k.size].reshape(k.shape).astype(bool)
        if p.dtype == W.BF16:
            used = k != _BF16_NAN
            code = np.where(neg, _BF16_MINUS_ONE, _BF16_ONE)
        else:
            used = ~np.isnan(k)
            code = np.where(neg, np.float32(-1.0), np.float32(1.0))
        k[used] = code[used]


def _segment_edges(p, r):
    """Token indices of the first and last token of each segment of request
    r's token list: its prefix levels, root first, then its suffix."""
    lens = [int(p.prefix_len[g]) for g in p.chain(r)] + [int(p.suffix_len[r])]
    edges, start = [], 0
    for n in lens:
        if n > 0:
            edges += [start, start + n - 1]
        start += n
    return np.unique(np.asarray(edges, np.int64))


def _pick(rng, n_vis, edges):
    """Token a row selects among its first n_vis tokens: the last visible one
    (a prefill row's causal boundary, a decode row's last suffix token), a
    segment edge, or a uniform pick."""
    u = rng.random()
    if u < 0.2:
        return n_vis - 1
    e = edges[edges < n_vis]
    if u < 0.6 and e.size:
        return int(e[rng.integers(0, e.size)])
    return int(rng.integers(0, n_vis))


def one_hot(p, seed, q_len=None):
    """Make p's attention one-hot.  Codes p.pool's K slots in place.  Returns
    (q, expected_out float64 [rows][Hq][d], expected_lse float64 [rows][Hq]).
    Rows are the requests, or with q_len the prefill rows request by request:
    row i of request r sees the first n_tok - q_len[r] + i + 1 tokens."""
    _code_pool(p, seed)
    rng = np.random.default_rng([seed, 29])
    Hq, Hkv, d = p.num_q_heads, p.num_kv_heads, p.head_dim
    G = Hq // Hkv
    ql = np.ones(p.num_req, np.int64) if q_len is None else np.asarray(q_len, np.int64)
    rows = int(ql.sum())
    q = np.zeros((rows, Hq, d), np.float32)
    want = np.zeros((rows, Hq, d), np.float64)
    row0 = np.r_[0, np.cumsum(ql)[:-1]]
    for r in range(p.num_req):
        edges = _segment_edges(p, r)
        for kvh in range(Hkv):
            K, V = oracle.gather_kv(p, r, kvh)
            n = K.shape[0]
            assert edges[-1] == n - 1
            # selections of every (row, q head) reading this KV head
            js = np.array([[_pick(rng, n - int(ql[r]) + i + 1, edges) for _ in range(G)]
                           for i in range(int(ql[r]))])
            dots = K @ K[js.ravel()].T  # [n][rows * G]
            dots[js.ravel(), np.arange(js.size)] = -np.inf
            if n > 1:
                margin = p.scale * BOOST * (d - dots.max(axis=0))
                assert margin.min() >= MIN_MARGIN, (r, kvh, float(margin.min()))
            rr = row0[r] + np.arange(int(ql[r]))
            q[rr, kvh * G:(kvh + 1) * G] = BOOST * K[js]
            want[rr, kvh * G:(kvh + 1) * G] = V[js]
    lse = np.full((rows, Hq), p.scale * BOOST * d, np.float64)
    if p.dtype == W.BF16:
        q = W.f32_to_bf16_bits(q)
    return q, want, lse


def _compare(p, out, lse, want, want_lse):
    if p.dtype == W.BF16:
        bad = out != want  # both exact bf16 values held in float64
        assert not bad.any(), (f"{p.name}: {int(bad.sum())} outputs differ from the selected V "
                               f"rows, first at {np.argwhere(bad)[0].tolist()}")
    else:
        np.testing.assert_allclose(out, want, rtol=1e-6, atol=0)
    assert np.abs(lse - want_lse).max() <= 1e-3


# ---------------------------------------------------------------- CPU


@pytest.mark.parametrize("name", ["tiny_fp32", "llama8b", "long_prefix", "skewed", "two_level",
                                  "two_level_flat"])
def test_oracle_sees_one_hot(name):
    """The construction's premise, checked with the oracle: attention over the
    coded pool returns the selected V rows and LSE = scale * B * d."""
    p = W.make(name, small=name != "tiny_fp32")
    q, want, want_lse = one_hot(p, seed=3)  # the inputs of the small GPU cases
    o, l = oracle.attention(dataclasses.replace(p, q=q))
    assert np.abs(o - want).max() <= 1e-12
    assert np.abs(l - want_lse).max() <= 1e-9 * float(want_lse.max())


@pytest.mark.parametrize("seed", [6, 7])
def test_oracle_sees_one_hot_chunked(seed):
    p, ql, _ = W.make_chunked(seed=seed, small=True)
    q, want, want_lse = one_hot(p, seed=seed, q_len=ql)  # as the small GPU cases
    o, l = oracle.attention_chunked(p, ql, q)
    assert np.abs(o - want).max() <= 1e-12
    assert np.abs(l - want_lse).max() <= 1e-9 * float(want_lse.max())


# ---------------------------------------------------------------- GPU


def _run_decode(p, flags):
    from workloads.device import DeviceProblem
    d = DeviceProblem(p)
    with d.plan(flags) as pl:
        d.decode(pl)
        out, lse = d.result()
        rc, dev_flags = pl.status()
    assert rc == 0 and dev_flags == 0, (rc, dev_flags)
    return out, lse


SMALL = [(n, f) for n in ("tiny_fp32", "llama8b", "long_prefix", "skewed", "two_level",
                          "two_level_flat") for f in ("0",)] + \
        [(n, f) for n in ("llama8b", "skewed") for f in ("NO_DEDUP", "SIMT", "NO_TENSOR_PREFIX")] + \
        [("two_level", "NO_FOLD"), ("two_level", "FLATTEN")]


@pytest.mark.gpu
@pytest.mark.parametrize("name,flag", SMALL)
def test_gather_exact_small(name, flag):
    pytest.importorskip("torch")
    import shared_prefix_kv_gb300 as ps
    p = W.make(name, small=name != "tiny_fp32")
    q, want, want_lse = one_hot(p, seed=3)
    p = dataclasses.replace(p, q=q)
    out, lse = _run_decode(p, 0 if flag == "0" else getattr(ps, flag))
    _compare(p, out, lse, want, want_lse)


@pytest.mark.gpu
@pytest.mark.parametrize("name,flag", [("llama8b", "0"), ("long_prefix", "0"), ("skewed", "0"),
                                       ("two_level", "0"), ("two_level", "NO_FOLD")])
def test_gather_exact_full_size(name, flag):
    """Every output of the full-size batch, in the benchmark's launch
    configuration.  The two-level batch also runs with every level its own
    partial (NO_FOLD): its 4096 requests then merge three partials each (the
    shared level 1, their level-2 group, their suffix) in the one launch."""
    pytest.importorskip("torch")
    import shared_prefix_kv_gb300 as ps
    p = W.make(name)
    q, want, want_lse = one_hot(p, seed=4)
    p = dataclasses.replace(p, q=q)
    out, lse = _run_decode(p, 0 if flag == "0" else getattr(ps, flag))
    _compare(p, out, lse, want, want_lse)


@pytest.mark.gpu
def test_gather_exact_long_context():
    """The long-context batch (a 131072-token shared prefix, a 100000-token
    suffix): every chunk boundary of the long split-k spans."""
    pytest.importorskip("torch")
    from tests.test_decode_gpu import long_context_problem
    p = long_context_problem()
    q, want, want_lse = one_hot(p, seed=5)
    p = dataclasses.replace(p, q=q)
    out, lse = _run_decode(p, 0)
    _compare(p, out, lse, want, want_lse)


@pytest.mark.gpu
@pytest.mark.parametrize("flag", ["0", "NO_TENSOR_PREFIX"])
@pytest.mark.parametrize("seed,small", [(6, True), (7, True), (6, False)])
def test_gather_exact_chunked_ragged(seed, small, flag):
    """Prefill rows in the ragged form: per-row limits on the tensor-core
    tiles (or on the mma.sync items), each row's causal boundary token among
    the selections.  The full-size batch (seed 6, not small) is the
    benchmark's chunked-prefill batch: 7 chunks of 256-512 queries beside 256
    decode requests."""
    pytest.importorskip("torch")
    import shared_prefix_kv_gb300 as ps
    from shared_prefix_kv_gb300 import chunked as C
    from workloads.device import DeviceProblem, shape_of
    p, ql, _ = W.make_chunked(seed=seed, small=small)
    q, want, want_lse = one_hot(p, seed=seed, q_len=ql)
    sh, bt, gor, gpar, plen, slen, leaf = C.expand_ragged(
        shape_of(p), p.block_table, p.group_of_req, p.group_parent, p.prefix_len, p.suffix_len, ql)
    p2 = dataclasses.replace(p, name=p.name + "_ragged", q=q, block_table=bt, group_of_req=gor,
                             group_parent=gpar, prefix_len=plen, suffix_len=slen)
    d = DeviceProblem(p2)
    with ps.Plan(sh, bt, gor, gpar, plen, slen, flags=0 if flag == "0" else getattr(ps, flag),
                 leaf_len=leaf) as pl:
        d.decode(pl)
        out, lse = d.result()
        rc, dev_flags = pl.status()
    assert rc == 0 and dev_flags == 0, (rc, dev_flags)
    _compare(p, out, lse, want, want_lse)
