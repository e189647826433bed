"""Pins of the CPU oracle to things other than itself.

- hand-worked cases whose softmax weights are small rationals (golden file);
- brute force in 50-digit arithmetic without the max shift, on tiny inputs;
- closed forms (one token, zero query, identical keys, a dominant key);
- BatchLLM's split (papercache.org, section 2.2, Eq. 1): attention over a cut
  of the token list, merged by online softmax, equals attention over the
  whole list, for every cut point and for three-way cuts;
- a library special case: torch's scaled_dot_product_attention in float64 on
  the dense K/V that the test scatters into pages (multi-level chains, ragged
  segment ends, GQA).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.dense_pack import pack, single_request

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def _arr(x):
    return np.asarray(x, dtype=np.float64)


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_hand_worked_golden(case):
    Hkv, d = case["Hkv"], case["d"]
    levels = [(_arr(g["K"]), _arr(g["V"])) for g in case["groups"]]
    reqs = case["requests"]
    sufs = [(_arr(r["suffix_K"]), _arr(r["suffix_V"])) for r in reqs]
    q = np.stack([_arr(r["q"]) for r in reqs])
    p, _ = pack(levels, case["parent"], [r["group"] for r in reqs], sufs, q, Hkv=Hkv,
                B=case["B"], scale=case["scale"])
    out, lse = oracle.attention(p)
    np.testing.assert_allclose(out, _arr(case["expected_out"]), atol=case["tol"], rtol=0)
    np.testing.assert_allclose(lse, _arr(case["expected_lse"]), atol=case["tol"], rtol=0)


def _rand_f32(rng, *shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float32).astype(np.float64)


@pytest.mark.parametrize("seed", range(12))
def test_bruteforce_mpmath(seed):
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 9))
    d = int(rng.integers(1, 5))
    Hkv = int(rng.integers(1, 3))
    G = int(rng.integers(1, 3))
    K = _rand_f32(rng, Hkv, n, d, scale=2.0)
    V = _rand_f32(rng, Hkv, n, d)
    q = _rand_f32(rng, Hkv * G, d, scale=2.0)
    scale = float(np.float32(rng.uniform(0.2, 1.5)))
    p = single_request(K, V, q, B=3, scale=scale, seed=seed)
    out, lse = oracle.attention(p)
    for h in range(Hkv * G):
        kv = h // G
        w = [mp.exp(mp.mpf(scale) * mp.fsum(mp.mpf(q[h, e]) * mp.mpf(K[kv, t, e]) for e in range(d)))
             for t in range(n)]
        z = mp.fsum(w)
        assert abs(float(mp.log(z)) - lse[0, h]) < 1e-12
        for e in range(d):
            o = mp.fsum(w[t] * mp.mpf(V[kv, t, e]) for t in range(n)) / z
            assert abs(float(o) - out[0, h, e]) < 1e-12


def test_closed_form_single_token():
    rng = np.random.default_rng(1)
    K = _rand_f32(rng, 1, 1, 8)
    V = _rand_f32(rng, 1, 1, 8)
    q = _rand_f32(rng, 1, 8)
    p = single_request(K, V, q, scale=0.5)
    out, lse = oracle.attention(p)
    np.testing.assert_allclose(out[0, 0], V[0, 0], rtol=0, atol=1e-15)
    assert lse[0, 0] == pytest.approx(0.5 * float(q[0] @ K[0, 0]), abs=1e-13)


def test_closed_form_zero_query_is_mean():
    rng = np.random.default_rng(2)
    n = 37
    K = _rand_f32(rng, 2, n, 16, scale=3.0)
    V = _rand_f32(rng, 2, n, 16)
    q = np.zeros((4, 16))
    p = single_request(K, V, q, B=8)
    out, lse = oracle.attention(p)
    for h in range(4):
        np.testing.assert_allclose(out[0, h], V[h // 2].mean(axis=0), atol=1e-13)
        assert lse[0, h] == pytest.approx(math.log(n), abs=1e-13)


def test_closed_form_identical_keys():
    rng = np.random.default_rng(3)
    n, d = 21, 8
    k = _rand_f32(rng, d)
    K = np.broadcast_to(k, (1, n, d)).copy()
    V = _rand_f32(rng, 1, n, d)
    q = _rand_f32(rng, 1, d)
    p = single_request(K, V, q, B=4, scale=0.25)
    out, lse = oracle.attention(p)
    np.testing.assert_allclose(out[0, 0], V[0].mean(axis=0), atol=1e-13)
    assert lse[0, 0] == pytest.approx(0.25 * float(q[0] @ k) + math.log(n), abs=1e-12)


def test_closed_form_dominant_key():
    rng = np.random.default_rng(4)
    n, d = 50, 4
    K = _rand_f32(rng, 1, n, d, scale=0.1)
    K[0, 17] = [40.0, 0, 0, 0]
    V = _rand_f32(rng, 1, n, d)
    q = np.array([[1.0, 0, 0, 0]])
    p = single_request(K, V, q, B=16, scale=1.0)
    out, lse = oracle.attention(p)
    np.testing.assert_allclose(out[0, 0], V[0, 17], atol=1e-14)
    assert lse[0, 0] == pytest.approx(40.0, abs=1e-12)


def _merge(parts):
    """Online-softmax reduction of partial results (Milakov & Gimelshein, cited by
    BatchLLM section 2.2): each part is (out normalised over its tokens, lse)."""
    m = max(l for _, l in parts)
    w = [math.exp(l - m) for _, l in parts]
    z = sum(w)
    return sum(wi * o for wi, (o, _) in zip(w, parts)) / z, m + math.log(z)


def test_split_merge_equals_unsplit_every_cut():
    rng = np.random.default_rng(5)
    n, d = 23, 6
    K = _rand_f32(rng, 1, n, d, scale=1.5)
    V = _rand_f32(rng, 1, n, d)
    q = _rand_f32(rng, 1, d, scale=1.5)
    full_o, full_l = oracle.attention(single_request(K, V, q, B=4))
    for c in range(1, n):
        a = oracle.attention(single_request(K[:, :c], V[:, :c], q, B=4, seed=c))
        b = oracle.attention(single_request(K[:, c:], V[:, c:], q, B=4, seed=c + 100))
        o, l = _merge([(a[0][0, 0], a[1][0, 0]), (b[0][0, 0], b[1][0, 0])])
        np.testing.assert_allclose(o, full_o[0, 0], atol=1e-12)
        assert l == pytest.approx(full_l[0, 0], abs=1e-12)


def test_split_merge_three_way():
    rng = np.random.default_rng(6)
    n, d = 40, 5
    K = _rand_f32(rng, 1, n, d, scale=2.0)
    V = _rand_f32(rng, 1, n, d)
    q = _rand_f32(rng, 1, d)
    full_o, full_l = oracle.attention(single_request(K, V, q, B=8))
    for c1, c2 in [(1, 2), (5, 33), (16, 32), (38, 39), (13, 14)]:
        parts = []
        for lo, hi in [(0, c1), (c1, c2), (c2, n)]:
            o, l = oracle.attention(single_request(K[:, lo:hi], V[:, lo:hi], q, B=8, seed=lo))
            parts.append((o[0, 0], l[0, 0]))
        o, l = _merge(parts)
        np.testing.assert_allclose(o, full_o[0, 0], atol=1e-12)
        assert l == pytest.approx(full_l[0, 0], abs=1e-12)


def _sdpa(q, K, V, scale):
    """torch SDPA in float64: q [Hq][d], K/V [Hkv][n][d] with q head h reading KV
    head h // (Hq/Hkv)."""
    G = q.shape[0] // K.shape[0]
    Kt = torch.from_numpy(K).repeat_interleave(G, dim=0)
    Vt = torch.from_numpy(V).repeat_interleave(G, dim=0)
    qt = torch.from_numpy(q)[:, None, :]
    o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=scale)
    lse = torch.logsumexp((qt @ Kt.transpose(1, 2)).squeeze(1) * scale, dim=-1)
    return o[:, 0, :].numpy(), lse.numpy()


@pytest.mark.parametrize("seed", range(4))
def test_sdpa_library_case_multilevel_gqa(seed):
    rng = np.random.default_rng(100 + seed)
    Hkv, G, d, B = 2, 3, 16, 4
    # level lengths deliberately not multiples of B: segments start at fresh blocks
    plen = [7, 5, 0, 9]
    parent = [-1, 0, -1, 2]
    levels = [(_rand_f32(rng, Hkv, n, d), _rand_f32(rng, Hkv, n, d)) for n in plen]
    members = [1, 3, -1, 0, 2, 1]
    sufs = []
    for r in range(len(members)):
        s = int(rng.integers(0 if members[r] >= 0 else 1, 11))
        sufs.append((_rand_f32(rng, Hkv, s, d), _rand_f32(rng, Hkv, s, d)))
    q = _rand_f32(rng, len(members), Hkv * G, d)
    p, dense = pack(levels, parent, members, sufs, q, Hkv=Hkv, B=B, seed=seed)
    out, lse = oracle.attention(p)
    for r in range(len(members)):
        o_ref, l_ref = _sdpa(q[r], dense[r][0], dense[r][1], p.scale)
        np.testing.assert_allclose(out[r], o_ref, atol=1e-12)
        np.testing.assert_allclose(lse[r], l_ref, atol=1e-12)


def test_sdpa_library_case_bf16_storage():
    rng = np.random.default_rng(7)
    Hkv, G, d, B = 2, 4, 32, 16
    f = lambda *s: W.bf16_bits_to_f32(W.f32_to_bf16_bits(rng.standard_normal(s))).astype(np.float64)
    levels = [(f(Hkv, 40, d), f(Hkv, 40, d))]
    sufs = [(f(Hkv, 3, d), f(Hkv, 3, d)), (f(Hkv, 18, d), f(Hkv, 18, d))]
    q = f(2, Hkv * G, d)
    p, dense = pack(levels, None, [0, 0], sufs, q, Hkv=Hkv, B=B, dtype=W.BF16)
    out, lse = oracle.attention(p)
    for r in range(2):
        o_ref, l_ref = _sdpa(q[r], dense[r][0], dense[r][1], p.scale)
        np.testing.assert_allclose(out[r], o_ref, atol=1e-12)
        np.testing.assert_allclose(lse[r], l_ref, atol=1e-12)


def test_gather_matches_scatter():
    rng = np.random.default_rng(8)
    levels = [(_rand_f32(rng, 2, 9, 8), _rand_f32(rng, 2, 9, 8))]
    sufs = [(_rand_f32(rng, 2, 5, 8), _rand_f32(rng, 2, 5, 8))]
    p, dense = pack(levels, None, [0], sufs, _rand_f32(rng, 1, 2, 8), Hkv=2, B=4)
    for h in range(2):
        K, V = oracle.gather_kv(p, 0, h)
        np.testing.assert_array_equal(K, dense[0][0][h])
        np.testing.assert_array_equal(V, dense[0][1][h])


def test_oracle_thread_count_invariant():
    p = W.make("skewed", small=True)
    req = list(range(0, p.num_req, 7))
    a = oracle.attention(p, req, nthreads=1)
    b = oracle.attention(p, req, nthreads=4)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_oracle_subset_matches_full():
    p = W.make("tiny_fp32")
    full = oracle.attention(p)
    sub = oracle.attention(p, [3, 0, 11])
    np.testing.assert_array_equal(sub[0], full[0][[3, 0, 11]])


def test_oracle_rejects_bad_block():
    p = W.make("tiny_fp32")
    p.block_table[2, 0] = p.num_pool_blocks + 5
    with pytest.raises(oracle.OracleError):
        oracle.attention(p)


def test_oracle_never_reads_poison():
    # NaN-poisoned unused slots and blocks never reach the output
    for name in ("tiny_fp32", "skewed", "two_level"):
        p = W.make(name, small=True)
        out, lse = oracle.attention(p, list(range(0, p.num_req, 5)))
        assert np.isfinite(out).all() and np.isfinite(lse).all()


# ---- chunked prefill (oracle.attention_chunked): query i of a chunk of n
# queries attends to the first n_tok - n + i + 1 tokens of its request

def _causal_dense(K, V, q, scale, n_q):
    """K, V [Hkv][n][d] of one request, q [n_q][Hq][d] its chunk's queries."""
    Hkv, n, _ = K.shape
    Hq = q.shape[1]
    G = Hq // Hkv
    out = np.zeros(q.shape)
    lse = np.zeros(q.shape[:2])
    for i in range(n_q):
        vis = n - n_q + i + 1
        for h in range(Hq):
            s = (K[h // G, :vis] @ q[i, h]) * scale
            m = s.max()
            w = np.exp(s - m)
            out[i, h] = (w / w.sum()) @ V[h // G, :vis]
            lse[i, h] = m + np.log(w.sum())
    return out, lse


@pytest.mark.parametrize("seed", range(8))
def test_chunked_matches_dense_causal(seed):
    rng = np.random.default_rng(500 + seed)
    Hkv, G, d, B = 2, 2, 8, 4
    P0 = int(rng.integers(0, 9))
    levels = [(_rand_f32(rng, Hkv, P0, d), _rand_f32(rng, Hkv, P0, d))]
    R = 4
    sl = rng.integers(1, 12, R)
    ql = np.array([int(rng.integers(1, s + 1)) for s in sl])
    members = [int(rng.integers(-1, 1)) for _ in range(R)]
    sufs = [(_rand_f32(rng, Hkv, s, d), _rand_f32(rng, Hkv, s, d)) for s in sl]
    q_dec = _rand_f32(rng, R, Hkv * G, d)
    p, dense = pack(levels, None, members, sufs, q_dec, Hkv=Hkv, B=B, seed=seed)
    qc = _rand_f32(rng, int(ql.sum()), Hkv * G, d)
    out, lse = oracle.attention_chunked(p, ql, qc.astype(np.float32))
    row = 0
    for r in range(R):
        K, V = dense[r]
        eo, el = _causal_dense(K, V, qc[row:row + ql[r]], p.scale, int(ql[r]))
        np.testing.assert_allclose(out[row:row + ql[r]], eo, atol=1e-12, rtol=0)
        np.testing.assert_allclose(lse[row:row + ql[r]], el, atol=1e-12, rtol=0)
        row += ql[r]


def test_chunked_one_query_is_decode():
    p = W.make("skewed", small=True)
    ones = np.ones(p.num_req, np.int32)
    out, lse = oracle.attention_chunked(p, ones, p.q)
    eo, el = oracle.attention(p)
    assert np.array_equal(out, eo) and np.array_equal(lse, el)


def test_chunked_first_query_sees_its_first_token():
    # no prefix, the chunk is the whole suffix: query 0 sees token 0 only
    rng = np.random.default_rng(3)
    K = _rand_f32(rng, 1, 5, 4)
    V = _rand_f32(rng, 1, 5, 4)
    p = single_request(K, V, _rand_f32(rng, 1, 4), B=2)
    qc = _rand_f32(rng, 5, 1, 4).astype(np.float32)
    out, lse = oracle.attention_chunked(p, [5], qc)
    assert np.array_equal(out[0, 0], V[0, 0])
    assert lse[0, 0] == pytest.approx(float(qc[0, 0] @ K[0, 0]) * p.scale, abs=1e-13)
    # the last query sees all five, as a decode query would
    p.q = qc[4:5].copy()
    eo, el = oracle.attention(p)
    assert np.array_equal(out[4], eo[0]) and np.array_equal(lse[4], el[0])


def test_chunked_rejects_chunk_longer_than_request():
    p = W.make("tiny_fp32", small=True)
    ql = np.ones(p.num_req, np.int32)
    ql[0] = int(oracle.gather_kv(p, 0, 0)[0].shape[0]) + 1
    with pytest.raises(oracle.OracleError):
        oracle.attention_chunked(p, ql, np.zeros((int(ql.sum()), p.num_q_heads, p.head_dim),
                                                 np.float32))
