"""Token batches (include/psattn_sched.h) against a plain simulation.

The simulation below is written from the rules of BatchLLM section 4.3 as the
header states them, request by request and iteration by iteration, without
the library's queues: each iteration it re-scans every request for decode
tokens, distinct-prompt chunks and prefix chunks.  The library must produce
the same admission order and the same per-iteration token counts, request
counts and resident KV tokens.  Invariants (every token processed once, the
N_chunk and request-count caps, prefix before distinct prompt) are checked
on the library's output directly.
"""
import numpy as np
import pytest

from shared_prefix_kv_gb300 import sched as S
import shared_prefix_kv_gb300 as ps


def simulate(group_prefix, gor, dl, ol, n_chunk, m_thr=-1, max_req=0, reorder=False):
    R, NG = len(gor), len(group_prefix)
    groups, where = [], {}
    for r in range(R):
        g = int(gor[r])
        if g < 0:
            groups.append((NG + r, 0, [r]))
        else:
            if g not in where:
                where[g] = len(groups)
                groups.append((g, int(group_prefix[g]), []))
            groups[where[g]][2].append(r)
    keys = [p + sum(int(dl[r]) for r in m) for _, p, m in groups]
    order = list(range(len(groups)))
    if reorder:
        order.sort(key=lambda i: (keys[i], i))
    rank = {gi: k for k, gi in enumerate(order)}
    rank_of = [0] * R
    for gi, (_, _, m) in enumerate(groups):
        for r in m:
            rank_of[r] = rank[gi]
    prompt = [int(x) for x in dl]
    out = [int(x) for x in ol]
    own = [0] * R
    elig = [None] * R
    dec_at = [None] * R
    done = [False] * R
    pre_done = [0] * len(order)
    left = [len(groups[gi][2]) for gi in order]
    cur, resident, t = 0, 0, 0
    toks, mems = [], []
    while not all(done):
        budget, nreq, nd, nds, npf = n_chunk, 0, 0, 0, 0
        fin = []

        def room():
            return max_req == 0 or nreq < max_req

        def fits(c):
            return nreq == 0 or m_thr < 0 or resident + c <= m_thr

        for r in sorted((r for r in range(R) if dec_at[r] is not None and not done[r]
                         and dec_at[r] <= t and out[r] > 0), key=lambda r: (dec_at[r], r)):
            if budget == 0 or not room():
                break
            budget -= 1; nreq += 1; nd += 1; resident += 1; own[r] += 1; out[r] -= 1
            if out[r] == 0:
                fin.append(r)
        open_ = True
        for r in sorted(range(R), key=lambda r: (rank_of[r], r)):
            if budget == 0 or not room():
                break
            if elig[r] is None or elig[r] > t or prompt[r] == 0:
                continue
            c = min(prompt[r], budget)
            if not fits(c):
                open_ = False
                break
            budget -= c; nreq += 1; nds += c; resident += c; own[r] += c; prompt[r] -= c
            if prompt[r] == 0:
                dec_at[r] = t + 1
        while open_ and cur < len(order):
            _, p, members = groups[order[cur]]
            rem = p - pre_done[cur]
            if rem > 0:
                if budget == 0 or not room():
                    break
                c = min(rem, budget)
                if not fits(c):
                    break
                budget -= c; nreq += 1; npf += c; resident += c; pre_done[cur] += c
                if pre_done[cur] < p:
                    break
            for r in members:
                elig[r] = t + 1
                if prompt[r] == 0:
                    dec_at[r] = t + 1
            cur += 1
        toks.append((nd, nds, npf, nreq))
        mems.append(resident)
        for r in fin:
            done[r] = True
            resident -= own[r]
            k = rank_of[r]
            left[k] -= 1
            if left[k] == 0:
                resident -= groups[order[k]][1]
        t += 1
    return [groups[gi][0] for gi in order], np.array(toks, np.int32).reshape(-1, 4), np.array(mems)


def random_case(rng, NG=None, R=None):
    NG = int(rng.integers(0, 6)) if NG is None else NG
    R = int(rng.integers(1, 14)) if R is None else R
    gp = rng.integers(0, 60, NG)
    gor = rng.integers(-1, max(NG, 1), R) if NG else -np.ones(R, int)
    dl = rng.integers(0, 40, R)
    ol = rng.integers(1, 12, R)
    return gp, gor, dl, ol


def check(gp, gor, dl, ol, **kw):
    got = S.token_batches(gp, gor, dl, ol, **kw)
    exp = simulate(gp, gor, dl, ol, kw["n_chunk"], kw.get("m_threshold", -1),
                   kw.get("max_requests", 0), kw.get("reorder", False))
    assert got[0].tolist() == exp[0]
    assert got[1].tolist() == exp[1].tolist()
    assert got[2].tolist() == exp[2].tolist()
    # invariants on the library's own output
    order, tok, mem = got
    used = set(int(g) for g in np.asarray(gor) if g >= 0)
    assert tok[:, 0].sum() == np.sum(ol)
    assert tok[:, 1].sum() == np.sum(dl)
    assert tok[:, 2].sum() == sum(int(gp[g]) for g in used)
    assert (tok[:, :3].sum(axis=1) <= kw["n_chunk"]).all()
    if kw.get("max_requests", 0):
        assert (tok[:, 3] <= kw["max_requests"]).all()
    assert (mem >= 0).all()
    return got


@pytest.mark.parametrize("seed", range(60))
def test_matches_simulation(seed):
    rng = np.random.default_rng(seed)
    gp, gor, dl, ol = random_case(rng)
    n_chunk = int(rng.integers(1, 64))
    m_thr = int(rng.choice([-1, int(rng.integers(0, 200))]))
    max_req = int(rng.choice([0, int(rng.integers(1, 6))]))
    check(gp, gor, dl, ol, n_chunk=n_chunk, m_threshold=m_thr, max_requests=max_req,
          reorder=bool(seed % 2))


def test_reorder_is_r_group_order():
    # R_group = 1 / (L_prefix + sum L_distinct): groups with fewer prompt tokens first
    gp = [100, 10, 50]
    gor = [0, 1, 2, 1, -1, 0]
    dl = [5, 80, 1, 30, 20, 5]
    ol = [1] * 6
    order, _, _ = check(gp, gor, dl, ol, n_chunk=64, reorder=True)
    keys = {0: 110, 1: 120, 2: 51, 3 + 4: 20}
    assert order.tolist() == sorted(keys, key=lambda g: (keys[g], [0, 1, 2, 7].index(g)))
    order, _, _ = check(gp, gor, dl, ol, n_chunk=64, reorder=False)
    assert order.tolist() == [0, 1, 2, 7]  # input order: first member 0, 1, 2, 4


def test_prefix_before_distinct_and_decode_first():
    # one group: 30 prefix tokens, two requests of 10 distinct tokens and 3 outputs
    _, tok, mem = check([30], [0, 0], [10, 10], [3, 3], n_chunk=16)
    # it 0: 16 prefix; it 1: 14 prefix (group complete); it 2: distinct 10 + 6;
    # it 3: 4 distinct; request 0 decodes from it 3 on
    assert tok[0].tolist() == [0, 0, 16, 1]
    assert tok[1].tolist() == [0, 0, 14, 1]
    assert tok[2].tolist() == [0, 16, 0, 2]
    assert tok[3].tolist() == [1, 4, 0, 2]
    assert tok[4].tolist() == [2, 0, 0, 2]
    # request 0 is freed after its third output (iteration 5); the last
    # iteration holds the prefix and request 1's 10 + 3 tokens
    assert mem[5] == 30 + (10 + 3) + (10 + 2)
    assert mem[-1] == 30 + 10 + 3


def test_memory_gate_holds_prefill_back():
    # each prompt is 40 tokens; a threshold of 90 lets two prompts in at a time
    # (requests without a group are admitted in iteration 0 and start the next)
    gor = [-1] * 4
    _, tok, mem = check([], gor, [40] * 4, [5] * 4, n_chunk=200, m_threshold=90)
    assert tok[0].tolist() == [0, 0, 0, 0]
    assert tok[1].tolist() == [0, 80, 0, 2]
    # the other two prompts wait until the first two have finished (their
    # outputs in iterations 2-6 keep memory above 50)
    again = next(i for i in range(2, len(tok)) if tok[i, 1] > 0)
    assert again == 7 and tok[again, 1] == 80
    assert mem[6] == 90


def test_request_cap_versus_memory_centric():
    # 300 decode-heavy requests under one prefix, then long prompts: with a
    # cap of 256 requests per batch the decode tokens fill every batch; the
    # memory-centric batch keeps adding prefill while memory lasts
    rng = np.random.default_rng(5)
    R = 600
    gor = np.r_[np.zeros(300, int), -np.ones(300, int)]
    dl = np.r_[np.full(300, 8), rng.integers(200, 400, 300)]
    ol = np.r_[np.full(300, 64), np.full(300, 4)]
    kw = dict(n_chunk=2048, m_threshold=400_000)
    _, cap_tok, _ = check([512], gor, dl, ol, max_requests=256, **kw)
    _, mem_tok, _ = check([512], gor, dl, ol, **kw)
    assert len(mem_tok) < len(cap_tok)
    assert mem_tok[:, :3].sum(axis=1).mean() > cap_tok[:, :3].sum(axis=1).mean()


def test_edge_cases():
    check([], [], [], [], n_chunk=1)
    check([0], [0], [0], [1], n_chunk=1)
    check([5, 7], [-1, -1], [0, 0], [1, 2], n_chunk=1)  # groups without requests
    check([3], [0, 0, 0], [0, 0, 0], [1, 1, 1], n_chunk=1, max_requests=1)
    check([1000], [0], [1000], [1], n_chunk=7, m_threshold=1)  # only the empty-batch rule admits


def test_invalid_arguments():
    with pytest.raises(ps.PsattnError):
        S.token_batches([1], [1], [1], [1], n_chunk=4)  # group id out of range
    with pytest.raises(ps.PsattnError):
        S.token_batches([1], [0], [1], [0], n_chunk=4)  # decode_len < 1
    with pytest.raises(ps.PsattnError):
        S.token_batches([1], [0], [1], [1], n_chunk=0)
    with pytest.raises(ps.PsattnError):
        S.token_batches([-1], [0], [1], [1], n_chunk=4)


def test_total_tokens_limit():
    """Iterations are counted in int32, so a batch may hold at most 2^29
    tokens in all (each used group's prefix once, every prompt and output).
    One token more is rejected before any simulation; the limit itself runs."""
    with pytest.raises(ps.PsattnError) as e:
        S.token_batches([], [-1, -1], [10, 10], [2 ** 30, 3], n_chunk=512)
    assert e.value.status == ps.ERR_INVALID_ARG
    with pytest.raises(ps.PsattnError):  # a prefix counts once, but counts
        S.token_batches([2 ** 29 - 5], [0, 0], [3, 3], [1, 1], n_chunk=512)
    order, tok, mem = S.token_batches([2 ** 29 - 8], [0, 0], [3, 3], [1, 1], n_chunk=2 ** 28)
    assert tok[:, 2].sum() == 2 ** 29 - 8 and tok[:, 1].sum() == 6
