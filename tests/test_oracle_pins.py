"""Pins for the fp64 oracle: each test checks it against something other than
itself -- numbers printed on the pages, closed forms, library routines that
compute special cases, brute force on tiny inputs, or an independent
streaming formulation.  No GPU involved."""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import bsfa_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _sdpa(q, k, v, mask=None, causal=False, sigma=None):
    """torch CPU fp64 scaled_dot_product_attention over [H, L, d] arrays."""
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x)) for x in (q, k, v))
    m = None if mask is None else torch.from_numpy(mask)
    out = torch.nn.functional.scaled_dot_product_attention(
        tq[None], tk[None], tv[None], attn_mask=m, is_causal=causal, scale=sigma)
    return out[0].numpy()


def _repeat_kv(x, g):
    return np.repeat(x, g, axis=0)


# ---------------------------------------------------------------------------
# The page's worked example (Block Sparse Flash Attention, "A Worked Example")
# ---------------------------------------------------------------------------
def _worked_inputs(keys_cand, diag_key=0.5):
    keys = list(keys_cand) + [diag_key]
    L = len(keys)
    q = np.ones((1, L, 1))
    k = np.array(keys, dtype=np.float64).reshape(1, L, 1)
    v = np.arange(10.0, 10.0 * (L + 1), 10.0).reshape(1, L, 1)
    return q, k, v


def test_worked_example_keep_set_and_output():
    g = _load("worked_example.json")
    q, k, v = _worked_inputs(g["candidate_block_maxima"])
    L = q.shape[1]
    T = np.full((1, L), -np.inf)
    T[0, L - 1] = g["threshold"]
    r = orc.prefill(q, k, v, Bq=1, Bk=1, sigma=1.0, thresholds=T)
    i = L - 1
    cand = g["candidate_block_maxima"]
    kept = [cand[j] for j in range(len(cand)) if r["keep"][0, i, j]]
    skipped = [cand[j] for j in range(len(cand)) if not r["keep"][0, i, j]]
    assert sorted(kept) == sorted(g["expected_kept_maxima"])
    assert sorted(skipped) == sorted(g["expected_skipped_maxima"])
    assert len(kept) == g["expected_kept_count"]
    assert r["keep"][0, i, i]  # diagonal region kept on top
    # Renormalisation over kept keys only: closed form with the page's numbers.
    s = [c for c in cand if c >= g["threshold"]] + [0.5]
    vals = [v[0, j, 0] for j in range(len(cand)) if cand[j] >= g["threshold"]] + [v[0, i, 0]]
    num = sum(math.exp(x) * y for x, y in zip(s, vals))
    den = sum(math.exp(x) for x in s)
    assert abs(r["out"][0, i, 0] - num / den) < 1e-12
    assert abs(r["lse"][0, i] - math.log(den)) < 1e-12


def test_worked_example_calibration_kth():
    g = _load("worked_example.json")
    q, k, _ = _worked_inputs(g["candidate_block_maxima"])
    T = orc.calibrate([q], [k], Bq=1, Bk=1, ks=[g["budget_k"]], sigma=1.0)
    assert T[0, 0, -1] == g["kth_largest_for_budget"]
    # fewer than k = 2 candidates at query blocks 0 and 1 -> -inf
    assert T[0, 0, 0] == -np.inf and T[0, 0, 1] == -np.inf
    # query block 2 sees candidates {1, 4}: 2nd largest is 1
    assert T[0, 0, 2] == 1.0


# ---------------------------------------------------------------------------
# lambda mode ("Vote, then skip")
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", ["main", "boundary"])
def test_lambda_hand_example(case):
    g = _load("lambda_vote_example.json")
    keys = g["keys"] if case == "main" else g["boundary_case"]["keys"]
    expect = g["expected_kept"] if case == "main" else g["boundary_case"]["expected_kept"]
    L = len(keys)
    q = np.ones((1, L, 1))
    k = np.array(keys).reshape(1, L, 1)
    v = _rand((1, L, 1), 3)
    r = orc.prefill(q, k, v, Bq=1, Bk=1, sigma=1.0, mode="lambda",
                    log_lambda=g["log_lambda"])
    kept = [j for j in range(L) if r["keep"][0, L - 1, j]]
    assert kept == expect


def _stat(x):
    return math.inf if x == "inf" else float(x)


def test_lambda_skipped_block_never_raises_the_running_max():
    """With ln(lambda) > 0 a skipped block can lie above the running max; it
    must still leave it alone (hand trace)."""
    g = _load("lambda_vote_example.json")["positive_log_lambda"]
    keys = g["keys"]
    L = len(keys)
    q, k = np.ones((L, 1)), np.array(keys).reshape(L, 1)
    got = orc.decision_statistics(q, k, L - 1, 1, 1, 1.0, log_lambda=g["log_lambda"])
    assert [x for _, x in got] == [_stat(x) for x in g["expected_statistics"]]
    r = orc.prefill(q[None], k[None], np.ones((1, L, 1)), Bq=1, Bk=1, sigma=1.0, mode="lambda",
                    log_lambda=g["log_lambda"])
    assert [j for j in range(L) if r["keep"][0, L - 1, j]] == g["expected_kept"]


@pytest.mark.parametrize("case", ["main", "boundary"])
def test_lambda_decision_statistics_hand_trace(case):
    """The decision statistic of every candidate, max_r(rowmax_r - m_r) with
    m_r taken before the block is visited, equals the hand trace (a running
    max read after the update would give 0 for every kept block)."""
    g = _load("lambda_vote_example.json")
    keys = g["keys"] if case == "main" else g["boundary_case"]["keys"]
    expect = (g["expected_statistics"]["values"] if case == "main"
              else g["boundary_case"]["expected_statistics"])
    L = len(keys)
    q = np.ones((L, 1))
    k = np.array(keys).reshape(L, 1)
    got = orc.decision_statistics(q, k, L - 1, 1, 1, 1.0, log_lambda=g["log_lambda"])
    assert [j for j, _ in got] == list(range(L - 1))
    assert [x for _, x in got] == [_stat(x) for x in expect]


def test_lambda_decision_statistics_two_rows():
    """Two rows with opposite queries: the statistic is the maximum over rows
    of each row's own difference, with skips leaving the running max alone."""
    g = _load("lambda_vote_example.json")["two_rows"]
    keys = g["keys"]
    L = len(keys)
    q = np.array([0.0, 0.0, 0.0, 0.0, 1.0, -1.0]).reshape(L, 1)
    k = np.array(keys).reshape(L, 1)
    got = orc.decision_statistics(q, k, 2, 2, 1, 1.0, log_lambda=g["log_lambda"])
    assert [j for j, _ in got] == [0, 1, 2, 3]
    assert [x for _, x in got] == [_stat(x) for x in g["expected_statistics"]]
    r = orc.prefill(q[None], k[None], np.ones((1, L, 1)), Bq=2, Bk=1, sigma=1.0, mode="lambda",
                    log_lambda=g["log_lambda"])
    assert [j for j in range(L) if r["keep"][0, 2, j]] == g["expected_kept"]
    # the keep decision is the statistic against ln(lambda), block by block
    for j, x in got:
        assert bool(r["keep"][0, 2, j]) == (x >= g["log_lambda"])


@pytest.mark.parametrize("Bq,Bk,L", [(4, 4, 37), (8, 4, 40), (4, 8, 33)])
def test_lambda_skipped_weights_bounded(Bq, Bk, L):
    """Every post-softmax weight in a skipped block is below lambda."""
    Hq, Hkv, d = 2, 1, 8
    q, k, v = _rand((Hq, L, d), 1), _rand((Hkv, L, d), 2), _rand((Hkv, L, d), 3)
    for j in range(1, orc.num_blocks(L, Bk), 2):  # make some key blocks skippable
        k[:, j * Bk:(j + 1) * Bk] *= 0.01
    q *= 2.0
    loglam = -0.3
    sigma = 1 / math.sqrt(d)
    r = orc.prefill(q, k, v, Bq=Bq, Bk=Bk, sigma=sigma, mode="lambda", log_lambda=loglam)
    n_skipped = 0
    for h in range(Hq):
        s = sigma * q[h] @ k[0].T
        for i in range(orc.num_blocks(L, Bq)):
            rows = range(i * Bq, min((i + 1) * Bq, L))
            for j in range(orc.num_blocks(L, Bk)):
                if not r["visible"][h, i, j] or r["keep"][h, i, j]:
                    continue
                n_skipped += 1
                for rr in rows:
                    cols = [c for c in range(j * Bk, min((j + 1) * Bk, L)) if c <= rr]
                    w = np.exp(s[rr, cols] - r["lse"][h, rr])
                    assert np.all(w < math.exp(loglam))
    assert n_skipped > 0


def test_lambda_limits():
    """ln(lambda) = -inf keeps everything (dense); ln(lambda) = +inf keeps the
    first visited candidate (running max starts at -inf) and the diagonal."""
    Hq, L, d, B = 2, 48, 8, 8
    q, k, v = _rand((Hq, L, d), 4), _rand((Hq, L, d), 5), _rand((Hq, L, d), 6)
    sigma = 1 / math.sqrt(d)
    dense = _sdpa(q, k, v, causal=True, sigma=sigma)
    r = orc.prefill(q, k, v, Bq=B, Bk=B, sigma=sigma, mode="lambda", log_lambda=-math.inf)
    assert np.max(np.abs(r["out"] - dense)) < 1e-12
    r = orc.prefill(q, k, v, Bq=B, Bk=B, sigma=sigma, mode="lambda", log_lambda=math.inf)
    mask = np.zeros((L, L), dtype=bool)
    for rr in range(L):
        for c in range(rr + 1):
            if c // B == rr // B or c // B == 0:
                mask[rr, c] = True
    assert np.max(np.abs(r["out"] - _sdpa(q, k, v, mask=mask, sigma=sigma))) < 1e-12


# ---------------------------------------------------------------------------
# Special cases that reduce to library routines
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("Hq,Hkv,L,d,Bq,Bk", [
    (2, 2, 64, 16, 16, 16), (4, 2, 77, 8, 8, 8), (4, 1, 50, 8, 16, 8), (2, 2, 45, 8, 4, 16)])
def test_threshold_minus_inf_is_dense_causal(Hq, Hkv, L, d, Bq, Bk):
    q, k, v = _rand((Hq, L, d), 7), _rand((Hkv, L, d), 8), _rand((Hkv, L, d), 9)
    sigma = 1 / math.sqrt(d)
    T = np.full((Hq, 3), -np.inf)
    r = orc.prefill(q, k, v, Bq=Bq, Bk=Bk, thresholds=T)
    g = Hq // Hkv
    ref = _sdpa(q, _repeat_kv(k, g), _repeat_kv(v, g), causal=True, sigma=sigma)
    assert np.max(np.abs(r["out"] - ref)) < 1e-12
    # log-sum-exp of the causal scores (library logsumexp)
    s = torch.from_numpy(sigma * np.einsum("hld,hmd->hlm", q, _repeat_kv(k, g)))
    s = s.masked_fill(~torch.ones(L, L, dtype=torch.bool).tril(), -math.inf)
    assert np.max(np.abs(r["lse"] - torch.logsumexp(s, -1).numpy())) < 1e-12
    assert r["keep"][r["visible"]].all()


# Diagonal-region masks written out by hand for tiny unequal tiles.
# Bq=4, Bk=2, L=8: rows 0-3 see key blocks {0,1} as diagonal; rows 4-7 see
# blocks 0,1 as candidates and {2,3} as diagonal -> keys 4..r.
# Bq=2, Bk=4, L=8: rows 0-3 have key block 0 diagonal; rows 4-7 have block 0
# as a candidate and block 1 diagonal -> keys 4..r.
HAND_DIAG_WINDOWS = {(4, 2): [0, 0, 0, 0, 4, 4, 4, 4], (2, 4): [0, 0, 0, 0, 4, 4, 4, 4],
                     (4, 4): [0, 0, 0, 0, 4, 4, 4, 4], (2, 2): [0, 0, 2, 2, 4, 4, 6, 6]}


@pytest.mark.parametrize("BqBk", sorted(HAND_DIAG_WINDOWS))
def test_threshold_plus_inf_is_diagonal_only(BqBk):
    Bq, Bk = BqBk
    Hq, L, d = 2, 8, 4
    q, k, v = _rand((Hq, L, d), 10), _rand((Hq, L, d), 11), _rand((Hq, L, d), 12)
    sigma = 1 / math.sqrt(d)
    T = np.full((Hq, 4), np.inf)
    r = orc.prefill(q, k, v, Bq=Bq, Bk=Bk, thresholds=T)
    first = HAND_DIAG_WINDOWS[BqBk]
    mask = np.array([[first[rr] <= c <= rr for c in range(L)] for rr in range(L)])
    assert np.max(np.abs(r["out"] - _sdpa(q, k, v, mask=mask, sigma=sigma))) < 1e-12


@pytest.mark.parametrize("Bq,Bk,L", [(8, 8, 64), (8, 4, 61), (4, 8, 50)])
def test_skipped_blocks_contribute_exactly_zero(Bq, Bk, L):
    """Output equals masked SDPA with the mask built from the keep bitmap."""
    Hq, Hkv, d = 4, 2, 8
    q, k, v = _rand((Hq, L, d), 13), _rand((Hkv, L, d), 14), _rand((Hkv, L, d), 15)
    sigma = 1 / math.sqrt(d)
    T = _rand((Hq, orc.num_blocks(L, Bq)), 16) * 0.5 + 1.0
    r = orc.prefill(q, k, v, Bq=Bq, Bk=Bk, thresholds=T)
    assert 0 < r["keep"].sum() < r["visible"].sum()
    g = Hq // Hkv
    for h in range(Hq):
        mask = np.zeros((L, L), dtype=bool)
        for rr in range(L):
            for c in range(rr + 1):
                mask[rr, c] = r["keep"][h, rr // Bq, c // Bk]
        ref = _sdpa(q[h:h + 1], k[h // g:h // g + 1], v[h // g:h // g + 1], mask=mask, sigma=sigma)
        assert np.max(np.abs(r["out"][h] - ref[0])) < 1e-12


# ---------------------------------------------------------------------------
# Brute force on tiny inputs
# ---------------------------------------------------------------------------
def _brute_scores(qh, kh, sigma):
    L, d = qh.shape
    return [[sigma * sum(qh[r][t] * kh[c][t] for t in range(d)) for c in range(L)] for r in range(L)]


def _brute_candidates(i, Bq, Bk, L):
    """Key blocks j such that every key of j strictly precedes every row of i
    (the tile lies below the causal diagonal)."""
    rows = [r for r in range(i * Bq, min((i + 1) * Bq, L))]
    out = []
    for j in range((L + Bk - 1) // Bk):
        keys = [c for c in range(j * Bk, min((j + 1) * Bk, L))]
        if rows and keys and all(c < r for r in rows for c in keys) and len(keys) == Bk:
            out.append(j)
    return out


def _brute_block_max(s, i, j, Bq, Bk, L):
    return max(s[r][c] for r in range(i * Bq, min((i + 1) * Bq, L))
               for c in range(j * Bk, min((j + 1) * Bk, L)) if c <= r)


@pytest.mark.parametrize("Bq,Bk,L", [(3, 3, 20), (4, 2, 19), (2, 4, 21), (3, 2, 23)])
def test_threshold_keep_set_brute_force(Bq, Bk, L):
    d = 3
    q, k, v = _rand((1, L, d), 17), _rand((1, L, d), 18), _rand((1, L, d), 19)
    sigma = 0.7
    T = _rand((1, orc.num_blocks(L, Bq)), 20) * 0.3 + 0.6
    r = orc.prefill(q, k, v, Bq=Bq, Bk=Bk, sigma=sigma, thresholds=T)
    s = _brute_scores(q[0], k[0], sigma)
    for i in range((L + Bq - 1) // Bq):
        cands = _brute_candidates(i, Bq, Bk, L)
        for j in range((L + Bk - 1) // Bk):
            vis = any(c <= rr for rr in range(i * Bq, min((i + 1) * Bq, L))
                      for c in range(j * Bk, min((j + 1) * Bk, L)))
            assert r["visible"][0, i, j] == vis
            if not vis:
                continue
            if j in cands:
                assert r["keep"][0, i, j] == (_brute_block_max(s, i, j, Bq, Bk, L) >= T[0, i])
                assert r["candidate"][0, i, j]
            else:
                assert r["keep"][0, i, j] and not r["candidate"][0, i, j]


@pytest.mark.parametrize("Bq,Bk,L,ks", [(4, 4, 40, [1, 2, 3, 5]), (4, 2, 30, [1, 4]), (2, 4, 26, [2])])
def test_calibration_brute_force(Bq, Bk, L, ks):
    Hq, Hkv, d, N = 2, 1, 4, 3
    qs = [_rand((Hq, L, d), 30 + n) for n in range(N)]
    kk = [_rand((Hkv, L, d), 40 + n) for n in range(N)]
    sigma = 0.5
    T = orc.calibrate(qs, kk, Bq=Bq, Bk=Bk, ks=ks, sigma=sigma)
    nq = (L + Bq - 1) // Bq
    for h in range(Hq):
        for i in range(nq):
            for a, kk_ in enumerate(ks):
                vals = []
                for n in range(N):
                    s = _brute_scores(qs[n][h], kk[n][0], sigma)
                    maxima = sorted((_brute_block_max(s, i, j, Bq, Bk, L)
                                     for j in _brute_candidates(i, Bq, Bk, L)), reverse=True)
                    vals.append(maxima[kk_ - 1] if len(maxima) >= kk_ else -math.inf)
                expect = sum(vals) / N
                if expect == -math.inf:
                    assert T[a, h, i] == -math.inf
                else:
                    assert abs(T[a, h, i] - expect) < 1e-12
    if Bq == Bk:  # exactly the first k query blocks lack k candidates
        for a, kk_ in enumerate(ks):
            assert np.all(T[a, :, :kk_] == -math.inf)
            assert np.all(np.isfinite(T[a, :, kk_:]))


# ---------------------------------------------------------------------------
# Independent formulation: streaming online softmax in arbitrary block order
# ("Skipping attention blocks was the easy part", section FlashAttention:
# running max, running sum, rescale by e^{m_old - m_new}).
# ---------------------------------------------------------------------------
def _streaming(qh, kh, vh, i, Bq, Bk, L, sigma, kept_blocks, order_seed):
    rows = np.arange(i * Bq, min((i + 1) * Bq, L))
    blocks = list(kept_blocks)
    np.random.default_rng(order_seed).shuffle(blocks)
    m = np.full(len(rows), -np.inf)
    l = np.zeros(len(rows))
    acc = np.zeros((len(rows), vh.shape[1]))
    for j in blocks:
        cols = np.arange(j * Bk, min((j + 1) * Bk, L))
        s = sigma * qh[rows] @ kh[cols].T
        s = np.where(cols[None, :] <= rows[:, None], s, -np.inf)
        m_new = np.maximum(m, s.max(axis=1))
        ref = np.where(np.isfinite(m_new), m_new, 0.0)  # rows with nothing visible yet
        c = np.exp(m - ref)
        p = np.exp(s - ref[:, None])
        l = l * c + p.sum(axis=1)
        acc = acc * c[:, None] + p @ vh[cols]
        m = m_new
    return acc / l[:, None]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_order_invariance_against_streaming(seed):
    Hq, L, d, Bq, Bk = 2, 52, 8, 8, 4
    q, k, v = _rand((Hq, L, d), 50 + seed), _rand((Hq, L, d), 60 + seed), _rand((Hq, L, d), 70 + seed)
    sigma = 1 / math.sqrt(d)
    T = _rand((Hq, orc.num_blocks(L, Bq)), 80 + seed) * 0.3 + 0.9
    r = orc.prefill(q, k, v, Bq=Bq, Bk=Bk, thresholds=T)
    for h in range(Hq):
        for i in range(orc.num_blocks(L, Bq)):
            kept = [j for j in range(orc.num_blocks(L, Bk)) if r["keep"][h, i, j]]
            for order_seed in range(3):
                o = _streaming(q[h], k[h], v[h], i, Bq, Bk, L, sigma, kept, order_seed)
                assert np.max(np.abs(o - r["out"][h, i * Bq:min((i + 1) * Bq, L)])) < 1e-12


# ---------------------------------------------------------------------------
# Structural equivalences
# ---------------------------------------------------------------------------
def test_last_position_reuse():
    """Query blocks past the calibrated length take the last threshold (Key
    Designs 1): a short table equals the same table padded with copies of its
    last entry, at thresholds that skip some blocks and keep others."""
    Hq, L, d, B = 2, 64, 8, 8
    q, k, v = _rand((Hq, L, d), 90), _rand((Hq, L, d), 91), _rand((Hq, L, d), 92)
    T_short = _rand((Hq, 3), 93) * 0.3 + 2.4  # around the maxima of 8 x 8 N(0, 1) tiles
    T_long = np.concatenate([T_short, np.repeat(T_short[:, -1:], 5, axis=1)], axis=1)
    a = orc.prefill(q, k, v, Bq=B, Bk=B, thresholds=T_short)
    b = orc.prefill(q, k, v, Bq=B, Bk=B, thresholds=T_long)
    late = a["candidate"][:, 3:]
    assert 0 < a["keep"][:, 3:][late].sum() < late.sum()  # reuse decides something
    assert np.array_equal(a["keep"], b["keep"])
    assert np.array_equal(a["out"], b["out"])


def test_last_position_reuse_closed_form():
    """T = [-inf, -inf, +inf] over 8 query blocks: blocks 0 and 1 attend
    densely, every later block (reusing +inf) only to its diagonal block."""
    Hq, L, d, B = 1, 64, 8, 8
    q, k, v = _rand((Hq, L, d), 94), _rand((Hq, L, d), 95), _rand((Hq, L, d), 96)
    sigma = 1 / math.sqrt(d)
    T = np.array([[-np.inf, -np.inf, np.inf]])
    r = orc.prefill(q, k, v, Bq=B, Bk=B, sigma=sigma, thresholds=T)
    mask = np.array([[c <= rr and (rr < 2 * B or c // B == rr // B) for c in range(L)]
                     for rr in range(L)])
    assert np.max(np.abs(r["out"] - _sdpa(q, k, v, mask=mask, sigma=sigma))) < 1e-12


def test_gqa_equals_repeated_kv():
    Hq, Hkv, L, d, B = 4, 2, 40, 8, 8
    q, k, v = _rand((Hq, L, d), 94), _rand((Hkv, L, d), 95), _rand((Hkv, L, d), 96)
    T = _rand((Hq, 5), 97) * 0.3 + 2.4  # around the maxima of 8 x 8 N(0, 1) tiles
    a = orc.prefill(q, k, v, Bq=B, Bk=B, thresholds=T)
    b = orc.prefill(q, _repeat_kv(k, 2), _repeat_kv(v, 2), Bq=B, Bk=B, thresholds=T)
    assert 0 < a["keep"][a["candidate"]].sum() < a["candidate"].sum()
    assert np.array_equal(a["keep"], b["keep"])
    assert np.array_equal(a["out"], b["out"])


def test_thresholds_are_indexed_by_query_head():
    """Under GQA each query head reads its own threshold row and the KV head
    h // (Hq / Hkv): rows alternating -inf / +inf make the even query heads
    dense and the odd ones diagonal-only (library SDPA for both)."""
    Hq, Hkv, L, d, B = 4, 2, 40, 8, 8
    q, k, v = _rand((Hq, L, d), 110), _rand((Hkv, L, d), 111), _rand((Hkv, L, d), 112)
    sigma = 1 / math.sqrt(d)
    T = np.array([[-np.inf], [np.inf], [-np.inf], [np.inf]])
    r = orc.prefill(q, k, v, Bq=B, Bk=B, sigma=sigma, thresholds=T)
    diag = np.array([[c <= rr and c // B == rr // B for c in range(L)] for rr in range(L)])
    for h in range(Hq):
        kh = h // 2
        if h % 2 == 0:
            ref = _sdpa(q[h:h + 1], k[kh:kh + 1], v[kh:kh + 1], causal=True, sigma=sigma)
        else:
            ref = _sdpa(q[h:h + 1], k[kh:kh + 1], v[kh:kh + 1], mask=diag, sigma=sigma)
        assert np.max(np.abs(r["out"][h] - ref[0])) < 1e-12, f"head {h}"


def test_varlen_equals_separate_calls():
    Hq, Hkv, d, B = 2, 1, 8, 8
    lens = [13, 0, 32, 7]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T_ = int(cu[-1])
    q, k, v = _rand((Hq, T_, d), 98), _rand((Hkv, T_, d), 99), _rand((Hkv, T_, d), 100)
    th = _rand((Hq, 4), 101) * 0.2 + 1.0
    r = orc.prefill_varlen(q, k, v, cu, Bq=B, Bk=B, thresholds=th)
    for b in range(len(lens)):
        a, e = cu[b], cu[b + 1]
        if a == e:
            continue
        s = orc.prefill(q[:, a:e], k[:, a:e], v[:, a:e], Bq=B, Bk=B, thresholds=th)
        assert np.array_equal(s["out"], r["out"][:, a:e])
        assert np.array_equal(s["keep"], r["keep"][b])


def test_zero_queries_give_uniform_average():
    """Q = 0 makes every score 0: with T = 0 everything is kept (0 >= 0) and
    row r averages V over keys 0..r; with T = 0.5 only the diagonal region
    survives and row r averages V over its own block's keys up to r."""
    Hq, L, d, B = 1, 24, 4, 8
    q = np.zeros((Hq, L, d))
    k, v = _rand((Hq, L, d), 102), _rand((Hq, L, d), 103)
    r = orc.prefill(q, k, v, Bq=B, Bk=B, thresholds=np.zeros((Hq, 3)))
    for rr in range(L):
        assert np.max(np.abs(r["out"][0, rr] - v[0, :rr + 1].mean(axis=0))) < 1e-12
    r = orc.prefill(q, k, v, Bq=B, Bk=B, thresholds=np.full((Hq, 3), 0.5))
    for rr in range(L):
        a = (rr // B) * B
        assert np.max(np.abs(r["out"][0, rr] - v[0, a:rr + 1].mean(axis=0))) < 1e-12


def test_effective_flops_counts():
    keep = np.array([[[True, False], [True, True]]])
    vis = np.array([[[True, False], [True, True]]])
    assert orc.effective_flops(keep, vis, 2, 2, 3) == 2 * 2 * 2 * 3 * (3 + 3)


# ---------------------------------------------------------------------------
# Mean correction ("FlashPrefill V2" summary: a pruned block J enters the
# numerator as |B_J| e^{sbar_J} vbar_J and the denominator as |B_J| e^{sbar_J})
# ---------------------------------------------------------------------------
def _constant_blocks(Hkv, L, d, B, seed):
    """K and V whose rows are identical inside every B-row block."""
    nb = orc.num_blocks(L, B)
    kb, vb = _rand((Hkv, nb, d), seed), _rand((Hkv, nb, d), seed + 1)
    return np.repeat(kb, B, axis=1)[:, :L], np.repeat(vb, B, axis=1)[:, :L]


@pytest.mark.parametrize("Bq,Bk,L", [(8, 8, 61), (1, 1, 9), (8, 4, 40), (4, 8, 37)])
def test_mean_correction_is_exact_for_constant_blocks(Bq, Bk, L):
    """When every key (and value) of a block equals the block mean, the stand-in
    reproduces the block's exact contribution: the corrected output with every
    candidate skipped equals dense causal attention."""
    Hq, Hkv, d = 2, 1, 5
    q = _rand((Hq, L, d), 70)
    k, v = _constant_blocks(Hkv, L, d, Bk, 71)
    dense = _sdpa(q, _repeat_kv(k, Hq), _repeat_kv(v, Hq), causal=True, sigma=0.5)
    T = np.full((Hq, 1), np.inf)
    r = orc.prefill(q, k, v, Bq=Bq, Bk=Bk, sigma=0.5, thresholds=T, mean_correction=True)
    assert r["keep"][r["candidate"]].sum() == 0  # every candidate skipped
    assert np.abs(r["out"] - dense).max() < 1e-12
    plain = orc.prefill(q, k, v, Bq=Bq, Bk=Bk, sigma=0.5, thresholds=T)
    if r["candidate"].any():
        assert np.abs(plain["out"] - dense).max() > 1e-3  # the stand-ins did the work


@pytest.mark.parametrize("Bq,Bk,L", [(8, 8, 70), (8, 4, 50)])
def test_mean_correction_equals_replicated_mean_keys(Bq, Bk, L):
    """Independent form: each skipped candidate block replaced by |B_J| copies
    of its mean key and value, then plain masked attention (library SDPA)."""
    Hq, Hkv, d, sigma = 1, 1, 6, 0.4
    q, k, v = _rand((Hq, L, d), 80), _rand((Hkv, L, d), 81), _rand((Hkv, L, d), 82)
    rng = np.random.default_rng(83)
    T = rng.uniform(1.8, 2.8, size=(Hq, orc.num_blocks(L, Bq)))
    r = orc.prefill(q, k, v, Bq=Bq, Bk=Bk, sigma=sigma, thresholds=T, mean_correction=True)
    for i in range(orc.num_blocks(L, Bq)):
        r0, r1 = i * Bq, min((i + 1) * Bq, L)
        keys, vals, vis = [], [], []
        for j in range(orc.num_blocks(L, Bk)):
            cls = orc.block_class(i, j, Bq, Bk, L)
            if cls is None:
                continue
            c0, c1 = j * Bk, min((j + 1) * Bk, L)
            if r["keep"][0, i, j]:
                for c in range(c0, c1):
                    keys.append(k[0, c]), vals.append(v[0, c])
                    vis.append([c <= row for row in range(r0, r1)])
            else:
                for _ in range(c1 - c0):
                    keys.append(k[0, c0:c1].mean(axis=0)), vals.append(v[0, c0:c1].mean(axis=0))
                    vis.append([True] * (r1 - r0))
        mask = np.array(vis).T
        ref = _sdpa(q[:, r0:r1], np.array(keys)[None], np.array(vals)[None], mask=mask,
                    sigma=sigma)
        assert np.abs(r["out"][0, r0:r1] - ref[0]).max() < 1e-12, f"query block {i}"
    assert (~r["keep"][r["candidate"]]).sum() > 0  # some blocks were skipped


def test_mean_correction_without_skips_changes_nothing():
    Hq, Hkv, L, d = 2, 2, 90, 4
    q, k, v = _rand((Hq, L, d), 90), _rand((Hkv, L, d), 91), _rand((Hkv, L, d), 92)
    T = np.full((Hq, 1), -np.inf)
    a = orc.prefill(q, k, v, Bq=16, Bk=16, thresholds=T)
    b = orc.prefill(q, k, v, Bq=16, Bk=16, thresholds=T, mean_correction=True)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"])
    lam = orc.prefill(q, k, v, Bq=16, Bk=16, mode="lambda", log_lambda=-np.inf,
                      mean_correction=True)
    assert np.array_equal(lam["out"], a["out"])


# ---------------------------------------------------------------------------
# Whole-head forms used for full-size bitmap comparisons
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("Bq,Bk,L", [(4, 4, 37), (8, 4, 41), (4, 8, 35), (3, 2, 17)])
def test_block_maxima_brute_force(Bq, Bk, L):
    """Every candidate's s_max from explicit loops over its rows and keys
    (dot products one by one); NaN exactly where j is not a candidate."""
    d, sigma = 3, 0.6
    q, k = _rand((L, d), 90 + L), _rand((L, d), 91 + L)
    got = orc.block_maxima(q, k, Bq, Bk, sigma)
    nq, nk = -(-L // Bq), -(-L // Bk)
    assert got.shape == (nq, nk)
    for i in range(nq):
        rows = range(i * Bq, min((i + 1) * Bq, L))
        for j in range(nk):
            keys = range(j * Bk, min((j + 1) * Bk, L))
            if (j + 1) * Bk <= i * Bq:  # every key precedes every row
                best = max(sigma * sum(q[r, t] * k[c, t] for t in range(d))
                           for r in rows for c in keys)
                assert abs(got[i, j] - best) < 1e-12
            else:
                assert np.isnan(got[i, j])


@pytest.mark.parametrize("Bq,Bk,L", [(4, 4, 37), (8, 4, 40), (4, 8, 33)])
def test_whole_head_threshold_gate_equals_per_block_gate(Bq, Bk, L):
    Hq, Hkv, d = 2, 1, 8
    q, k, v = _rand((Hq, L, d), 93), _rand((Hkv, L, d), 94), _rand((Hkv, L, d), 95)
    sigma = 1 / math.sqrt(d)
    T = _rand((Hq, 3), 96) * 0.4 + 0.6  # three entries: reuse past the table's end
    r = orc.prefill(q, k, v, Bq=Bq, Bk=Bk, sigma=sigma, thresholds=T)
    for h in range(Hq):
        got = orc.keep_threshold_all(orc.block_maxima(q[h], k[0], Bq, Bk, sigma), T[h], L, Bq, Bk)
        assert np.array_equal(got, r["keep"][h])
    assert (~r["keep"] & r["candidate"]).any() and (r["keep"] & r["candidate"]).any()


def test_whole_head_gates_on_the_worked_example():
    g = _load("worked_example.json")
    q, k, _ = _worked_inputs(g["candidate_block_maxima"])
    L = q.shape[1]
    smax = orc.block_maxima(q[0], k[0], 1, 1, 1.0)
    T = np.full(L, -np.inf)
    T[L - 1] = g["threshold"]
    keep = orc.keep_threshold_all(smax, T, L, 1, 1)
    cand = g["candidate_block_maxima"]
    assert sorted(cand[j] for j in range(len(cand)) if keep[L - 1, j]) == \
        sorted(g["expected_kept_maxima"])
    assert keep[L - 1, L - 1]
    # a maximum equal to the threshold is kept (">=")
    T[L - 1] = 4.0
    keep = orc.keep_threshold_all(smax, T, L, 1, 1)
    assert sorted(cand[j] for j in range(len(cand)) if keep[L - 1, j]) == [4.0, 5.0]


@pytest.mark.parametrize("case", ["main", "boundary", "two_rows", "positive_log_lambda"])
def test_whole_head_lambda_on_the_hand_traces(case):
    g = _load("lambda_vote_example.json")
    if case == "positive_log_lambda":
        c = g[case]
        keys, ll, Bq = c["keys"], c["log_lambda"], 1
        q = np.ones((len(keys), 1))
        i = len(keys) - 1
        stats, kept = c["expected_statistics"], c["expected_kept"]
    elif case == "two_rows":
        c = g["two_rows"]
        keys, ll, i, Bq = c["keys"], c["log_lambda"], 2, 2
        q = np.array([0.0, 0.0, 0.0, 0.0, 1.0, -1.0]).reshape(-1, 1)
        stats, kept = c["expected_statistics"], c["expected_kept"]
    else:
        keys = g["keys"] if case == "main" else g["boundary_case"]["keys"]
        ll, Bq = g["log_lambda"], 1
        q = np.ones((len(keys), 1))
        i = len(keys) - 1
        stats = (g["expected_statistics"]["values"] if case == "main"
                 else g["boundary_case"]["expected_statistics"])
        kept = g["expected_kept"] if case == "main" else g["boundary_case"]["expected_kept"]
    k = np.array(keys).reshape(-1, 1)
    keep, st = orc.lambda_all(q, k, Bq, 1, 1.0, ll)
    assert [x for x in st[i] if not np.isnan(x)] == [_stat(x) for x in stats]
    assert [j for j in range(len(keys)) if keep[i, j]] == kept


@pytest.mark.parametrize("Bq,Bk,L", [(4, 4, 37), (8, 4, 40), (4, 8, 33)])
def test_whole_head_lambda_equals_per_block_gate(Bq, Bk, L):
    Hq, Hkv, d = 2, 1, 8
    q, k, v = _rand((Hq, L, d), 97), _rand((Hkv, L, d), 98), _rand((Hkv, L, d), 99)
    for j in range(1, orc.num_blocks(L, Bk), 2):
        k[:, j * Bk:(j + 1) * Bk] *= 0.05
    q *= 2.0
    sigma, ll = 1 / math.sqrt(d), -0.4
    r = orc.prefill(q, k, v, Bq=Bq, Bk=Bk, sigma=sigma, mode="lambda", log_lambda=ll)
    for h in range(Hq):
        keep, st = orc.lambda_all(q[h], k[0], Bq, Bk, sigma, ll)
        assert np.array_equal(keep, r["keep"][h])
        for i in range(orc.num_blocks(L, Bq)):
            ref = orc.decision_statistics(q[h], k[0], i, Bq, Bk, sigma, log_lambda=ll)
            assert [j for j, _ in ref] == [j for j in range(st.shape[1]) if not np.isnan(st[i, j])]
            for j, x in ref:
                assert st[i, j] == x or abs(st[i, j] - x) < 1e-12
    assert (~r["keep"] & r["visible"]).any()
