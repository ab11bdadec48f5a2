"""Plain fp64 CPU oracle for block-sparse gated causal prefill attention.

TEST INFRASTRUCTURE ONLY.  This module is the independent reference that the
CUDA path is checked against.  Only the test suite, ``__graft_entry__.smoke()``
and the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
it.  It shares no code with the CUDA library and never imports the product
package; the product path never imports it.

What it computes is taken directly from the definitions on the pages, without
any online-softmax streaming, tiling or reordering beyond what the definitions
state:

  scores -> block max -> keep set -> softmax over kept keys -> P.V

Sources (page title, section):

* "Block Sparse Flash Attention" (papernotes.org note on BSFA, arXiv 2512.07011)
  - Key Designs 1, "Offline Threshold Calibration": per sample, layer, head and
    query block take the k-th largest maximum over the visible off-diagonal key
    blocks, average over samples; -inf when fewer than k candidates exist;
    positions past the calibrated length reuse the last calibrated threshold.
  - Key Designs 2, "Exact-Score Gating", displayed equation:
    s_max(i,j) = max over the whole tile of the scaled scores QK^T/sqrt(d);
    keep(i,j) iff s_max(i,j) >= T[l,h,i].  The causal diagonal region is
    always executed with the causal mask applied.
  - Key Designs 3, "Selective Streaming Aggregation": a rejected block adds
    nothing to the numerator or the denominator; the output is attention
    renormalised over the retained blocks.
  - "A Worked Example": maxima 1, 4, 2, 5, 3.5 against T = 3 keep 4, 5, 3.5.
* "FlashPrefill V2: Block-Sparse Prefill Attention for Long-Context LLM
  Serving" (agihunt.info summary), mean correction (optional here): every
  pruned block J enters as a zero-order stand-in built from its mean key and
  mean value, |B_J| e^{sbar_J} vbar_J in the numerator and |B_J| e^{sbar_J} in
  the denominator.
* "Skipping attention blocks was the easy part" (yash-agarwal.org, BLASST in
  an SM100 prefill kernel), section "Vote, then skip": skip a block when its
  local max minus the running max is below ln(lambda) for every row
  (one row that wants the block vetoes the skip); a skipped block leaves the
  running max untouched; the running max used for the vote is exact.

Readings taken where the pages are silent or ambiguous:

* ">=" (not ">") in the threshold test.
* Candidate ("off-diagonal") key block j for query block i: every key of j
  precedes every row of i, i.e. (j+1)*Bk <= i*Bq -- the tile lies strictly
  below the causal diagonal.  A visible block that is not a candidate is in
  the diagonal region (always kept, causal mask applied).  For Bq == Bk this
  is j < i / j == i for every block size, including 1.
* Thresholds are indexed by query head; q-head h reads KV head h // (Hq/Hkv).
* T is looked up at min(i, nT - 1) (last-position reuse).
* lambda mode visits candidate blocks in ascending key order, the diagonal
  region last; the running max m_r starts at -inf, so the first visited
  candidate is always kept.  ln(lambda) is a natural log.
* Rows and keys past the sequence end take no part in anything.
* Mean correction: sbar_J = sigma * q_r . kbar_J for each row r; |B_J| is the
  number of keys of block J (Bk for every candidate); only skipped candidate
  blocks get a stand-in (the diagonal region is always kept); the gate's
  decisions are taken without the stand-ins (the lambda running max sees
  real scores only).

Every function below works on one sequence at a time with layout
q: [Hq, L, d], k/v: [Hkv, L, d], all float64 (bf16 inputs widen exactly).
"""
from __future__ import annotations

import math
from typing import Iterable, Sequence

import numpy as np

NEG_INF = -math.inf
POS_INF = math.inf

CANDIDATE = "candidate"
DIAGONAL = "diagonal"


# ---------------------------------------------------------------------------
# Block geometry ("Exact-Score Gating": the diagonal region vs off-diagonal
# candidates; the page notes that j == i is not a complete mapping once the
# query and key tiles differ, so the general visibility test is used).
# ---------------------------------------------------------------------------
def num_blocks(length: int, block: int) -> int:
    return (length + block - 1) // block


def block_class(i: int, j: int, Bq: int, Bk: int, L: int):
    """Classify key block j as seen from query block i of a length-L sequence.

    Returns CANDIDATE (every key of j strictly precedes every row of i, so the
    tile lies below the causal diagonal), DIAGONAL (some key of j is visible to
    some row of i, but the tile is not a candidate), or None (nothing
    visible)."""
    first_row = i * Bq
    last_row = min((i + 1) * Bq, L) - 1
    first_key = j * Bk
    last_key = min((j + 1) * Bk, L) - 1
    if first_row > last_row or first_key > last_key:
        return None
    if (j + 1) * Bk <= first_row:
        return CANDIDATE
    if first_key <= last_row:
        return DIAGONAL
    return None


def threshold_index(i: int, nT: int) -> int:
    """Last-position reuse past the calibrated length (Key Designs 1)."""
    return min(i, nT - 1)


# ---------------------------------------------------------------------------
# Scores of one query block (Key Designs 2, displayed equation).
# ---------------------------------------------------------------------------
def query_block_scores(q_h: np.ndarray, k_h: np.ndarray, i: int, Bq: int,
                       sigma: float) -> tuple[np.ndarray, np.ndarray]:
    """Scaled scores sigma * Q_i K^T of query block i against every key that
    is causally visible to some row of it, with invisible entries at -inf.

    Returns (s, rows) where s has shape [rows_in_block, last_row + 1]."""
    L = q_h.shape[0]
    r0, r1 = i * Bq, min((i + 1) * Bq, L)
    rows = np.arange(r0, r1)
    s = sigma * (q_h[r0:r1] @ k_h[:r1].T)
    cols = np.arange(r1)
    s = np.where(cols[None, :] <= rows[:, None], s, NEG_INF)
    return s, rows


def tile_max(s: np.ndarray, j: int, Bk: int) -> float:
    """s_max(i,j): the maximum over the whole Bq x Bk tile of visible scores."""
    return float(np.max(s[:, j * Bk:(j + 1) * Bk]))


# ---------------------------------------------------------------------------
# Keep sets.
# ---------------------------------------------------------------------------
def keep_threshold(s: np.ndarray, i: int, Bq: int, Bk: int, L: int,
                   T_hi: float) -> dict[int, bool]:
    """Threshold gate: keep(i,j) iff s_max(i,j) >= T for candidates; the
    diagonal region is always kept ("Exact-Score Gating")."""
    keep = {}
    for j in range(num_blocks(s.shape[1], Bk)):
        cls = block_class(i, j, Bq, Bk, L)
        if cls is None:
            continue
        if cls == DIAGONAL:
            keep[j] = True
        else:
            keep[j] = tile_max(s, j, Bk) >= T_hi
    return keep


def visit_order_ascending(i: int, Bq: int, Bk: int, L: int) -> list[int]:
    """Key blocks in ascending position, diagonal region last."""
    nk = num_blocks(min((i + 1) * Bq, L), Bk)
    cands = [j for j in range(nk) if block_class(i, j, Bq, Bk, L) == CANDIDATE]
    diags = [j for j in range(nk) if block_class(i, j, Bq, Bk, L) == DIAGONAL]
    return cands + diags


def keep_lambda(s: np.ndarray, i: int, Bq: int, Bk: int, L: int,
                log_lambda: float, trace: list | None = None) -> dict[int, bool]:
    """lambda-relative gate ("Vote, then skip").

    Blocks are visited in ascending key position, the diagonal region last
    (``visit_order_ascending``).  Each row r keeps an exact running max m_r over the
    scores of the blocks kept so far, starting at -inf.  A candidate block is
    skipped iff rowmax_r - m_r < ln(lambda) for every row r of the query
    block; one row at or above the bound keeps it.  A kept block raises m_r to
    max(m_r, rowmax_r); a skipped block leaves m_r unchanged.  The diagonal
    region is always kept.

    If ``trace`` is a list, (j, m_before, rowmax, kept) tuples are appended."""
    order = visit_order_ascending(i, Bq, Bk, L)
    m = np.full(s.shape[0], NEG_INF)
    keep = {}
    for j in order:
        cls = block_class(i, j, Bq, Bk, L)
        if cls is None:
            continue
        rowmax = np.max(s[:, j * Bk:(j + 1) * Bk], axis=1)
        if cls == DIAGONAL:
            kept = True
        else:
            with np.errstate(invalid="ignore"):
                stat = rowmax - m  # m == -inf gives +inf: never below the bound
            kept = not bool(np.all(stat < log_lambda))
        if trace is not None:
            trace.append((j, m.copy(), rowmax.copy(), kept))
        keep[j] = kept
        if kept:
            m = np.maximum(m, rowmax)
    return keep


def decision_statistics(q_h, k_h, i, Bq, Bk, sigma, log_lambda=NEG_INF):
    """For lambda mode: the per-candidate statistic max_r(rowmax_r - m_r),
    with m_r the running max as it stands when block j is visited (before
    block j can raise it), under the keep decisions that ``log_lambda``
    produces.  Block j is kept exactly when its statistic is >= ln(lambda).
    Used to keep generated inputs clear of the decision boundary.

    Returns [(j, statistic)] in visiting order, candidates only."""
    s, _ = query_block_scores(q_h, k_h, i, Bq, sigma)
    L = q_h.shape[0]
    trace: list = []
    keep_lambda(s, i, Bq, Bk, L, log_lambda, trace)
    out = []
    for j, m_before, rowmax, kept in trace:
        if block_class(i, j, Bq, Bk, L) != CANDIDATE:
            continue
        with np.errstate(invalid="ignore"):
            out.append((j, float(np.max(rowmax - m_before))))
    return out


# ---------------------------------------------------------------------------
# Whole-head forms of the two gates, for comparing every block of a long
# sequence: the same definitions as above, one query block at a time.
# ---------------------------------------------------------------------------
def _as_torch64(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))


def _key_major_scores(qt, kt, r0, r1, nkeys, sigma):
    """sigma * K[:nkeys] Q[r0:r1]^T in fp64 ([keys, rows]) from torch fp64
    copies of one head's queries and keys: the scores of the query rows
    against the first nkeys keys, with the keys as rows (each key block is
    then one contiguous run of Bk rows).  torch's CPU matmul is the library
    product (multithreaded)."""
    return (kt[:nkeys] @ qt[r0:r1].T) * sigma


def block_maxima(q_h, k_h, Bq, Bk, sigma) -> np.ndarray:
    """s_max(i, j) of every candidate pair of one head ("Exact-Score Gating":
    the maximum over the whole Bq x Bk tile of the scaled scores), as an
    [nq, nk] float64 array with NaN where j is not a candidate of i.

    A candidate's keys all precede every row of its query block, so its tile
    needs no causal mask: for query block i the scores of its rows against
    the keys of its candidates (key blocks 0 .. ncand-1) are one product,
    and each candidate's maximum is taken over its Bk keys and all rows."""
    import torch
    L = q_h.shape[0]
    nq, nk = num_blocks(L, Bq), num_blocks(L, Bk)
    out = np.full((nq, nk), np.nan)
    qt, kt = _as_torch64(q_h), _as_torch64(k_h)
    for i in range(nq):
        r0, r1 = i * Bq, min((i + 1) * Bq, L)
        ncand = (i * Bq) // Bk  # key blocks j with (j + 1) * Bk <= i * Bq
        if ncand == 0:
            continue
        sT = _key_major_scores(qt, kt, r0, r1, ncand * Bk, sigma)
        out[i, :ncand] = torch.amax(sT.reshape(ncand, Bk * (r1 - r0)), dim=1).numpy()
    return out


def keep_threshold_all(smax: np.ndarray, T_h, L: int, Bq: int, Bk: int) -> np.ndarray:
    """Threshold keep matrix [nq, nk] of one head from its block maxima
    (``block_maxima``) and its threshold row T_h (length nT, looked up at
    min(i, nT - 1)): candidates kept iff s_max >= T, the diagonal region
    always kept, invisible blocks False."""
    nq, nk = smax.shape
    keep = np.zeros((nq, nk), dtype=bool)
    for i in range(nq):
        t = float(T_h[threshold_index(i, len(T_h))])
        for j in range(min(nk, num_blocks(min((i + 1) * Bq, L), Bk))):  # j past these: invisible
            cls = block_class(i, j, Bq, Bk, L)
            if cls == CANDIDATE:
                keep[i, j] = smax[i, j] >= t
            elif cls == DIAGONAL:
                keep[i, j] = True
    return keep


def lambda_all(q_h, k_h, Bq, Bk, sigma, log_lambda):
    """lambda gate ("Vote, then skip") over every query block of one head:
    returns (keep [nq, nk] bool, statistic [nq, nk] float64 with NaN off the
    candidates).  Per query block the candidates are visited in ascending
    key order, each row keeping its exact running max over kept blocks
    (from -inf); block j's statistic is max_r(rowmax_r - m_r) before the
    visit, and it is kept iff that is >= ln(lambda).  The diagonal region is
    kept; its scores never reach a decision, since it is visited last."""
    import torch
    L = q_h.shape[0]
    nq, nk = num_blocks(L, Bq), num_blocks(L, Bk)
    keep = np.zeros((nq, nk), dtype=bool)
    stat = np.full((nq, nk), np.nan)
    qt, kt = _as_torch64(q_h), _as_torch64(k_h)
    for i in range(nq):
        r0, r1 = i * Bq, min((i + 1) * Bq, L)
        ncand = (i * Bq) // Bk
        for j in range(ncand, min(nk, num_blocks(r1, Bk))):  # the diagonal region
            if block_class(i, j, Bq, Bk, L) == DIAGONAL:
                keep[i, j] = True
        if ncand == 0:
            continue
        sT = _key_major_scores(qt, kt, r0, r1, ncand * Bk, sigma)
        rowmax = torch.amax(sT.reshape(ncand, Bk, r1 - r0), dim=1).numpy()  # [candidate, row]
        m = np.full(r1 - r0, NEG_INF)
        for j in range(ncand):
            with np.errstate(invalid="ignore"):
                st = float(np.max(rowmax[j] - m))  # +inf while m is -inf
            stat[i, j] = st
            if st >= log_lambda:
                keep[i, j] = True
                m = np.maximum(m, rowmax[j])
    return keep, stat


# ---------------------------------------------------------------------------
# Renormalised attention over the kept keys ("Selective Streaming
# Aggregation": a skipped block is absent from numerator and denominator).
# ---------------------------------------------------------------------------
def attend_kept(s: np.ndarray, v_h: np.ndarray, keep: dict[int, bool],
                Bk: int, stand_in=None) -> tuple[np.ndarray, np.ndarray]:
    """out[r] = sum_{c in K_r} e^{s[r,c] - M_r} v[c] / Z_r and
    lse[r] = M_r + ln Z_r, K_r = visible keys of kept blocks.

    stand_in: optional (logits [rows, n], values [n, d]) of extra terms that
    join the numerator and the denominator (mean correction); a logit that
    already carries ln|B_J| weighs the term |B_J| times."""
    ncols = s.shape[1]
    col_kept = np.zeros(ncols, dtype=bool)
    for j, kept in keep.items():
        if kept:
            col_kept[j * Bk:min((j + 1) * Bk, ncols)] = True
    sk = np.where(col_kept[None, :], s, NEG_INF)
    vals = v_h[:ncols]
    if stand_in is not None and stand_in[0].shape[1] > 0:
        sk = np.concatenate([sk, stand_in[0]], axis=1)
        vals = np.concatenate([vals, stand_in[1]], axis=0)
    M = np.max(sk, axis=1, keepdims=True)
    e = np.exp(sk - M)
    Z = np.sum(e, axis=1, keepdims=True)
    out = (e @ vals) / Z
    lse = (M + np.log(Z))[:, 0]
    return out, lse


def mean_stand_ins(q_rows: np.ndarray, k_h: np.ndarray, v_h: np.ndarray,
                   keep: dict[int, bool], i: int, Bq: int, Bk: int, L: int,
                   sigma: float) -> tuple[np.ndarray, np.ndarray]:
    """Mean correction ("FlashPrefill V2" summary): for every skipped
    candidate block J of query block i, with |B_J| keys, mean key kbar_J and
    mean value vbar_J, the row-r logit sigma * q_r . kbar_J + ln|B_J| and the
    value vbar_J.  Returns (logits [rows, n], values [n, d])."""
    skipped = [j for j, kept in sorted(keep.items())
               if not kept and block_class(i, j, Bq, Bk, L) == CANDIDATE]
    logits = np.zeros((q_rows.shape[0], len(skipped)))
    vbar = np.zeros((len(skipped), v_h.shape[1]))
    for n, j in enumerate(skipped):
        c0, c1 = j * Bk, min((j + 1) * Bk, L)
        kbar = k_h[c0:c1].mean(axis=0)
        vbar[n] = v_h[c0:c1].mean(axis=0)
        logits[:, n] = sigma * (q_rows @ kbar) + math.log(c1 - c0)
    return logits, vbar


# ---------------------------------------------------------------------------
# One query block, one head: the unit everything else loops over.
# ---------------------------------------------------------------------------
def query_block(q_h, k_h, v_h, i, *, Bq, Bk, sigma, mode, T_hi=None,
                log_lambda=None, mean_correction=False):
    """Gated attention for query block i of one head.

    mode: "threshold", "lambda" or "dense" (every visible block kept).
    mean_correction: add the mean stand-in of every skipped candidate block.

    Returns dict(out [rows, d], lse [rows], keep {j: bool}, smax {j: float})."""
    L = q_h.shape[0]
    s, rows = query_block_scores(q_h, k_h, i, Bq, sigma)
    if mode == "threshold":
        keep = keep_threshold(s, i, Bq, Bk, L, T_hi)
    elif mode == "lambda":
        keep = keep_lambda(s, i, Bq, Bk, L, log_lambda)
    elif mode == "dense":
        keep = {j: True for j in range(num_blocks(s.shape[1], Bk))
                if block_class(i, j, Bq, Bk, L) is not None}
    else:
        raise ValueError(mode)
    smax = {j: tile_max(s, j, Bk) for j in keep}
    stand_in = None
    if mean_correction:
        stand_in = mean_stand_ins(q_h[rows], k_h, v_h, keep, i, Bq, Bk, L, sigma)
    out, lse = attend_kept(s, v_h, keep, Bk, stand_in)
    return {"out": out, "lse": lse, "keep": keep, "smax": smax}


def _kv_head(h: int, Hq: int, Hkv: int) -> int:
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return h // (Hq // Hkv)


def prefill(q, k, v, *, Bq, Bk, sigma=None, mode="threshold",
            thresholds=None, log_lambda=None, blocks=None,
            mean_correction=False):
    """Gated causal prefill of one sequence.

    q: [Hq, L, d]; k, v: [Hkv, L, d] (float64 or anything np.float64 takes).
    thresholds: [Hq, nT] (threshold mode).  sigma defaults to 1/sqrt(d).
    blocks: optional iterable of (h, i) to evaluate; others are left NaN.
    mean_correction: add the mean stand-ins of skipped candidate blocks.

    Returns dict(out [Hq, L, d], lse [Hq, L], keep [Hq, nq, nk] bool,
    visible [Hq, nq, nk] bool, candidate [Hq, nq, nk] bool)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    Hq, L, d = q.shape
    Hkv = k.shape[0]
    if sigma is None:
        sigma = 1.0 / math.sqrt(d)
    nq, nk = num_blocks(L, Bq), num_blocks(L, Bk)
    out = np.full((Hq, L, v.shape[2]), np.nan)
    lse = np.full((Hq, L), np.nan)
    keep = np.zeros((Hq, nq, nk), dtype=bool)
    visible = np.zeros((Hq, nq, nk), dtype=bool)
    cand = np.zeros((Hq, nq, nk), dtype=bool)
    todo = blocks if blocks is not None else [(h, i) for h in range(Hq) for i in range(nq)]
    for h, i in todo:
        kh = _kv_head(h, Hq, Hkv)
        T_hi = None
        if mode == "threshold":
            T_hi = float(thresholds[h][threshold_index(i, len(thresholds[h]))])
        res = query_block(q[h], k[kh], v[kh], i, Bq=Bq, Bk=Bk, sigma=sigma,
                          mode=mode, T_hi=T_hi, log_lambda=log_lambda,
                          mean_correction=mean_correction)
        r0, r1 = i * Bq, min((i + 1) * Bq, L)
        out[h, r0:r1] = res["out"]
        lse[h, r0:r1] = res["lse"]
        for j, kept in res["keep"].items():
            visible[h, i, j] = True
            keep[h, i, j] = kept
            cand[h, i, j] = block_class(i, j, Bq, Bk, L) == CANDIDATE
    return {"out": out, "lse": lse, "keep": keep, "visible": visible, "candidate": cand}


def prefill_varlen(q, k, v, cu_seqlens, **kw):
    """Packed varlen form: q [Hq, T, d], k/v [Hkv, T, d], cu_seqlens [nseq+1].
    Sequences are independent; positions are local to each sequence.
    Returns out [Hq, T, d], lse [Hq, T] and per-sequence keep/visible lists."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    Hq, T, _ = q.shape
    out = np.full((Hq, T, v.shape[2]), np.nan)
    lse = np.full((Hq, T), np.nan)
    keeps, visibles, cands = [], [], []
    for b in range(len(cu_seqlens) - 1):
        a, e = int(cu_seqlens[b]), int(cu_seqlens[b + 1])
        if e == a:
            keeps.append(None), visibles.append(None), cands.append(None)
            continue
        r = prefill(q[:, a:e], k[:, a:e], v[:, a:e], **kw)
        out[:, a:e] = r["out"]
        lse[:, a:e] = r["lse"]
        keeps.append(r["keep"]), visibles.append(r["visible"]), cands.append(r["candidate"])
    return {"out": out, "lse": lse, "keep": keeps, "visible": visibles, "candidate": cands}


# ---------------------------------------------------------------------------
# Offline threshold calibration (Key Designs 1).
# ---------------------------------------------------------------------------
def candidate_maxima(q_h, k_h, i, Bq, Bk, sigma) -> list[float]:
    """s_max(i,j) for every candidate (off-diagonal) key block j of query
    block i."""
    L = q_h.shape[0]
    s, _ = query_block_scores(q_h, k_h, i, Bq, sigma)
    return [tile_max(s, j, Bk) for j in range(num_blocks(s.shape[1], Bk))
            if block_class(i, j, Bq, Bk, L) == CANDIDATE]


def kth_largest(values: Sequence[float], k: int) -> float:
    """k-th largest (1-indexed, duplicates counted); -inf when fewer than k
    values exist (early query blocks keep their whole history)."""
    if k < 1:
        raise ValueError("k must be >= 1")
    if len(values) < k:
        return NEG_INF
    return float(sorted(values, reverse=True)[k - 1])


def calibrate(q_samples, k_samples, *, Bq, Bk, ks: Iterable[int], sigma=None,
              rows=None):
    """Threshold tables T[k][h][i] = mean over samples of the k-th largest
    candidate block maximum (Key Designs 1).  Samples share one length L.

    q_samples: list of [Hq, L, d]; k_samples: list of [Hkv, L, d].
    rows: optional iterable of (h, i) to compute; others are NaN.
    Returns float64 array [len(ks), Hq, ceil(L/Bq)]."""
    ks = list(ks)
    N = len(q_samples)
    if N == 0 or N != len(k_samples):
        raise ValueError("need matching non-empty sample lists")
    Hq, L, d = np.asarray(q_samples[0]).shape
    Hkv = np.asarray(k_samples[0]).shape[0]
    if sigma is None:
        sigma = 1.0 / math.sqrt(d)
    nq = num_blocks(L, Bq)
    T = np.full((len(ks), Hq, nq), np.nan)
    todo = rows if rows is not None else [(h, i) for h in range(Hq) for i in range(nq)]
    for h, i in todo:
        kh = _kv_head(h, Hq, Hkv)
        acc = np.zeros(len(ks))
        for n in range(N):
            qn = np.asarray(q_samples[n], dtype=np.float64)
            kn = np.asarray(k_samples[n], dtype=np.float64)
            c = candidate_maxima(qn[h], kn[kh], i, Bq, Bk, sigma)
            acc += np.array([kth_largest(c, kk) for kk in ks])
        T[:, h, i] = acc / N
    return T


# ---------------------------------------------------------------------------
# Accounting used by tests and the CPU baseline.
# ---------------------------------------------------------------------------
def effective_flops(keep, visible, Bq, Bk, d) -> float:
    """QK^T for every visible block plus P.V for every kept block, each
    2*Bq*Bk*d (the per-tile accounting of "Selective Streaming Aggregation")."""
    F = 2.0 * Bq * Bk * d
    return F * (float(np.count_nonzero(visible)) + float(np.count_nonzero(keep)))
