"""Guard band for generated test inputs.  TEST INFRASTRUCTURE ONLY.

The kept-block bitmap is compared bit for bit between the fp64 oracle and the
fp32 GPU kernel.  A block maximum that sits within rounding distance of its
threshold could legitimately fall either way, so generated workloads are kept
clear of the decision boundary: any threshold entry (or the single ln(lambda))
that lies within ``band`` of a value it is compared against is moved to the
middle of the nearest gap of width >= ``min_gap`` among those values.  The same
adjusted table is then fed to both sides.  Entries at -inf are never touched
(nothing can tie with them).

The values compared against the thresholds come from the oracle only.
"""
from __future__ import annotations

import math
from typing import Callable, Mapping

import numpy as np

from . import bsfa_oracle as orc


def nearest_clear_value(x: float, values: np.ndarray, band: float = 1e-3,
                        min_gap: float = 2e-3, margin: float = 1e-2) -> float:
    """Return x if no value lies within ``band`` of it, else the midpoint of
    the gap (between consecutive sorted values, or beyond either end) closest
    to x whose width is at least ``min_gap``."""
    vals = np.sort(np.asarray(values, dtype=np.float64))
    vals = vals[np.isfinite(vals)]
    if vals.size == 0 or not np.any(np.abs(vals - x) < band):
        return x
    cands = [vals[0] - margin, vals[-1] + margin]
    gaps = np.diff(vals)
    idx = np.nonzero(gaps >= min_gap)[0]
    cands.extend(((vals[idx] + vals[idx + 1]) * 0.5).tolist())
    cands = np.asarray(cands)
    return float(cands[np.argmin(np.abs(cands - x))])


def guard_thresholds(T: np.ndarray, compared: Mapping[tuple[int, int], np.ndarray],
                     band: float = 1e-3, min_gap: float = 2e-3):
    """T: [Hq, nT] float table (modified copy returned, float32-representable).
    compared: {(h, t): array of block maxima compared against T[h, t]}.
    Returns (T_adjusted, n_adjusted, max_abs_shift)."""
    T = np.array(T, dtype=np.float64, copy=True)
    n_adj, max_shift = 0, 0.0
    for (h, t), vals in compared.items():
        x = T[h, t]
        if not math.isfinite(x):
            continue
        y = nearest_clear_value(x, vals, band, min_gap)
        y = float(np.float32(y))
        if y != x:
            n_adj += 1
            max_shift = max(max_shift, abs(y - x))
            T[h, t] = y
    return T.astype(np.float32), n_adj, max_shift


def compared_maxima(q, k, *, Bq, Bk, sigma, nT, blocks, seq_slices=None):
    """Collect {(h, t): candidate block maxima} for the (h, i) query blocks in
    ``blocks`` of one sequence (q [Hq,L,d], k [Hkv,L,d]), t = min(i, nT-1).
    ``seq_slices`` lets varlen callers pass several sequences: a list of
    (q_seq, k_seq, blocks)."""
    out: dict[tuple[int, int], list] = {}
    items = seq_slices if seq_slices is not None else [(q, k, blocks)]
    for qs, ks_, blks in items:
        qs = np.asarray(qs, dtype=np.float64)
        ks_ = np.asarray(ks_, dtype=np.float64)
        Hq, Hkv = qs.shape[0], ks_.shape[0]
        g = Hq // Hkv
        for h, i in blks:
            c = orc.candidate_maxima(qs[h], ks_[h // g], i, Bq, Bk, sigma)
            out.setdefault((h, orc.threshold_index(i, nT)), []).extend(c)
    return {key: np.asarray(v) for key, v in out.items()}


def guard_log_lambda(log_lambda: float,
                     statistics: Callable[[float], np.ndarray],
                     band: float = 1e-3, min_gap: float = 2e-3,
                     max_iter: int = 8):
    """lambda mode: the decision statistic max_r(rowmax_r - m_r) of every
    candidate depends on earlier decisions, so the statistics are recomputed
    for each trial value.  ``statistics(log_lambda)`` returns them all.
    Returns (log_lambda_adjusted, n_moves); raises if no clear value is found."""
    x = log_lambda
    if not math.isfinite(x):
        return x, 0
    for it in range(max_iter):
        st = statistics(x)
        y = float(np.float32(nearest_clear_value(x, st, band, min_gap)))
        if y == x:
            return x, it
        x = y
    raise RuntimeError("no ln(lambda) clear of the decision statistics")
