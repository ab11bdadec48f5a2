"""Shared helpers for the GPU parity tests: run the CUDA path through the
C ABI (via the package binding) and the fp64 oracle on the same bf16 inputs,
and compare them."""
from __future__ import annotations

import math

import numpy as np
import torch

from oracle import bsfa_oracle as orc
from oracle import guard

# Output tolerance for bf16 inputs with fp32 accumulation (max-abs, mean-abs).
MAX_ABS = 2e-2
MEAN_ABS = 2e-3
LSE_ABS = 2e-3


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def unpack_bitmap(bm: torch.Tensor, Hq: int, lens, Bq: int, Bk: int):
    """int32 [rows, Hq, words] -> list over sequences of bool [Hq, nq_b, nk_b];
    also returns whether every bit past a row's last key block is zero."""
    words = bm.detach().cpu().numpy().view(np.uint32)
    out, clean, rb = [], True, 0
    for L in lens:
        nq, nk = orc.num_blocks(L, Bq), orc.num_blocks(L, Bk)
        if nq == 0:
            out.append(np.zeros((Hq, 0, 0), dtype=bool))
            continue
        w = words[rb:rb + nq]  # [nq, Hq, W]
        bits = ((w[..., :, None] >> np.arange(32, dtype=np.uint32)) & 1).astype(bool)
        bits = bits.reshape(nq, Hq, -1)
        out.append(np.transpose(bits[:, :, :nk], (1, 0, 2)))
        clean &= not bits[:, :, nk:].any()
        rb += nq
    return out, clean


def compare_outputs(gpu: np.ndarray, ref: np.ndarray, rows_mask=None):
    """Max-abs and mean-abs error over finite reference entries."""
    g, r = np.asarray(gpu, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    m = np.isfinite(r)
    if rows_mask is not None:
        m &= rows_mask
    diff = np.abs(g[m] - r[m])
    return float(diff.max(initial=0.0)), float(diff.mean()) if diff.size else 0.0


def assert_close(gpu, ref, what="out", max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    mx, mean = compare_outputs(gpu, ref)
    assert mx <= max_abs and mean <= mean_abs, f"{what}: max-abs {mx:.3e}, mean-abs {mean:.3e}"
    return mx, mean


def guarded_thresholds(q64, k64, T, Bq, Bk, sigma, blocks=None, seq_slices=None):
    """Move threshold entries away from every block maximum they are compared
    with (oracle maxima), so that fp32 vs fp64 rounding cannot flip a bit."""
    nT = T.shape[1]
    if seq_slices is None:
        Hq = q64.shape[0]
        L = q64.shape[1]
        if blocks is None:
            blocks = [(h, i) for h in range(Hq) for i in range(orc.num_blocks(L, Bq))]
        comp = guard.compared_maxima(q64, k64, Bq=Bq, Bk=Bk, sigma=sigma, nT=nT, blocks=blocks)
    else:
        comp = guard.compared_maxima(None, None, Bq=Bq, Bk=Bk, sigma=sigma, nT=nT, blocks=None,
                                     seq_slices=seq_slices)
    Tg, n_adj, shift = guard.guard_thresholds(T, comp)
    return Tg, n_adj, shift


def median_table(q64, k64, Bq, Bk, sigma, jitter_seed=0, seq_slices=None):
    """A threshold table [Hq, nq] that gates about half the candidates: the
    median of each query block's candidate maxima (from the oracle) plus a
    little seeded jitter; -inf where a block has no candidates."""
    rng = np.random.default_rng(jitter_seed)
    items = seq_slices if seq_slices is not None else [(q64, k64)]
    Hq = items[0][0].shape[0]
    nq = max(orc.num_blocks(qs.shape[1], Bq) for qs, _ in items)
    vals = {}
    for qs, ks in items:
        g = Hq // ks.shape[0]
        for h in range(Hq):
            for i in range(orc.num_blocks(qs.shape[1], Bq)):
                vals.setdefault((h, i), []).extend(
                    orc.candidate_maxima(qs[h], ks[h // g], i, Bq, Bk, sigma))
    T = np.full((Hq, nq), -np.inf, dtype=np.float32)
    for (h, i), v in vals.items():
        if v:
            T[h, i] = np.median(v) + 0.05 * rng.standard_normal()
    return T


def default_sigma(d):
    return 1.0 / math.sqrt(d)


def guarded_log_lambda(log_lambda, Bq, Bk, sigma, seq_slices):
    """ln(lambda) moved clear (>= 1e-3) of every lambda decision statistic
    max_r(rowmax_r - m_r) of every compared query block, computed by the
    oracle; the same value then goes to the GPU and to the oracle.
    seq_slices: [(q64 [Hq,L,d], k64 [Hkv,L,d])] per sequence (empty ones
    allowed)."""

    def stats(ll):
        out = []
        for qs, ks in seq_slices:
            Hq, L = qs.shape[0], qs.shape[1]
            if L == 0:
                continue
            g = Hq // ks.shape[0]
            for h in range(Hq):
                for i in range(orc.num_blocks(L, Bq)):
                    out += [x for _, x in orc.decision_statistics(qs[h], ks[h // g], i, Bq, Bk,
                                                                   sigma, log_lambda=ll)]
        return np.asarray(out)

    ll, _ = guard.guard_log_lambda(log_lambda, stats)
    return ll


def varlen_slices(q64, k64, cu):
    """Per-sequence (q, k) views of packed [H, T, d] arrays."""
    c = [int(x) for x in cu]
    return [(q64[:, a:e], k64[:, a:e]) for a, e in zip(c[:-1], c[1:])]

