"""GPU parity at the full workload sizes (the shapes and kernels bench.py
times), checked on sampled (head, query block) units that the fp64 oracle
computes one by one: the first and last query blocks, the block at the
calibrated length, and seeded random ones.

Thresholds for the sampled rows come from the oracle's own calibration on
the same seeded calibration inputs, kept clear of the compared block maxima
by the guard band; every other row gets a constant, so no input of the
oracle comes from the CUDA path.  The GPU calibration is checked against
the oracle on the sampled rows as well."""
import math
import random

import numpy as np
import pytest
import torch

import block_sparse_gated_gb300 as bsfa
from block_sparse_gated_gb300 import workloads as wl
from oracle import bsfa_oracle as orc
from oracle import guard
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


class HostCache:
    """fp64 host copies of single heads, made on first use."""

    def __init__(self, q, k, v, g):
        self.q, self.k, self.v, self.g = q, k, v, g
        self.cq, self.ck, self.cv = {}, {}, {}

    def qh(self, h):
        if h not in self.cq:
            self.cq[h] = gu.to64(self.q[h])
        return self.cq[h]

    def kh(self, h):
        kh = h // self.g
        if kh not in self.ck:
            self.ck[kh] = gu.to64(self.k[kh])
        return self.ck[kh]

    def vh(self, h):
        kh = h // self.g
        if kh not in self.cv:
            self.cv[kh] = gu.to64(self.v[kh])
        return self.cv[kh]


def _sample(n_q, nT, heads, per_head, seed):
    rnd = random.Random(seed)
    out = []
    for h in heads:
        fixed = {0, 1, nT - 1, min(nT, n_q - 1), n_q - 1}
        out += [(h, i) for i in sorted(fixed | set(rnd.sample(range(n_q), per_head)))]
    return out


def _oracle_rows_T(cal, heads_rows, Bq, Bk, ks, sigma, g):
    """Oracle calibration of the table entries (h, t) in heads_rows."""
    res = {}
    for (h, t) in heads_rows:
        vals = np.zeros(len(ks))
        for qn, kn in cal:
            c = orc.candidate_maxima(gu.to64(qn[h]), gu.to64(kn[h // g]), t, Bq, Bk, sigma)
            vals += np.array([orc.kth_largest(c, kk) for kk in ks])
        res[(h, t)] = vals / len(cal)
    return res


def _check_blocks(hc, blocks, Bq, Bk, sigma, L, bitmap_rows, out, lse, mode, T=None,
                  log_lambda=None, mean_correction=False):
    """Compare sampled query blocks of one sequence with the oracle."""
    Hq = out.shape[0]
    worst = 0.0
    nT = T.shape[1] if T is not None else 1
    for h, i in blocks:
        r = orc.query_block(hc.qh(h), hc.kh(h), hc.vh(h), i, Bq=Bq, Bk=Bk, sigma=sigma,
                            mode=mode,
                            T_hi=None if T is None else float(T[h, orc.threshold_index(i, nT)]),
                            log_lambda=log_lambda, mean_correction=mean_correction)
        words = bitmap_rows[i, h].astype(np.uint32)
        for j, kept in r["keep"].items():
            bit = bool((int(words[j >> 5]) >> (j & 31)) & 1)
            assert bit == kept, f"bitmap (h={h}, i={i}, j={j}): gpu {bit} oracle {kept}"
        r0, r1 = i * Bq, min((i + 1) * Bq, L)
        o = gu.to64(out[h, r0:r1])
        mx, mean = gu.compare_outputs(o, r["out"])
        assert mx <= gu.MAX_ABS and mean <= gu.MEAN_ABS, f"out (h={h}, i={i}): {mx:.3e} {mean:.3e}"
        ml, _ = gu.compare_outputs(gu.to64(lse[h, r0:r1]), r["lse"])
        assert ml <= gu.LSE_ABS, f"lse (h={h}, i={i}): {ml:.3e}"
        worst = max(worst, mx)
    return worst


def _threshold_case(dev, name, k_index=0, mean_correction=False):
    cfg = wl.WORKLOADS[name]
    Hq, Hkv, d, Bq, Bk, L = (cfg[x] for x in ("Hq", "Hkv", "d", "Bq", "Bk", "L"))
    g, sigma = Hq // Hkv, 1.0 / math.sqrt(d)
    cal = []
    for n in range(cfg["n_cal"]):
        x = wl.layer_inputs(Hq, Hkv, cfg["cal_L"], d, wl.cal_seed(cfg["index"], n), dev,
                            with_v=False, sink_tokens=cfg["sink_tokens"],
                            needles=cfg["cal_needles"], block=Bk)
        cal.append((x.q, x.k))
    # GPU calibration (the product path) against the oracle on sampled rows.
    T_gpu = bsfa.calibrate([c[0] for c in cal], [c[1] for c in cal], cfg["ks"], block_q=Bq,
                           block_k=Bk).cpu().numpy()
    nT = T_gpu.shape[2]
    x = wl.layer_inputs(Hq, Hkv, L, d, wl.eval_seed(cfg["index"]), dev,
                        sink_tokens=cfg["sink_tokens"], needles=cfg["needles"], block=Bk)
    n_q = orc.num_blocks(L, Bq)
    heads = [0, Hq - 1]
    blocks = _sample(n_q, nT, heads, 4, cfg["index"])
    rows = sorted({(h, orc.threshold_index(i, nT)) for h, i in blocks})
    T_rows = _oracle_rows_T(cal, rows, Bq, Bk, cfg["ks"], sigma, g)
    for (h, t), vals in T_rows.items():
        for a in range(len(cfg["ks"])):
            gv, ov = float(T_gpu[a, h, t]), float(vals[a])
            if math.isinf(ov):
                assert gv == ov, f"calibration (k={cfg['ks'][a]}, h={h}, t={t}) -inf pattern"
            else:
                assert abs(gv - ov) < 1e-4, f"calibration (k={cfg['ks'][a]}, h={h}, t={t})"
    del cal
    # Threshold table for the forward pass: oracle values on sampled rows,
    # a constant elsewhere, then the guard band on the sampled rows.
    fin = [v[k_index] for v in T_rows.values() if math.isfinite(v[k_index])]
    fill = float(np.mean(fin)) if fin else -math.inf  # an all -inf slice stays all -inf
    T = np.full((Hq, nT), fill, dtype=np.float64)
    for (h, t), vals in T_rows.items():
        T[h, t] = vals[k_index]
    hc = HostCache(x.q, x.k, x.v, g)
    comp = {}
    for h, i in blocks:
        c = orc.candidate_maxima(hc.qh(h), hc.kh(h), i, Bq, Bk, sigma)
        comp.setdefault((h, orc.threshold_index(i, nT)), []).extend(c)
    Tg, _, _ = guard.guard_thresholds(T, {kk: np.asarray(vv) for kk, vv in comp.items()})
    r = bsfa.prefill(x.q[None], x.k[None], x.v[None], block_q=Bq, block_k=Bk, mode="threshold",
                     thresholds=torch.from_numpy(Tg).to(dev), return_bitmap=True,
                     return_lse=True, return_counts=True, mean_correction=mean_correction)
    torch.cuda.synchronize()
    assert bsfa.api.device_error() == 0
    bm = r["bitmap"].cpu().numpy().view(np.uint32)
    worst = _check_blocks(hc, blocks, Bq, Bk, sigma, L, bm, r["out"][0],
                          r["lse"].reshape(Hq, L), "threshold", T=Tg.astype(np.float64),
                          mean_correction=mean_correction)
    kc, cand, diag = r["counts"].cpu().tolist()
    return worst, 1 - kc / cand


def test_llama_32k_full_size(cuda_device):
    worst, skip = _threshold_case(cuda_device, "llama8b-L32768")
    assert 0.0 < skip < 1.0


def test_llama_128k_k128_mean_correction_full_size(cuda_device):
    """The bench's k = 128 slice at 128K with mean correction for the skipped
    blocks (about 70% of the candidates get a stand-in)."""
    worst, skip = _threshold_case(cuda_device, "llama8b-L131072", k_index=1, mean_correction=True)
    assert 0.5 < skip < 1.0


@pytest.mark.parametrize("k_index", [0, 1, 2])
def test_llama_128k_full_size(cuda_device, k_index):
    """k = 32 and k = 128 gate; k = 512 has no table entry with 512
    candidates at the 64K calibration length, so every entry is -inf and
    nothing is skipped."""
    worst, skip = _threshold_case(cuda_device, "llama8b-L131072", k_index)
    if k_index == 2:
        assert skip == 0.0
    else:
        assert skip > 0.0


@pytest.mark.parametrize("rate", [0.25, 0.5, 0.75, 0.9])
def test_lambda_sweep_64k_full_size(cuda_device, rate):
    cfg = wl.WORKLOADS["lambda-sweep-L65536"]
    Hq, Hkv, d, B, L = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["Bk"], cfg["L"]
    g, sigma = Hq // Hkv, 1.0 / math.sqrt(d)
    x = wl.layer_inputs(Hq, Hkv, L, d, wl.eval_seed(cfg["index"], 7), cuda_device,
                        skip_rate=rate, block=B)
    hc = HostCache(x.q, x.k, x.v, g)
    n_q = orc.num_blocks(L, B)
    blocks = _sample(n_q, n_q, [3, 20], 3, 17)

    def stats(ll):
        out = []
        for h, i in blocks:
            out += [s for _, s in orc.decision_statistics(hc.qh(h), hc.kh(h), i, B, B, sigma,
                                                          log_lambda=ll)]
        return np.asarray(out)

    ll, _ = guard.guard_log_lambda(cfg["log_lambda"], stats)
    r = bsfa.prefill(x.q[None], x.k[None], x.v[None], mode="lambda", log_lambda=ll,
                     return_bitmap=True, return_lse=True, return_counts=True)
    torch.cuda.synchronize()
    assert bsfa.api.device_error() == 0
    bm = r["bitmap"].cpu().numpy().view(np.uint32)
    _check_blocks(hc, blocks, B, B, sigma, L, bm, r["out"][0], r["lse"].reshape(Hq, L),
                  "lambda", log_lambda=ll)
    kc, cand, _ = r["counts"].cpu().tolist()
    assert abs((1 - kc / cand) - rate) < 0.1


def test_varlen_8seq_full_size(cuda_device):
    cfg = wl.WORKLOADS["varlen-8seq-32layer"]
    Hq, Hkv, d, B = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["Bk"]
    g, sigma = Hq // Hkv, 1.0 / math.sqrt(d)
    lens = cfg["lens"]
    parts = [wl.layer_inputs(Hq, Hkv, Ln, d, wl.eval_seed(cfg["index"], n), cuda_device,
                             sink_tokens=cfg["sink_tokens"],
                             needles=max(1, round(cfg["needles_per_64k"] * Ln / 65536)), block=B)
             for n, Ln in enumerate(lens)]
    q, cu = wl.pack_varlen([p.q for p in parts])
    k, _ = wl.pack_varlen([p.k for p in parts])
    v, _ = wl.pack_varlen([p.v for p in parts])
    del parts
    nT = orc.num_blocks(cfg["cal_L"], B)
    # One layer's table: a constant plus oracle-side guard on the sampled rows.
    T = np.full((Hq, nT), 4.2, dtype=np.float64)
    cu_l = cu.tolist()
    picks = [(b, h, i) for b in (0, 3, 7) for h in (1, 30)
             for i in sorted({0, orc.num_blocks(lens[b], B) - 1,
                              orc.num_blocks(lens[b], B) // 2})]
    caches = {}
    comp = {}
    for b, h, i in picks:
        a, e = cu_l[b], cu_l[b + 1]
        if b not in caches:
            caches[b] = HostCache(q[:, a:e], k[:, a:e], v[:, a:e], g)
        c = orc.candidate_maxima(caches[b].qh(h), caches[b].kh(h), i, B, B, sigma)
        comp.setdefault((h, orc.threshold_index(i, nT)), []).extend(c)
    Tg, _, _ = guard.guard_thresholds(T, {kk: np.asarray(vv) for kk, vv in comp.items()})
    r = bsfa.prefill(q, k, v, cu_seqlens=cu.to(cuda_device), max_seqlen=max(lens),
                     mode="threshold", thresholds=torch.from_numpy(Tg).to(cuda_device),
                     return_bitmap=True, return_lse=True)
    torch.cuda.synchronize()
    assert bsfa.api.device_error() == 0
    bm = r["bitmap"].cpu().numpy().view(np.uint32)
    rowbase = np.concatenate([[0], np.cumsum([orc.num_blocks(Ln, B) for Ln in lens])])
    for b in (0, 3, 7):
        a, e = cu_l[b], cu_l[b + 1]
        blocks = [(h, i) for bb, h, i in picks if bb == b]
        _check_blocks(caches[b], blocks, B, B, sigma, lens[b],
                      bm[rowbase[b]:rowbase[b + 1]], r["out"][:, a:e], r["lse"][:, a:e],
                      "threshold", T=Tg.astype(np.float64))
