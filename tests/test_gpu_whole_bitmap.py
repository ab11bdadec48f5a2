"""Whole kept-block bitmaps at the full workload sizes, bit for bit against
the fp64 oracle: every query block of the compared heads (all 32 heads of the
32K layer and, at one skip rate, of the 64K lambda layer; four heads of the
128K layer for each budget slice, the other lambda rates and every sequence
of the varlen batch).

The oracle's whole-head forms (``block_maxima``, ``keep_threshold_all``,
``lambda_all``) give every candidate's block maximum or lambda statistic.
Threshold tables are built from the oracle alone: one entry per query block
(no reuse past the table's end, so that every row can be guarded on its
own), set to the k-th largest candidate maximum of that row for the slice's
budget k and then moved by the guard band until no compared maximum lies
within 1e-3 of it.  ln(lambda) is guarded against every statistic of the
compared heads.  The same table or ln(lambda) goes to the GPU and to the
oracle; the GPU still computes every head."""
import math

import numpy as np
import pytest
import torch

import block_sparse_gated_gb300 as bsfa
from block_sparse_gated_gb300 import workloads as wl
from oracle import bsfa_oracle as orc
from oracle import guard
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

HEADS4 = (0, 13, 22, 31)  # four query heads on four different KV heads


def _budget_table(smax_rows, Hq, nq, k, fill):
    """smax_rows: {(h, i): candidate maxima compared with T[h, i]}.  Returns
    the guarded table [Hq, nq] (float32): the k-th largest of each compared
    row (-inf when the row has fewer than k), ``fill`` elsewhere."""
    T = np.full((Hq, nq), fill, dtype=np.float64)
    for (h, i), vals in smax_rows.items():
        T[h, i] = orc.kth_largest(list(vals), k)
    Tg, _, _ = guard.guard_thresholds(T, smax_rows)
    return Tg


def _rows_of(smax, h):
    return {(h, i): smax[i][np.isfinite(smax[i])] for i in range(smax.shape[0])}


def _gpu_bits(r, Hq, lens, B):
    bits, clean = gu.unpack_bitmap(r["bitmap"], Hq, lens, B, B)
    assert clean
    return bits


def _layer(dev, name, seed_rep=0, **kw):
    cfg = wl.WORKLOADS[name]
    x = wl.layer_inputs(cfg["Hq"], cfg["Hkv"], cfg["L"], cfg["d"],
                        wl.eval_seed(cfg["index"], seed_rep), dev,
                        sink_tokens=cfg.get("sink_tokens", 0), needles=cfg.get("needles", 0),
                        block=cfg["Bk"], **kw)
    return cfg, x


def _threshold_whole(dev, cfg, x, smax, heads, k, schedule="auto"):
    Hq, Hkv, L, B = cfg["Hq"], cfg["Hkv"], cfg["L"], cfg["Bk"]
    nq = orc.num_blocks(L, B)
    rows = {}
    for h in heads:
        rows.update(_rows_of(smax[h], h))
    fin = [v for kk, v in rows.items() if v.size]
    fill = float(np.median(np.concatenate(fin))) if fin else 0.0
    T = _budget_table(rows, Hq, nq, k, fill)
    r = bsfa.prefill(x.q[None], x.k[None], x.v[None], block_q=B, block_k=B, mode="threshold",
                     thresholds=torch.from_numpy(T).to(dev), return_bitmap=True,
                     return_counts=True, schedule=schedule)
    torch.cuda.synchronize()
    assert bsfa.api.device_error() == 0
    bits = _gpu_bits(r, Hq, [L], B)[0]
    kept = cand = 0
    for h in heads:
        ref = orc.keep_threshold_all(smax[h], T[h].astype(np.float64), L, B, B)
        mism = np.argwhere(bits[h] != ref)
        assert mism.size == 0, f"head {h}: {len(mism)} bitmap mismatches, first {mism[:5].tolist()}"
        c = np.isfinite(smax[h])
        kept += int((ref & c).sum())
        cand += int(c.sum())
    return r, kept, cand


@pytest.fixture(scope="module")
def llama_32k(cuda_device):
    cfg, x = _layer(cuda_device, "llama8b-L32768")
    Hq, g, d, B = cfg["Hq"], cfg["Hq"] // cfg["Hkv"], cfg["d"], cfg["Bk"]
    sigma = 1.0 / math.sqrt(d)
    smax = {h: orc.block_maxima(gu.to64(x.q[h]), gu.to64(x.k[h // g]), B, B, sigma)
            for h in range(Hq)}
    return cfg, x, smax


@pytest.mark.parametrize("schedule", ["auto", "paired"])
def test_llama_32k_whole_bitmap_all_heads(cuda_device, llama_32k, schedule):
    """The 32K layer, every head and query block, budget k = 64 per row, in
    the default (one-head) and the paired schedule."""
    cfg, x, smax = llama_32k
    Hq, B = cfg["Hq"], cfg["Bk"]
    r, kept, cand = _threshold_whole(cuda_device, cfg, x, smax, range(Hq), cfg["ks"][0],
                                     schedule=schedule)
    kc, cc, diag = r["counts"].cpu().tolist()
    assert (kc, cc) == (kept, cand)
    assert diag == Hq * orc.num_blocks(cfg["L"], B)
    assert 0.3 < 1 - kept / cand < 0.95


@pytest.fixture(scope="module")
def llama_128k(cuda_device):
    cfg, x = _layer(cuda_device, "llama8b-L131072")
    g, d, B = cfg["Hq"] // cfg["Hkv"], cfg["d"], cfg["Bk"]
    sigma = 1.0 / math.sqrt(d)
    smax = {h: orc.block_maxima(gu.to64(x.q[h]), gu.to64(x.k[h // g]), B, B, sigma)
            for h in HEADS4}
    return cfg, x, smax


@pytest.mark.parametrize("k", [32, 128, 512])
def test_llama_128k_whole_bitmap(cuda_device, llama_128k, k):
    """The 128K layer, every query block of four heads, at the three budgets
    of the bench's slices (k = 512 leaves the first 512 query blocks at -inf,
    i.e. fully kept)."""
    cfg, x, smax = llama_128k
    _, kept, cand = _threshold_whole(cuda_device, cfg, x, smax, HEADS4, k)
    assert kept < cand


@pytest.mark.parametrize("rate,heads", [(0.5, "all"), (0.25, "four"), (0.75, "four"),
                                        (0.9, "four")])
def test_lambda_64k_whole_bitmap(cuda_device, rate, heads):
    """The lambda sweep layer at 64K: every query block of all 32 heads at
    the 50% rate, of four heads at 25, 75 and 90%."""
    cfg = wl.WORKLOADS["lambda-sweep-L65536"]
    Hq, Hkv, d, B, L = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["Bk"], cfg["L"]
    g, sigma = Hq // Hkv, 1.0 / math.sqrt(d)
    n = cfg["skip_rates"].index(rate)
    x = wl.layer_inputs(Hq, Hkv, L, d, wl.eval_seed(cfg["index"], n), cuda_device,
                        skip_rate=rate, block=B)
    hs = range(Hq) if heads == "all" else HEADS4
    q64 = {h: gu.to64(x.q[h]) for h in hs}
    k64 = {kh: gu.to64(x.k[kh]) for kh in {h // g for h in hs}}
    cache = {}

    def run(ll):
        if ll not in cache:
            cache[ll] = {h: orc.lambda_all(q64[h], k64[h // g], B, B, sigma, ll) for h in hs}
        return cache[ll]

    def stats(ll):
        return np.concatenate([st[np.isfinite(st)] for _, st in run(ll).values()])

    ll, _ = guard.guard_log_lambda(cfg["log_lambda"], stats)
    ref = run(ll)
    r = bsfa.prefill(x.q[None], x.k[None], x.v[None], mode="lambda", log_lambda=ll,
                     return_bitmap=True, return_counts=True)
    torch.cuda.synchronize()
    assert bsfa.api.device_error() == 0
    bits = _gpu_bits(r, Hq, [L], B)[0]
    kept = cand = 0
    for h in hs:
        keep, st = ref[h]
        mism = np.argwhere(bits[h] != keep)
        assert mism.size == 0, f"head {h}: {len(mism)} bitmap mismatches, first {mism[:5].tolist()}"
        c = ~np.isnan(st)
        kept += int((keep & c).sum())
        cand += int(c.sum())
    if heads == "all":
        kc, cc, _ = r["counts"].cpu().tolist()
        assert (kc, cc) == (kept, cand)
    assert abs((1 - kept / cand) - rate) < 0.1


def test_varlen_whole_bitmap(cuda_device):
    """The 8-sequence varlen batch (4K .. 64K packed): every query block of
    every sequence for four heads; each table entry T[h, i] is shared by the
    sequences that have query block i and is guarded against all of their
    maxima."""
    cfg = wl.WORKLOADS["varlen-8seq-32layer"]
    Hq, Hkv, d, B = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["Bk"]
    g, sigma = Hq // Hkv, 1.0 / math.sqrt(d)
    lens = cfg["lens"]
    parts = [wl.layer_inputs(Hq, Hkv, Ln, d, wl.eval_seed(cfg["index"], n), cuda_device,
                             sink_tokens=cfg["sink_tokens"],
                             needles=max(1, round(cfg["needles_per_64k"] * Ln / 65536)), block=B)
             for n, Ln in enumerate(lens)]
    smax = {(b, h): orc.block_maxima(gu.to64(p.q[h]), gu.to64(p.k[h // g]), B, B, sigma)
            for b, p in enumerate(parts) for h in HEADS4}
    q, cu = wl.pack_varlen([p.q for p in parts])
    k, _ = wl.pack_varlen([p.k for p in parts])
    v, _ = wl.pack_varlen([p.v for p in parts])
    del parts
    nq = orc.num_blocks(max(lens), B)
    rows = {}
    for (b, h), sm in smax.items():
        for i in range(sm.shape[0]):
            rows.setdefault((h, i), []).append(sm[i][np.isfinite(sm[i])])
    rows = {key: np.concatenate(v_) for key, v_ in rows.items()}
    T = _budget_table(rows, Hq, nq, cfg["ks"][0], 4.2)
    r = bsfa.prefill(q, k, v, cu_seqlens=cu.to(cuda_device), max_seqlen=max(lens),
                     mode="threshold", thresholds=torch.from_numpy(T).to(cuda_device),
                     return_bitmap=True)
    torch.cuda.synchronize()
    assert bsfa.api.device_error() == 0
    bits = _gpu_bits(r, Hq, lens, B)
    skipped = 0
    for (b, h), sm in smax.items():
        ref = orc.keep_threshold_all(sm, T[h].astype(np.float64), lens[b], B, B)
        mism = np.argwhere(bits[b][h] != ref)
        assert mism.size == 0, f"sequence {b}, head {h}: {len(mism)} mismatches {mism[:5].tolist()}"
        skipped += int((~ref & np.isfinite(sm)).sum())
    assert skipped > 0
