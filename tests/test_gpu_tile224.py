"""The 128 x 224 tile ("Block Sparse Flash Attention", "Loss & Training":
the H100 port's 128-row query tile and 224-key tile, recalibrated) against
the fp64 oracle: the gate's bitmap bit for bit (thresholds and ln(lambda)
guarded clear of every compared value), outputs and log-sum-exp within the
bf16 tolerances, and the calibration of that tile within 1e-4.  With
unequal tiles the diagonal region of a query block can hold two key blocks
(Key Designs 2: j = i is not a complete mapping); the oracle's general
block geometry decides which."""
import math

import numpy as np
import pytest
import torch

from block_sparse_gated_gb300 import workloads as wl
from oracle import bsfa_oracle as orc
from oracle import guard
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

BQ, BK = 128, 224


def _bsfa():
    import block_sparse_gated_gb300 as b
    return b


def _run(q, k, v, **kw):
    b = _bsfa()
    r = b.prefill(q, k, v, block_q=BQ, block_k=BK, return_bitmap=True, return_lse=True,
                  return_counts=True, **kw)
    torch.cuda.synchronize()
    assert b.api.device_error() == 0
    return r


def _check(r, ref, Hq, lens, max_abs=gu.MAX_ABS, mean_abs=gu.MEAN_ABS):
    bits, clean = gu.unpack_bitmap(r["bitmap"], Hq, lens, BQ, BK)
    assert clean
    keeps = ref["keep"] if isinstance(ref["keep"], list) else [ref["keep"]]
    for n, Ln in enumerate(lens):
        if Ln:
            mism = np.argwhere(bits[n] != keeps[n])
            assert mism.size == 0, f"sequence {n}: {len(mism)} mismatches {mism[:5].tolist()}"
    out = gu.to64(r["out"][0] if r["out"].dim() == 4 else r["out"])
    gu.assert_close(out, ref["out"], "out", max_abs=max_abs, mean_abs=mean_abs)
    lse = gu.to64(r["lse"]).reshape(ref["lse"].shape)
    gu.assert_close(lse, ref["lse"], "lse", max_abs=gu.LSE_ABS, mean_abs=gu.LSE_ABS)


@pytest.mark.parametrize("mode", ["none", "threshold", "lambda"])
@pytest.mark.parametrize("Hq,Hkv,L,d,dtype", [(4, 2, 1000, 128, torch.bfloat16),
                                              (2, 2, 700, 64, torch.bfloat16),
                                              (3, 1, 900, 128, torch.float16),
                                              (2, 1, 224, 128, torch.bfloat16)])
def test_tile224_matches_oracle(cuda_device, mode, Hq, Hkv, L, d, dtype):
    x = wl.layer_inputs(Hq, Hkv, L, d, 600 + L, needles=2, skip_rate=0.4, block=BK, dtype=dtype)
    q64, k64, v64 = gu.to64(x.q), gu.to64(x.k), gu.to64(x.v)
    sigma = gu.default_sigma(d)
    kw, okw = {}, {}
    if mode == "threshold":
        T = gu.median_table(q64, k64, BQ, BK, sigma, jitter_seed=L)
        T, _, _ = gu.guarded_thresholds(q64, k64, T, BQ, BK, sigma)
        kw = dict(thresholds=torch.from_numpy(T).to(cuda_device))
        okw = dict(thresholds=T.astype(np.float64))
    elif mode == "lambda":
        ll = gu.guarded_log_lambda(-1.0, BQ, BK, sigma, [(q64, k64)])
        kw = okw = dict(log_lambda=ll)
    q, k, v = (t.to(cuda_device)[None] for t in (x.q, x.k, x.v))
    r = _run(q, k, v, mode=mode, **kw)
    ref = orc.prefill(q64, k64, v64, Bq=BQ, Bk=BK, mode={"none": "dense"}.get(mode, mode), **okw)
    tol = dict(max_abs=4e-3, mean_abs=4e-4) if dtype == torch.float16 else {}
    _check(r, ref, Hq, [L], **tol)
    cand = ref["candidate"]
    cnt = r["counts"].cpu().tolist()
    assert cnt[0] == int((ref["keep"] & cand).sum())
    assert cnt[1] == int(cand.sum())
    assert cnt[2] == int((ref["visible"] & ~cand).sum())
    if mode == "threshold" and L > 2 * BK:
        assert 0 < cnt[0] < cnt[1]  # the case really gates (lambda: see the V-always case)


def test_tile224_diagonal_region_has_two_blocks():
    """A geometry fact the kernel relies on: with 128-row query blocks and
    224-key blocks, some query blocks see two key blocks that are visible
    but not candidates, and some see one (oracle geometry)."""
    L = 2000
    counts = set()
    for i in range(orc.num_blocks(L, BQ)):
        counts.add(sum(orc.block_class(i, j, BQ, BK, L) == orc.DIAGONAL
                       for j in range(orc.num_blocks(L, BK))))
    assert counts == {1, 2}


@pytest.mark.parametrize("mode", ["threshold", "lambda"])
def test_tile224_varlen_matches_oracle(cuda_device, mode):
    Hq, Hkv, d = 4, 2, 128
    lens = [100, 0, 500, 224, 900, 1]
    parts = [wl.layer_inputs(Hq, Hkv, Ln, d, 620 + n, skip_rate=0.4, block=BK) if Ln else None
             for n, Ln in enumerate(lens)]
    q, cu = wl.pack_varlen([p.q if p else torch.empty(Hq, 0, d, dtype=torch.bfloat16)
                            for p in parts])
    k, _ = wl.pack_varlen([p.k if p else torch.empty(Hkv, 0, d, dtype=torch.bfloat16)
                           for p in parts])
    v, _ = wl.pack_varlen([p.v if p else torch.empty(Hkv, 0, d, dtype=torch.bfloat16)
                           for p in parts])
    q64, k64, v64 = gu.to64(q), gu.to64(k), gu.to64(v)
    sigma = gu.default_sigma(d)
    bounds = [(a, e) for a, e in zip(cu[:-1].tolist(), cu[1:].tolist()) if e > a]
    if mode == "threshold":
        T = gu.median_table(None, None, BQ, BK, sigma,
                            seq_slices=[(q64[:, a:e], k64[:, a:e]) for a, e in bounds])
        T, _, _ = gu.guarded_thresholds(
            None, None, T, BQ, BK, sigma,
            seq_slices=[(q64[:, a:e], k64[:, a:e], [(h, i) for h in range(Hq)
                                                    for i in range(orc.num_blocks(e - a, BQ))])
                        for a, e in bounds])
        kw = dict(thresholds=torch.from_numpy(T).to(cuda_device))
        okw = dict(thresholds=T.astype(np.float64))
    else:
        ll = gu.guarded_log_lambda(-1.0, BQ, BK, sigma, gu.varlen_slices(q64, k64, cu.tolist()))
        kw = okw = dict(log_lambda=ll)
    r = _run(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
             cu_seqlens=cu.to(cuda_device), max_seqlen=max(lens), mode=mode, **kw)
    ref = orc.prefill_varlen(q64, k64, v64, cu.numpy(), Bq=BQ, Bk=BK, mode=mode, **okw)
    _check(r, ref, Hq, lens)


@pytest.mark.parametrize("d,Hq,Hkv", [(128, 4, 2), (64, 2, 2)])
def test_tile224_calibrate_matches_oracle(cuda_device, d, Hq, Hkv):
    L, N, ks = 1500, 3, [1, 2, 4]
    sam = [wl.layer_inputs(Hq, Hkv, L, d, 640 + n, with_v=False, needles=2, block=BK)
           for n in range(N)]
    b = _bsfa()
    T = b.calibrate([s.q.to(cuda_device) for s in sam], [s.k.to(cuda_device) for s in sam], ks,
                    block_q=BQ, block_k=BK)
    torch.cuda.synchronize()
    assert b.api.device_error() == 0
    ref = orc.calibrate([gu.to64(s.q) for s in sam], [gu.to64(s.k) for s in sam], Bq=BQ, Bk=BK,
                        ks=ks)
    got = T.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    fin = np.isfinite(ref)
    assert fin.any() and np.max(np.abs(got[fin] - ref[fin])) < 1e-4


def test_tile224_v_always_is_bit_identical(cuda_device):
    Hq, Hkv, L, d = 4, 2, 1500, 128
    x = wl.layer_inputs(Hq, Hkv, L, d, 660, skip_rate=0.6, block=BK)
    q, k, v = (t.to(cuda_device)[None] for t in (x.q, x.k, x.v))
    a = _run(q, k, v, mode="lambda", log_lambda=-1.0)
    b = _run(q, k, v, mode="lambda", log_lambda=-1.0, v_always=True)
    for key in ("out", "lse", "bitmap"):
        assert torch.equal(a[key], b[key]), key
    kept, cand = a["counts"].cpu().tolist()[:2]
    assert 0 < kept < cand


def test_tile224_32k_whole_bitmap(cuda_device):
    """The 32K layer shape at 128 x 224: every query block of four heads, a
    per-row budget table (the k-th largest candidate maximum of each row,
    k = 32) guarded against its own row."""
    cfg = wl.WORKLOADS["llama8b-L32768"]
    Hq, Hkv, d, L = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["L"]
    g, sigma = Hq // Hkv, 1.0 / math.sqrt(d)
    x = wl.layer_inputs(Hq, Hkv, L, d, wl.eval_seed(cfg["index"]), cuda_device,
                        sink_tokens=cfg["sink_tokens"], needles=cfg["needles"], block=BK)
    heads = (2, 11, 20, 29)
    smax = {h: orc.block_maxima(gu.to64(x.q[h]), gu.to64(x.k[h // g]), BQ, BK, sigma)
            for h in heads}
    nq = orc.num_blocks(L, BQ)
    rows = {(h, i): smax[h][i][np.isfinite(smax[h][i])] for h in heads for i in range(nq)}
    T = np.full((Hq, nq), float(np.median(np.concatenate([v_ for v_ in rows.values()
                                                           if v_.size]))))
    for (h, i), vals in rows.items():
        T[h, i] = orc.kth_largest(list(vals), 32)
    T, _, _ = guard.guard_thresholds(T, rows)
    r = _run(x.q[None], x.k[None], x.v[None], mode="threshold",
             thresholds=torch.from_numpy(T).to(cuda_device))
    bits, clean = gu.unpack_bitmap(r["bitmap"], Hq, [L], BQ, BK)
    assert clean
    skipped = 0
    for h in heads:
        ref = orc.keep_threshold_all(smax[h], T[h].astype(np.float64), L, BQ, BK)
        mism = np.argwhere(bits[0][h] != ref)
        assert mism.size == 0, f"head {h}: {len(mism)} mismatches {mism[:5].tolist()}"
        skipped += int((~ref & np.isfinite(smax[h])).sum())
    assert skipped > 0
