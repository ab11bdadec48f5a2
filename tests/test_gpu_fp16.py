"""GPU parity for fp16 inputs: the CUDA path (through the C ABI) against the
fp64 oracle on identical seeded fp16 inputs.

The gate compares fp32 scores, so the kept-block bitmaps are held to the same
bar as bf16: bit-exact with thresholds and ln(lambda) guarded 1e-3 clear of
every compared value.  The output bar is tighter than bf16's.  With fp32
accumulation the error of O comes from rounding P before the PV product and
rounding O once at the end; fp16 rounds with unit roundoff 2^-11 where bf16
has 2^-8, so each of those terms is 8x smaller.  The bar below is the bf16 one
(max-abs 2e-2, mean-abs 2e-3) divided by 5, which keeps a margin under that
factor.  The log-sum-exp is formed from fp32 scores alone and keeps 2e-3."""
import numpy as np
import pytest
import torch

from block_sparse_gated_gb300 import workloads as wl
from oracle import bsfa_oracle as orc
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

F16 = torch.float16
MAX_ABS = 4e-3
MEAN_ABS = 4e-4


def _bsfa():
    import block_sparse_gated_gb300 as b
    return b


def _inputs(Hq, Hkv, L, d, seed, dev, **kw):
    x = wl.layer_inputs(Hq, Hkv, L, d, seed, device="cpu", dtype=F16, **kw)
    assert x.q.dtype == F16
    return x, x.q.to(dev), x.k.to(dev), x.v.to(dev)


def _run(q, k, v, **kw):
    b = _bsfa()
    r = b.prefill(q[None], k[None], v[None], return_bitmap=True, return_lse=True, **kw)
    torch.cuda.synchronize()
    assert b.api.device_error() == 0
    assert r["out"].dtype == F16
    return r


def _check(r, ref, Hq, L, Bq, Bk):
    bits, clean = gu.unpack_bitmap(r["bitmap"], Hq, [L], Bq, Bk)
    assert clean
    mism = np.argwhere(bits[0] != ref["keep"])
    assert mism.size == 0, f"{len(mism)} bitmap mismatches, first {mism[:5].tolist()}"
    gu.assert_close(gu.to64(r["out"][0]), ref["out"], "out", max_abs=MAX_ABS, mean_abs=MEAN_ABS)
    gu.assert_close(gu.to64(r["lse"]).reshape(Hq, L), ref["lse"], "lse", max_abs=gu.LSE_ABS,
                    mean_abs=gu.LSE_ABS)


@pytest.mark.parametrize("Hq,Hkv,L,d", [(4, 2, 300, 128), (2, 2, 200, 64), (8, 2, 1000, 128),
                                        (3, 1, 257, 64)])
def test_fp16_dense_matches_oracle(cuda_device, Hq, Hkv, L, d):
    x, q, k, v = _inputs(Hq, Hkv, L, d, 111, cuda_device)
    r = _run(q, k, v, mode="none")
    ref = orc.prefill(gu.to64(x.q), gu.to64(x.k), gu.to64(x.v), Bq=128, Bk=128, mode="dense")
    _check(r, ref, Hq, L, 128, 128)


def test_fp16_uses_the_finer_mantissa(cuda_device):
    """The same fp32 draw rounded to fp16 and to bf16: the fp16 output is
    nearer the fp64 attention of the fp32 inputs than the bf16 output, which
    a kernel that treated fp16 bits as bf16 (or rounded P to bf16) misses."""
    Hq, Hkv, L, d = 4, 2, 640, 128
    b = _bsfa()
    x32 = wl.layer_inputs(Hq, Hkv, L, d, 112, dtype=torch.float32)
    ref = orc.prefill(gu.to64(x32.q), gu.to64(x32.k), gu.to64(x32.v), Bq=128, Bk=128,
                      mode="dense")["out"]
    errs = {}
    for dt in (torch.bfloat16, F16):
        q, k, v = (t.to(dt).to(cuda_device)[None] for t in (x32.q, x32.k, x32.v))
        o = b.prefill(q, k, v, mode="none")["out"]
        torch.cuda.synchronize()
        errs[dt] = float(np.abs(gu.to64(o[0]) - ref).mean())
    assert errs[F16] * 4 < errs[torch.bfloat16], errs


@pytest.mark.parametrize("Bq,Bk", [(128, 128), (64, 64), (128, 64)])
@pytest.mark.parametrize("Hq,Hkv,L,d", [(4, 2, 1000, 128), (2, 2, 700, 64)])
def test_fp16_threshold_gate_matches_oracle(cuda_device, Bq, Bk, Hq, Hkv, L, d):
    x, q, k, v = _inputs(Hq, Hkv, L, d, 121, cuda_device, needles=2, block=max(Bq, Bk))
    q64, k64, v64 = gu.to64(x.q), gu.to64(x.k), gu.to64(x.v)
    sigma = gu.default_sigma(d)
    table = gu.median_table(q64, k64, Bq, Bk, sigma)
    T, _, _ = gu.guarded_thresholds(q64, k64, table, Bq, Bk, sigma)
    r = _run(q, k, v, block_q=Bq, block_k=Bk, mode="threshold",
             thresholds=torch.from_numpy(T).to(cuda_device))
    ref = orc.prefill(q64, k64, v64, Bq=Bq, Bk=Bk, thresholds=T.astype(np.float64))
    _check(r, ref, Hq, L, Bq, Bk)
    cand = ref["candidate"]
    assert 0 < (ref["keep"] & cand).sum() < cand.sum()  # the case really gates


@pytest.mark.parametrize("Bq,Bk", [(128, 128), (64, 64)])
def test_fp16_lambda_gate_matches_oracle(cuda_device, Bq, Bk):
    Hq, Hkv, L, d = 4, 2, 1500, 128
    x, q, k, v = _inputs(Hq, Hkv, L, d, 131, cuda_device, skip_rate=0.5, block=Bk)
    q64, k64, v64 = gu.to64(x.q), gu.to64(x.k), gu.to64(x.v)
    sigma = gu.default_sigma(d)
    ll = gu.guarded_log_lambda(-1.0, Bq, Bk, sigma, [(q64, k64)])
    r = _run(q, k, v, block_q=Bq, block_k=Bk, mode="lambda", log_lambda=ll)
    ref = orc.prefill(q64, k64, v64, Bq=Bq, Bk=Bk, mode="lambda", log_lambda=ll)
    _check(r, ref, Hq, L, Bq, Bk)
    assert (~ref["keep"] & ref["visible"]).any()


def test_fp16_varlen_lambda_matches_oracle(cuda_device):
    Hq, Hkv, d, B = 4, 2, 128, 128
    lens = [100, 0, 300, 129, 640, 1]
    parts = [wl.layer_inputs(Hq, Hkv, Ln, d, 140 + n, skip_rate=0.4, dtype=F16) if Ln else None
             for n, Ln in enumerate(lens)]
    q, cu = wl.pack_varlen([p.q if p else torch.empty(Hq, 0, d, dtype=F16) for p in parts])
    k, _ = wl.pack_varlen([p.k if p else torch.empty(Hkv, 0, d, dtype=F16) for p in parts])
    v, _ = wl.pack_varlen([p.v if p else torch.empty(Hkv, 0, d, dtype=F16) for p in parts])
    b = _bsfa()
    dev = cuda_device
    ll = gu.guarded_log_lambda(-1.0, B, B, gu.default_sigma(d),
                               gu.varlen_slices(gu.to64(q), gu.to64(k), cu.tolist()))
    r = b.prefill(q.to(dev), k.to(dev), v.to(dev), cu_seqlens=cu.to(dev), max_seqlen=max(lens),
                  mode="lambda", log_lambda=ll, return_bitmap=True, return_lse=True)
    torch.cuda.synchronize()
    assert b.api.device_error() == 0
    ref = orc.prefill_varlen(gu.to64(q), gu.to64(k), gu.to64(v), cu.numpy(), Bq=B, Bk=B,
                             mode="lambda", log_lambda=ll)
    bits, clean = gu.unpack_bitmap(r["bitmap"], Hq, lens, B, B)
    assert clean
    for n, Ln in enumerate(lens):
        if Ln:
            assert np.array_equal(bits[n], ref["keep"][n]), f"sequence {n}"
    gu.assert_close(gu.to64(r["out"]), ref["out"], "out", max_abs=MAX_ABS, mean_abs=MEAN_ABS)
    gu.assert_close(gu.to64(r["lse"]), ref["lse"], "lse", max_abs=gu.LSE_ABS, mean_abs=gu.LSE_ABS)


@pytest.mark.parametrize("Bq,Bk,d", [(128, 128, 128), (64, 64, 64)])
def test_fp16_calibrate_matches_oracle(cuda_device, Bq, Bk, d):
    Hq, Hkv, L, N, ks = 4, 2, 1100, 3, [1, 3, 8]
    sam = [wl.layer_inputs(Hq, Hkv, L, d, 170 + n, with_v=False, needles=2, block=Bk, dtype=F16)
           for n in range(N)]
    b = _bsfa()
    T = b.calibrate([s.q.to(cuda_device) for s in sam], [s.k.to(cuda_device) for s in sam], ks,
                    block_q=Bq, block_k=Bk)
    torch.cuda.synchronize()
    assert b.api.device_error() == 0
    ref = orc.calibrate([gu.to64(s.q) for s in sam], [gu.to64(s.k) for s in sam], Bq=Bq, Bk=Bk,
                        ks=ks)
    got = T.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    fin = np.isfinite(ref)
    assert np.max(np.abs(got[fin] - ref[fin])) < 1e-4
