"""The pipelined schedule (one query head per CTA, Q.K^T of the next tiles
issued ahead of the current P.V) against the fp64 oracle, and against the
paired schedule: the same gate decisions bit for bit, outputs within the
bf16 tolerances of the oracle.  Thresholds and ln(lambda) are guarded clear
of every compared value, as in the other parity tests."""
import math

import numpy as np
import pytest
import torch

from block_sparse_gated_gb300 import workloads as wl
from oracle import bsfa_oracle as orc
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

B = 128


def _bsfa():
    import block_sparse_gated_gb300 as b
    return b


def _run(q, k, v, **kw):
    b = _bsfa()
    r = b.prefill(q, k, v, return_bitmap=True, return_lse=True, return_counts=True, **kw)
    torch.cuda.synchronize()
    assert b.api.device_error() == 0
    return r


def _check(r, ref, Hq, lens, max_abs=gu.MAX_ABS, mean_abs=gu.MEAN_ABS):
    bits, clean = gu.unpack_bitmap(r["bitmap"], Hq, lens, B, B)
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
                                              (3, 1, 513, 128, torch.float16)])
def test_pipelined_matches_oracle(cuda_device, mode, Hq, Hkv, L, d, dtype):
    x = wl.layer_inputs(Hq, Hkv, L, d, 500 + L, needles=2, skip_rate=0.4, dtype=dtype)
    q64, k64, v64 = gu.to64(x.q), gu.to64(x.k), gu.to64(x.v)
    sigma = gu.default_sigma(d)
    kw, okw = {}, {}
    if mode == "threshold":
        T = gu.median_table(q64, k64, B, B, sigma, jitter_seed=L)
        T, _, _ = gu.guarded_thresholds(q64, k64, T, B, B, sigma)
        kw = dict(thresholds=torch.from_numpy(T).to(cuda_device))
        okw = dict(thresholds=T.astype(np.float64))
    elif mode == "lambda":
        ll = gu.guarded_log_lambda(-1.0, B, B, sigma, [(q64, k64)])
        kw = okw = dict(log_lambda=ll)
    q, k, v = (t.to(cuda_device)[None] for t in (x.q, x.k, x.v))
    r = _run(q, k, v, mode=mode, schedule="pipelined", **kw)
    ref = orc.prefill(q64, k64, v64, Bq=B, Bk=B, mode={"none": "dense"}.get(mode, mode), **okw)
    tol = dict(max_abs=4e-3, mean_abs=4e-4) if dtype == torch.float16 else {}
    _check(r, ref, Hq, [L], **tol)
    cand = ref["candidate"]
    cnt = r["counts"].cpu().tolist()
    assert cnt[0] == int((ref["keep"] & cand).sum()) and cnt[1] == int(cand.sum())
    if mode != "none":
        assert 0 < cnt[0] < cnt[1]  # the case really gates
        # The paired schedule takes the same decisions.
        rp = _run(q, k, v, mode=mode, schedule="paired", **kw)
        assert torch.equal(rp["bitmap"], r["bitmap"])
        assert torch.equal(rp["counts"], r["counts"])


@pytest.mark.parametrize("mode", ["threshold", "lambda"])
def test_pipelined_varlen_matches_oracle(cuda_device, mode):
    Hq, Hkv, d = 4, 2, 128
    lens = [100, 0, 300, 129, 640, 1]
    parts = [wl.layer_inputs(Hq, Hkv, Ln, d, 520 + n, skip_rate=0.4) if Ln else None
             for n, Ln in enumerate(lens)]
    qs = [p.q if p else torch.empty(Hq, 0, d, dtype=torch.bfloat16) for p in parts]
    ks = [p.k if p else torch.empty(Hkv, 0, d, dtype=torch.bfloat16) for p in parts]
    vs = [p.v if p else torch.empty(Hkv, 0, d, dtype=torch.bfloat16) for p in parts]
    q, cu = wl.pack_varlen(qs)
    k, _ = wl.pack_varlen(ks)
    v, _ = wl.pack_varlen(vs)
    q64, k64, v64 = gu.to64(q), gu.to64(k), gu.to64(v)
    sigma = gu.default_sigma(d)
    slices = gu.varlen_slices(q64, k64, cu.tolist())
    if mode == "threshold":
        bounds = [(a, e) for a, e in zip(cu[:-1].tolist(), cu[1:].tolist()) if e > a]
        T = gu.median_table(None, None, B, B, sigma,
                            seq_slices=[(q64[:, a:e], k64[:, a:e]) for a, e in bounds])
        T, _, _ = gu.guarded_thresholds(
            None, None, T, B, B, sigma,
            seq_slices=[(q64[:, a:e], k64[:, a:e], [(h, i) for h in range(Hq)
                                                    for i in range(orc.num_blocks(e - a, B))])
                        for a, e in bounds])
        kw = dict(thresholds=torch.from_numpy(T).to(cuda_device))
        okw = dict(thresholds=T.astype(np.float64))
    else:
        ll = gu.guarded_log_lambda(-1.0, B, B, sigma, slices)
        kw = okw = dict(log_lambda=ll)
    r = _run(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
             cu_seqlens=cu.to(cuda_device), max_seqlen=max(lens), mode=mode,
             schedule="pipelined", **kw)
    ref = orc.prefill_varlen(q64, k64, v64, cu.numpy(), Bq=B, Bk=B, mode=mode, **okw)
    _check(r, ref, Hq, lens)


def test_pipelined_paged_equals_contiguous(cuda_device):
    """Paged K/V through the block table gives the same bytes as contiguous
    K/V on the pipelined schedule (pages of 256 tokens, seeded order)."""
    Hq, Hkv, L, d, page = 4, 2, 700, 128, 256
    x = wl.layer_inputs(Hq, Hkv, L, d, 540, skip_rate=0.4)
    q, k, v = (t.to(cuda_device)[None] for t in (x.q, x.k, x.v))
    n_pages = math.ceil(L / page)
    perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(9))

    def pool(t):
        pad = n_pages * page - L
        y = torch.nn.functional.pad(t.transpose(0, 1), (0, 0, 0, 0, 0, pad))
        y = y.reshape(n_pages, page, Hkv, d)
        out = torch.empty_like(y)
        out[perm] = y
        return out.to(cuda_device)

    table = perm.to(torch.int32)[None].to(cuda_device)
    ll = gu.guarded_log_lambda(-1.0, B, B, gu.default_sigma(d), [(gu.to64(x.q), gu.to64(x.k))])
    kw = dict(mode="lambda", log_lambda=ll, schedule="pipelined")
    a = _run(q, k, v, **kw)
    b = _run(q, pool(x.k), pool(x.v), block_table=table, **kw)
    for key in ("out", "lse", "bitmap", "counts"):
        assert torch.equal(a[key], b[key]), key


def test_pipelined_v_always_is_bit_identical(cuda_device):
    Hq, Hkv, L, d = 4, 2, 1500, 128
    x = wl.layer_inputs(Hq, Hkv, L, d, 550, skip_rate=0.6)
    q, k, v = (t.to(cuda_device)[None] for t in (x.q, x.k, x.v))
    kw = dict(mode="lambda", log_lambda=-1.0, schedule="pipelined")
    a = _run(q, k, v, **kw)
    b = _run(q, k, v, v_always=True, **kw)
    for key in ("out", "lse", "bitmap"):
        assert torch.equal(a[key], b[key]), key
    kept, cand = a["counts"].cpu().tolist()[:2]
    assert 0 < kept < cand


def test_pipelined_lambda_64k_whole_bitmap(cuda_device):
    """The 64K lambda layer at 50% skip: every query block of four heads."""
    cfg = wl.WORKLOADS["lambda-sweep-L65536"]
    Hq, Hkv, d, L = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["L"]
    g, sigma = Hq // Hkv, 1.0 / math.sqrt(d)
    x = wl.layer_inputs(Hq, Hkv, L, d, wl.eval_seed(cfg["index"], 2), cuda_device,
                        skip_rate=0.5, block=B)
    heads = (1, 10, 19, 28)
    q64 = {h: gu.to64(x.q[h]) for h in heads}
    k64 = {h // g: gu.to64(x.k[h // g]) for h in heads}
    cache = {}

    def run(ll):
        if ll not in cache:
            cache[ll] = {h: orc.lambda_all(q64[h], k64[h // g], B, B, sigma, ll) for h in heads}
        return cache[ll]

    from oracle import guard
    ll, _ = guard.guard_log_lambda(
        cfg["log_lambda"],
        lambda x_: np.concatenate([st[np.isfinite(st)] for _, st in run(x_).values()]))
    r = _run(x.q[None], x.k[None], x.v[None], mode="lambda", log_lambda=ll, schedule="pipelined")
    bits, clean = gu.unpack_bitmap(r["bitmap"], Hq, [L], B, B)
    assert clean
    for h in heads:
        mism = np.argwhere(bits[0][h] != run(ll)[h][0])
        assert mism.size == 0, f"head {h}: {len(mism)} mismatches {mism[:5].tolist()}"
