"""Paged K/V: the same gated prefill with K and V read from page pools through
a per-sequence block table (the serving-cache layout of the "FlashPrefill V2"
summary, agihunt.info: the sparse kernel reads K/V through the page table).

Paging changes where keys live, not what is computed, so:
  - every output of a paged call (O, log-sum-exp, kept-block bitmap, block
    counts) equals the contiguous call on the same keys bit for bit;
  - the varlen paged call matches the fp64 oracle on the gathered keys
    (bitmap bit-exact, outputs within the bf16 tolerance).
Pages are placed in a random order in pools whose unused rows (past each
sequence's last key, and whole spare pages) hold NaN: a kernel that let one of
them reach P.V would turn the output rows NaN."""
import math

import numpy as np
import pytest
import torch

from block_sparse_gated_gb300 import workloads as wl
from oracle import bsfa_oracle as orc
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


def _bsfa():
    import block_sparse_gated_gb300 as b
    return b


def _page_pool(seqs, page, kv_layout, seed, spare=3):
    """seqs: list of [Hkv, L_b, d] CPU tensors.  Returns (pool, table): pool
    [pages, page, Hkv, d] ("pthd") or [pages, Hkv, page, d] ("phtd") with
    NaN in every row no sequence owns, and an int32 [B, max pages + 1] block
    table (sequence b's pages in a seeded random order)."""
    Hkv, d, dt = seqs[0].shape[0], seqs[0].shape[2], seqs[0].dtype
    need = [math.ceil(s.shape[1] / page) for s in seqs]
    n_pages = sum(need) + spare
    perm = np.random.default_rng(seed).permutation(n_pages)
    pool = torch.full((n_pages, page, Hkv, d), float("nan"), dtype=dt)
    table = torch.full((len(seqs), max(need, default=0) + 1), n_pages + 5, dtype=torch.int32)
    nxt = 0
    for b, s in enumerate(seqs):
        for j in range(need[b]):
            pg = int(perm[nxt])
            nxt += 1
            table[b, j] = pg
            chunk = s[:, j * page:(j + 1) * page, :]
            pool[pg, :chunk.shape[1]] = chunk.transpose(0, 1)
    if kv_layout == "phtd":
        pool = pool.permute(0, 2, 1, 3).contiguous()
    return pool, table


def _median_T(x_list, Hq, B, sigma, dev):
    T = gu.median_table(None, None, B, B, sigma,
                        seq_slices=[(gu.to64(x.q), gu.to64(x.k)) for x in x_list])
    return torch.from_numpy(T).to(dev)


@pytest.mark.parametrize("mode", ["threshold", "lambda", "none"])
@pytest.mark.parametrize("page,kv_layout", [(128, "pthd"), (256, "phtd"), (384, "pthd")])
def test_paged_batched_equals_contiguous(cuda_device, mode, page, kv_layout):
    Hq, Hkv, L, d, B = 4, 2, 700, 128, 128
    xs = [wl.layer_inputs(Hq, Hkv, L, d, 300 + n, skip_rate=0.4) for n in range(2)]
    q = torch.stack([x.q for x in xs]).to(cuda_device)
    k = torch.stack([x.k for x in xs]).to(cuda_device)
    v = torch.stack([x.v for x in xs]).to(cuda_device)
    kpool, table = _page_pool([x.k for x in xs], page, kv_layout, seed=page)
    vpool, _ = _page_pool([x.v for x in xs], page, kv_layout, seed=page)
    kw = dict(mode=mode, return_bitmap=True, return_lse=True, return_counts=True)
    if mode == "threshold":
        kw["thresholds"] = _median_T(xs, Hq, B, gu.default_sigma(d), cuda_device)
    elif mode == "lambda":
        kw["log_lambda"] = gu.guarded_log_lambda(
            -1.0, B, B, gu.default_sigma(d), [(gu.to64(x.q), gu.to64(x.k)) for x in xs])
    b = _bsfa()
    ref = b.prefill(q, k, v, **kw)
    got = b.prefill(q, kpool.to(cuda_device), vpool.to(cuda_device),
                    block_table=table.to(cuda_device), kv_layout=kv_layout, **kw)
    torch.cuda.synchronize()
    assert b.api.device_error() == 0
    assert not torch.isnan(got["out"].float()).any()
    for key in ("out", "lse", "bitmap", "counts"):
        assert torch.equal(got[key], ref[key]), key


def test_paged_varlen_matches_oracle_and_contiguous(cuda_device):
    Hq, Hkv, d, B, page = 4, 2, 128, 128, 256
    lens = [300, 1000, 129, 1, 512]
    parts = [wl.layer_inputs(Hq, Hkv, Ln, d, 320 + n, skip_rate=0.4) for n, Ln in enumerate(lens)]
    q, cu = wl.pack_varlen([p.q for p in parts])
    k, _ = wl.pack_varlen([p.k for p in parts])
    v, _ = wl.pack_varlen([p.v for p in parts])
    kpool, table = _page_pool([p.k for p in parts], page, "pthd", seed=7)
    vpool, _ = _page_pool([p.v for p in parts], page, "pthd", seed=7)
    q64, k64, v64 = gu.to64(q), gu.to64(k), gu.to64(v)
    sigma = gu.default_sigma(d)
    bounds = list(zip(cu[:-1].tolist(), cu[1:].tolist()))
    T = gu.median_table(None, None, B, B, sigma,
                        seq_slices=[(q64[:, a:e], k64[:, a:e]) for a, e in bounds])
    slices = [(q64[:, a:e], k64[:, a:e], [(h, i) for h in range(Hq)
                                           for i in range(orc.num_blocks(e - a, B))])
              for a, e in bounds]
    T, _, _ = gu.guarded_thresholds(None, None, T, B, B, sigma, seq_slices=slices)
    b = _bsfa()
    common = dict(cu_seqlens=cu.to(cuda_device), max_seqlen=max(lens), mode="threshold",
                  thresholds=torch.from_numpy(T).to(cuda_device), return_bitmap=True,
                  return_lse=True, return_counts=True)
    qd = q.to(cuda_device)
    got = b.prefill(qd, kpool.to(cuda_device), vpool.to(cuda_device),
                    block_table=table.to(cuda_device), **common)
    con = b.prefill(qd, k.to(cuda_device), v.to(cuda_device), **common)
    torch.cuda.synchronize()
    assert b.api.device_error() == 0
    for key in ("out", "lse", "bitmap", "counts"):
        assert torch.equal(got[key], con[key]), key
    ref = orc.prefill_varlen(q64, k64, v64, cu.numpy(), Bq=B, Bk=B, mode="threshold",
                             thresholds=T.astype(np.float64))
    bits, clean = gu.unpack_bitmap(got["bitmap"], Hq, lens, B, B)
    assert clean
    for n in range(len(lens)):
        assert np.array_equal(bits[n], ref["keep"][n]), f"sequence {n}"
    gu.assert_close(gu.to64(got["out"]), ref["out"], "out")
    gu.assert_close(gu.to64(got["lse"]), ref["lse"], "lse", max_abs=gu.LSE_ABS,
                    mean_abs=gu.LSE_ABS)


def test_paged_fp16_and_64_blocks_equal_contiguous(cuda_device):
    """fp16 elements, head_dim 64, 64-row / 64-key semantic blocks."""
    Hq, Hkv, L, d, Bs, page = 2, 2, 450, 64, 64, 128
    x = wl.layer_inputs(Hq, Hkv, L, d, 340, skip_rate=0.4, dtype=torch.float16)
    q, k, v = (t.to(cuda_device)[None] for t in (x.q, x.k, x.v))
    kpool, table = _page_pool([x.k], page, "pthd", seed=3)
    vpool, _ = _page_pool([x.v], page, "pthd", seed=3)
    ll = gu.guarded_log_lambda(-1.0, Bs, Bs, gu.default_sigma(d), [(gu.to64(x.q), gu.to64(x.k))])
    kw = dict(mode="lambda", log_lambda=ll, block_q=Bs, block_k=Bs, return_bitmap=True,
              return_lse=True, return_counts=True)
    b = _bsfa()
    ref = b.prefill(q, k, v, **kw)
    got = b.prefill(q, kpool.to(cuda_device), vpool.to(cuda_device),
                    block_table=table.to(cuda_device), **kw)
    torch.cuda.synchronize()
    assert b.api.device_error() == 0
    for key in ("out", "lse", "bitmap", "counts"):
        assert torch.equal(got[key], ref[key]), key
