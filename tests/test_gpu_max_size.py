"""The longest sequence the library accepts: 16384 query tiles of 128 rows
(2,097,152 tokens) in one call, one head, d = 64.  It exercises the
scheduling pre-pass at its limit, 64-bit row and bitmap indexing and the
widest bitmap rows (512 words).  Half of the key blocks are scaled down (the
skip tier of the lambda-sweep recipe), so a threshold of 1.0 separates the
two tiers by far more than the 1e-3 guard band; the fp64 oracle checks
sampled query blocks, including the last one."""
import math

import numpy as np
import pytest
import torch

from block_sparse_gated_gb300 import workloads as wl
from oracle import bsfa_oracle as orc
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

B = 128
N_TILES = 16384


def test_two_million_token_sequence(cuda_device):
    import block_sparse_gated_gb300 as bsfa
    L, d = N_TILES * B, 64
    x = wl.layer_inputs(1, 1, L, d, 910, device=cuda_device, skip_rate=0.5, block=B)
    T = torch.full((1, 1), 1.0, device=cuda_device)
    r = bsfa.prefill(x.q[None], x.k[None], x.v[None], mode="threshold", thresholds=T,
                     return_bitmap=True, return_lse=True, return_counts=True)
    torch.cuda.synchronize()
    assert bsfa.api.device_error() == 0
    kept, cand, diag = r["counts"].cpu().tolist()
    assert cand == N_TILES * (N_TILES - 1) // 2 and diag == N_TILES
    assert 0.3 < 1 - kept / cand < 0.7
    q64, k64, v64 = gu.to64(x.q[0]), gu.to64(x.k[0]), gu.to64(x.v[0])
    bm = r["bitmap"].cpu().numpy().view(np.uint32)  # [N_TILES, 1, 512]
    assert bm.shape == (N_TILES, 1, N_TILES // 32)
    out, lse = r["out"][0, 0], r["lse"][0]
    sigma = 1.0 / math.sqrt(d)
    for i in (0, 1, 777, 5000, N_TILES - 1):
        ref = orc.query_block(q64, k64, v64, i, Bq=B, Bk=B, sigma=sigma, mode="threshold",
                              T_hi=1.0)
        for j, keep in ref["keep"].items():
            assert bool((int(bm[i, 0, j >> 5]) >> (j & 31)) & 1) == keep, f"bitmap ({i}, {j})"
        assert not np.any(bm[i, 0, (i >> 5) + 1:]), f"bits past the diagonal in row {i}"
        assert (int(bm[i, 0, i >> 5]) >> (i & 31)) >> 1 == 0, f"bits past the diagonal in row {i}"
        r0, r1 = i * B, (i + 1) * B
        gu.assert_close(gu.to64(out[r0:r1]), ref["out"], f"out block {i}")
        gu.assert_close(gu.to64(lse[r0:r1]), ref["lse"], f"lse block {i}", max_abs=gu.LSE_ABS,
                        mean_abs=gu.LSE_ABS)


def test_most_sequences_per_call(cuda_device):
    """The largest accepted batch: 4096 packed sequences (lengths 0-400,
    seeded) of 64-row / 64-key semantic blocks in one varlen call.  Block
    counts are checked against their closed form over every sequence, the
    bitmap rows are clean past each sequence's last key block, and sampled
    sequences (including the first and the last) against the oracle."""
    import block_sparse_gated_gb300 as bsfa
    Hq, Hkv, d, Bs, n_seq = 2, 1, 64, 64, 4096
    lens = np.random.default_rng(920).integers(0, 401, size=n_seq).tolist()
    lens[0], lens[-1], lens[7] = 400, 1, 0
    parts = [wl.layer_inputs(Hq, Hkv, Ln, d, 921 + n, skip_rate=0.5, block=Bs) for n, Ln in
             enumerate(lens)]
    q, cu = wl.pack_varlen([p.q for p in parts])
    k, _ = wl.pack_varlen([p.k for p in parts])
    v, _ = wl.pack_varlen([p.v for p in parts])
    T = torch.full((Hq, 1), 1.0, device=cuda_device)
    r = bsfa.prefill(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                     cu_seqlens=cu.to(cuda_device), max_seqlen=max(lens), block_q=Bs, block_k=Bs,
                     mode="threshold", thresholds=T, return_bitmap=True, return_lse=True,
                     return_counts=True)
    torch.cuda.synchronize()
    assert bsfa.api.device_error() == 0
    nb = [orc.num_blocks(Ln, Bs) for Ln in lens]
    kept, cand, diag = r["counts"].cpu().tolist()
    assert cand == Hq * sum(n * (n - 1) // 2 for n in nb) and diag == Hq * sum(nb)
    assert 0 < kept < cand
    bits, clean = gu.unpack_bitmap(r["bitmap"], Hq, lens, Bs, Bs)
    assert clean
    sigma = 1.0 / math.sqrt(d)
    cu_l = cu.tolist()
    picks = [0, 7, n_seq - 1] + np.random.default_rng(922).choice(n_seq, 13, replace=False).tolist()
    for b in picks:
        a, e = cu_l[b], cu_l[b + 1]
        if e == a:
            continue
        ref = orc.prefill(gu.to64(q[:, a:e]), gu.to64(k[:, a:e]), gu.to64(v[:, a:e]), Bq=Bs,
                          Bk=Bs, sigma=sigma, thresholds=np.full((Hq, 1), 1.0))
        assert np.array_equal(bits[b], ref["keep"]), f"bitmap of sequence {b}"
        gu.assert_close(gu.to64(r["out"][:, a:e]), ref["out"], f"out of sequence {b}")
        gu.assert_close(gu.to64(r["lse"][:, a:e]), ref["lse"], f"lse of sequence {b}",
                        max_abs=gu.LSE_ABS, mean_abs=gu.LSE_ABS)
