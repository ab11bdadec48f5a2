"""Mean correction for skipped blocks (the stand-in of the "FlashPrefill V2"
summary, agihunt.info) on the GPU path, against the fp64 oracle with the same
option.  The gate's decisions do not depend on it, so the bitmaps are still
compared bit for bit; outputs and log-sum-exp use the bf16 tolerances.  Both
kernels run it: the paired kernel and the one-head (pipelined) kernel, each
with its own correction tiles."""
import math

import numpy as np
import pytest
import torch

from block_sparse_gated_gb300 import workloads as wl
from oracle import bsfa_oracle as orc
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

B = 128
SCHEDULES = ["paired", "pipelined"]


def _bsfa():
    import block_sparse_gated_gb300 as b
    return b


def _run(q, k, v, **kw):
    b = _bsfa()
    r = b.prefill(q, k, v, return_bitmap=True, return_lse=True, return_counts=True, **kw)
    torch.cuda.synchronize()
    assert b.api.device_error() == 0
    return r


@pytest.mark.parametrize("schedule", SCHEDULES)
@pytest.mark.parametrize("Hq,Hkv,L,d", [(4, 2, 1000, 128), (2, 1, 777, 64), (1, 1, 640, 128)])
def test_corrected_threshold_gate_matches_oracle(cuda_device, Hq, Hkv, L, d, schedule):
    x = wl.layer_inputs(Hq, Hkv, L, d, 400 + L, skip_rate=0.4)
    q64, k64, v64 = gu.to64(x.q), gu.to64(x.k), gu.to64(x.v)
    sigma = gu.default_sigma(d)
    T = gu.median_table(q64, k64, B, B, sigma, jitter_seed=L)
    T, _, _ = gu.guarded_thresholds(q64, k64, T, B, B, sigma)
    r = _run(x.q.to(cuda_device)[None], x.k.to(cuda_device)[None], x.v.to(cuda_device)[None],
             mode="threshold", thresholds=torch.from_numpy(T).to(cuda_device),
             mean_correction=True, schedule=schedule)
    ref = orc.prefill(q64, k64, v64, Bq=B, Bk=B, thresholds=T.astype(np.float64),
                      mean_correction=True)
    bits, clean = gu.unpack_bitmap(r["bitmap"], Hq, [L], B, B)
    assert clean and np.array_equal(bits[0], ref["keep"])
    assert (~ref["keep"][ref["candidate"]]).sum() > 0  # some blocks were skipped
    gu.assert_close(gu.to64(r["out"][0]), ref["out"], "out")
    gu.assert_close(gu.to64(r["lse"]).reshape(Hq, L), ref["lse"], "lse", max_abs=gu.LSE_ABS,
                    mean_abs=gu.LSE_ABS)


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_corrected_lambda_gate_varlen_matches_oracle(cuda_device, schedule):
    Hq, Hkv, d = 4, 2, 128
    lens = [300, 1000, 129, 0, 513]
    parts = [wl.layer_inputs(Hq, Hkv, Ln, d, 420 + n, skip_rate=0.5) if Ln else None
             for n, Ln in enumerate(lens)]
    qs = [p.q if p else torch.empty(Hq, 0, d, dtype=torch.bfloat16) for p in parts]
    ks = [p.k if p else torch.empty(Hkv, 0, d, dtype=torch.bfloat16) for p in parts]
    vs = [p.v if p else torch.empty(Hkv, 0, d, dtype=torch.bfloat16) for p in parts]
    q, cu = wl.pack_varlen(qs)
    k, _ = wl.pack_varlen(ks)
    v, _ = wl.pack_varlen(vs)
    ll = gu.guarded_log_lambda(-1.0, B, B, gu.default_sigma(d),
                               gu.varlen_slices(gu.to64(q), gu.to64(k), cu.tolist()))
    r = _bsfa().prefill(q.to(cuda_device), k.to(cuda_device), v.to(cuda_device),
                        cu_seqlens=cu.to(cuda_device), max_seqlen=max(lens), mode="lambda",
                        log_lambda=ll, mean_correction=True, return_bitmap=True,
                        return_lse=True, schedule=schedule)
    torch.cuda.synchronize()
    assert _bsfa().api.device_error() == 0
    ref = orc.prefill_varlen(gu.to64(q), gu.to64(k), gu.to64(v), cu.numpy(), Bq=B, Bk=B,
                             mode="lambda", log_lambda=ll, mean_correction=True)
    bits, clean = gu.unpack_bitmap(r["bitmap"], Hq, lens, B, B)
    assert clean
    for n, Ln in enumerate(lens):
        if Ln:
            assert np.array_equal(bits[n], ref["keep"][n]), f"sequence {n}"
    gu.assert_close(gu.to64(r["out"]), ref["out"], "out")
    gu.assert_close(gu.to64(r["lse"]), ref["lse"], "lse", max_abs=gu.LSE_ABS, mean_abs=gu.LSE_ABS)


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_constant_blocks_make_the_correction_exact(cuda_device, schedule):
    """K and V constant inside every 128-key block: with every candidate
    skipped (T = +inf), the corrected output equals dense attention."""
    Hq, Hkv, L, d = 2, 1, 900, 128
    g = torch.Generator().manual_seed(430)
    nb = math.ceil(L / B)
    kb = torch.randn(Hkv, nb, d, generator=g) * 0.5
    vb = torch.randn(Hkv, nb, d, generator=g)
    k = kb.repeat_interleave(B, dim=1)[:, :L].to(torch.bfloat16)
    v = vb.repeat_interleave(B, dim=1)[:, :L].to(torch.bfloat16)
    q = torch.randn(Hq, L, d, generator=g).to(torch.bfloat16)
    qd, kd, vd = (t.to(cuda_device)[None] for t in (q, k, v))
    T = torch.full((Hq, 1), math.inf, device=cuda_device)
    corr = _run(qd, kd, vd, mode="threshold", thresholds=T, mean_correction=True,
                schedule=schedule)
    dense = _run(qd, kd, vd, mode="none")
    plain = _run(qd, kd, vd, mode="threshold", thresholds=T)
    assert int(corr["counts"][0]) == 0  # every candidate skipped
    gu.assert_close(gu.to64(corr["out"][0]), gu.to64(dense["out"][0]), "corrected vs dense")
    err_plain = np.abs(gu.to64(plain["out"][0]) - gu.to64(dense["out"][0])).max()
    assert err_plain > 0.05  # without the stand-ins the outputs differ


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_correction_without_skips_changes_nothing(cuda_device, schedule):
    """Nothing skipped: every correction tile is skipped too, and the output
    is the same bytes as without the option, in the same kernel."""
    Hq, Hkv, L, d = 4, 2, 700, 128
    x = wl.layer_inputs(Hq, Hkv, L, d, 440)
    q, k, v = (t.to(cuda_device)[None] for t in (x.q, x.k, x.v))
    T = torch.full((Hq, 1), -math.inf, device=cuda_device)
    a = _run(q, k, v, mode="threshold", thresholds=T, schedule=schedule)
    b = _run(q, k, v, mode="threshold", thresholds=T, mean_correction=True, schedule=schedule)
    for key in ("out", "lse", "bitmap", "counts"):
        assert torch.equal(a[key], b[key]), key


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_fp16_corrected_matches_oracle(cuda_device, schedule):
    Hq, Hkv, L, d = 2, 2, 600, 64
    x = wl.layer_inputs(Hq, Hkv, L, d, 450, skip_rate=0.5, dtype=torch.float16)
    q64, k64, v64 = gu.to64(x.q), gu.to64(x.k), gu.to64(x.v)
    ll = gu.guarded_log_lambda(-1.0, B, B, gu.default_sigma(d), [(q64, k64)])
    r = _run(x.q.to(cuda_device)[None], x.k.to(cuda_device)[None], x.v.to(cuda_device)[None],
             mode="lambda", log_lambda=ll, mean_correction=True, schedule=schedule)
    ref = orc.prefill(q64, k64, v64, Bq=B, Bk=B, mode="lambda", log_lambda=ll,
                      mean_correction=True)
    bits, _ = gu.unpack_bitmap(r["bitmap"], Hq, [L], B, B)
    assert np.array_equal(bits[0], ref["keep"])
    gu.assert_close(gu.to64(r["out"][0]), ref["out"], "out", max_abs=4e-3, mean_abs=4e-4)


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_correction_spans_several_mean_tiles(cuda_device, schedule):
    """A 16.9K-token layer: query blocks past 128 candidates take two
    correction tiles, and the kept bits of a row fill several 32-block words.
    About 70% of each compared row's candidates are skipped; the oracle
    evaluates the sampled query blocks of both heads (the GPU computes all)."""
    Hq, Hkv, d = 2, 1, 128
    L = 131 * B + 77
    x = wl.layer_inputs(Hq, Hkv, L, d, 470, skip_rate=0.5)
    q64, k64, v64 = gu.to64(x.q), gu.to64(x.k), gu.to64(x.v)
    sigma = gu.default_sigma(d)
    nq = orc.num_blocks(L, B)
    sampled = [0, 1, 31, 32, 33, 64, 100, 127, 128, 129, nq - 1]
    blocks = [(h, i) for h in range(Hq) for i in sampled]
    rng = np.random.default_rng(470)
    T = np.zeros((Hq, nq), dtype=np.float32)  # rows not compared: any table entry
    for h, i in blocks:
        m = orc.candidate_maxima(q64[h], k64[h // (Hq // Hkv)], i, B, B, sigma)
        T[h, i] = np.quantile(m, 0.7) + 0.05 * rng.standard_normal() if m else -np.inf
    T, _, _ = gu.guarded_thresholds(q64, k64, T, B, B, sigma, blocks=blocks)
    r = _run(x.q.to(cuda_device)[None], x.k.to(cuda_device)[None], x.v.to(cuda_device)[None],
             mode="threshold", thresholds=torch.from_numpy(T).to(cuda_device),
             mean_correction=True, schedule=schedule)
    ref = orc.prefill(q64, k64, v64, Bq=B, Bk=B, thresholds=T.astype(np.float64),
                      blocks=blocks, mean_correction=True)
    bits, clean = gu.unpack_bitmap(r["bitmap"], Hq, [L], B, B)
    assert clean
    for h, i in blocks:
        assert np.array_equal(bits[0][h, i], ref["keep"][h, i]), (h, i)
    skipped = sum(int((~ref["keep"][h, i] & ref["candidate"][h, i]).sum()) for h, i in blocks)
    assert skipped > 800
    gu.assert_close(gu.to64(r["out"][0]), ref["out"], "out")
    gu.assert_close(gu.to64(r["lse"]).reshape(Hq, L), ref["lse"], "lse", max_abs=gu.LSE_ABS,
                    mean_abs=gu.LSE_ABS)


def test_block_mean_pass_head_limit(cuda_device):
    """The block-mean pass takes one thread per (KV head, element): d * Hkv <=
    1024.  16 KV heads run at d = 64 (against the oracle) and are refused with
    BSFA_ERR_UNSUPPORTED at d = 128, leaving the device clean."""
    b = _bsfa()
    Hq = Hkv = 16
    L = 300
    T = torch.full((Hq, 1), 0.5, device=cuda_device)
    x = wl.layer_inputs(Hq, Hkv, L, 64, 460, skip_rate=0.5)
    r = _run(x.q.to(cuda_device)[None], x.k.to(cuda_device)[None], x.v.to(cuda_device)[None],
             mode="threshold", thresholds=T, mean_correction=True)
    ref = orc.prefill(gu.to64(x.q), gu.to64(x.k), gu.to64(x.v), Bq=B, Bk=B,
                      thresholds=np.full((Hq, 1), 0.5), mean_correction=True)
    bits, _ = gu.unpack_bitmap(r["bitmap"], Hq, [L], B, B)
    assert np.array_equal(bits[0], ref["keep"])
    gu.assert_close(gu.to64(r["out"][0]), ref["out"], "out")
    x = wl.layer_inputs(Hq, Hkv, L, 128, 461, skip_rate=0.5)
    with pytest.raises(b.BsfaError) as e:
        b.prefill(x.q.to(cuda_device)[None], x.k.to(cuda_device)[None],
                  x.v.to(cuda_device)[None], mode="threshold", thresholds=T,
                  mean_correction=True)
    assert e.value.status == 2
    torch.cuda.synchronize()
    assert b.api.device_error() == 0


def test_refused_call_writes_nothing(cuda_device):
    """A call refused for the block-mean pass's head limit (d * Hkv > 1024)
    returns BSFA_ERR_UNSUPPORTED before anything is launched: the caller's
    block counters, bitmap, output, LSE and workspace, filled with sentinels,
    come back untouched.  Called through the C ABI directly."""
    import ctypes

    from block_sparse_gated_gb300 import _native, api
    Hq = Hkv = 16
    L, d = 300, 128
    x = wl.layer_inputs(Hq, Hkv, L, d, 462, skip_rate=0.5)
    q, k, v = (t.to(cuda_device)[None] for t in (x.q, x.k, x.v))
    T = torch.full((Hq, 1), 0.5, device=cuda_device)
    sent = 0x5A5A5A5A5A5A5A5A
    counts = torch.full((3,), sent, dtype=torch.int64, device=cuda_device)
    o = torch.full_like(q, 7.0)
    bm = torch.full((3, Hq, 1), 0x12345678, dtype=torch.int32, device=cuda_device)
    lse = torch.full((Hq, L), 3.0, dtype=torch.float32, device=cuda_device)
    ws = torch.full((1 << 20,), 0xA5, dtype=torch.uint8, device=cuda_device)
    p = api._params(q, k, v, o, layout=None, cu_seqlens=None, max_seqlen=None, block_q=B,
                    block_k=B, softmax_scale=None, mode="threshold", thresholds=T,
                    log_lambda=None, mean_correction=True)
    p.block_counts, p.kept_bitmap, p.lse = counts.data_ptr(), bm.data_ptr(), lse.data_ptr()
    p.workspace, p.workspace_bytes = ws.data_ptr(), ws.numel()
    torch.cuda.synchronize()
    status = _native.lib().bsfa_prefill_fwd(ctypes.byref(p), api._stream(None, cuda_device))
    torch.cuda.synchronize()
    assert status == 2
    assert _bsfa().api.device_error() == 0
    assert torch.all(counts == sent)
    assert torch.all(o == 7.0)
    assert torch.all(bm == 0x12345678)
    assert torch.all(lse == 3.0)
    assert torch.all(ws == 0xA5)
