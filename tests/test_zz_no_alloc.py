"""bsfa_prefill_fwd_noalloc, the entry point for callers that may not allocate
device memory while attention runs (a fixed up-front memory plan, a plugin
whose host framework owns the allocator).  It takes no workspace; its scratch
is a fixed array inside the library.  Its results must equal
bsfa_prefill_fwd's byte for byte, also on consecutive calls that reuse that
array, whichever of them needs more of it.

This file sorts last so that a run stopping at the first failure has already
run every other test."""
import ctypes

import pytest
import torch

from block_sparse_gated_gb300 import _native, api
from block_sparse_gated_gb300 import workloads as wl
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

BSFA_ERR_UNSUPPORTED = 2


def _params(q, k, v, out, *, mode, thresholds=None, log_lambda=None, bitmap=None):
    p = api._params(q, k, v, out, layout=None, cu_seqlens=None, max_seqlen=None, block_q=128,
                    block_k=128, softmax_scale=None, mode=mode, thresholds=thresholds,
                    log_lambda=log_lambda)
    if bitmap is not None:
        p.kept_bitmap = bitmap.data_ptr()
    return p


def _case(dev, B, Hq, Hkv, L, d, seed, mode):
    xs = [wl.layer_inputs(Hq, Hkv, L, d, seed + n, needles=2, skip_rate=0.3) for n in range(B)]
    q = torch.stack([x.q for x in xs]).to(dev)
    k = torch.stack([x.k for x in xs]).to(dev)
    v = torch.stack([x.v for x in xs]).to(dev)
    kw = {}
    if mode == "threshold":
        T = gu.median_table(gu.to64(xs[0].q), gu.to64(xs[0].k), 128, 128, gu.default_sigma(d))
        kw["thresholds"] = torch.from_numpy(T).to(dev)
    else:
        kw["log_lambda"] = -1.0
    return q, k, v, kw


def test_noalloc_matches_workspace_entry_on_consecutive_calls(cuda_device):
    """Three calls in a row share the fixed scratch: one that needs more of
    it (3 sequences, 18 query tiles), then one that needs less (1 sequence,
    8 tiles) and would read stale schedule entries if the scratch were not
    rewritten, then the first again.  The same kernel on the same schedule
    gives identical bytes, so outputs and bitmaps must be equal, not close."""
    big = _case(cuda_device, 3, 8, 2, 700, 128, 910, "lambda")
    small = _case(cuda_device, 1, 4, 2, 1000, 128, 900, "threshold")
    cases = [(big, "lambda"), (small, "threshold"), (big, "lambda")]
    # Results of the existing entry point (caller-provided workspace).
    ref = []
    for (q, k, v, kw), mode in cases:
        r = api.prefill(q, k, v, mode=mode, return_bitmap=True, **kw)
        ref.append((r["out"], r["bitmap"]))
    torch.cuda.synchronize()
    L = _native.lib()
    got = []
    for ((q, k, v, kw), mode), (ro, rb) in zip(cases, ref):
        out = torch.full_like(q, float("nan"))
        bm = torch.full_like(rb, -1)
        p = _params(q, k, v, out, mode=mode, bitmap=bm, **kw)
        assert L.bsfa_prefill_fwd_noalloc(ctypes.byref(p), api._stream(None)) == 0
        got.append((out, bm))
    torch.cuda.synchronize()
    assert api.device_error() == 0
    for (ro, rb), (go, gb) in zip(ref, got):
        assert torch.equal(go, ro)
        assert torch.equal(gb, rb)


def test_noalloc_rejects_requests_beyond_its_scratch(cuda_device):
    """A request whose schedule would not fit the fixed scratch is refused
    before anything is launched: the output and bitmap keep their sentinels."""
    q, k, v, kw = _case(cuda_device, 1, 4, 2, 256, 128, 920, "lambda")
    out = torch.full_like(q, 7.0)
    bm = torch.full((2, 4, 1), 0x12345678, dtype=torch.int32, device=cuda_device)
    p = _params(q, k, v, out, mode="lambda", bitmap=bm, **kw)
    p.batch, p.seqlen = 1024, 32768  # ~2 MiB of schedule, beyond the 256 KiB scratch
    torch.cuda.synchronize()
    assert _native.lib().bsfa_prefill_fwd_noalloc(ctypes.byref(p), api._stream(None)) == \
        BSFA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert api.device_error() == 0
    assert torch.all(out == 7.0)
    assert torch.all(bm == 0x12345678)
