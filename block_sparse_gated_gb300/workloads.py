"""Seeded synthetic inputs shaped like the pages' workloads.

This module holds input recipes only -- no attention arithmetic.  The CUDA
path and the oracle both receive the tensors it produces (the oracle after an
exact bf16 -> float64 widening).  It imports nothing else from this package.

Recipe (every tensor is drawn in fp32 with a seeded torch generator on the
requested device, then rounded to bf16 round-to-nearest-even):

* Q, K, V ~ N(0, 1), layout [heads, tokens, head_dim].
* Needle key blocks: for KV head kh, ``needles`` key blocks are drawn without
  replacement from the blocks that are off-diagonal for some query block and
  lie past the sink prefix; their keys become
  ``needle_scale * sqrt(d) * u_kh + K`` with u_kh the unit mean query direction
  of the query heads that read kh.  The scaled score of a needle is then about
  ``needle_scale * (q . u_kh)``, well above the background tile maxima.
* Sink prefix: the first ``sink_tokens`` keys are multiplied by ``sink_scale``
  (large key norms, an attention sink).
* Per-block key scale (lambda sweep): for each KV head, every key block
  j >= 1 independently lands in a "skip tier" with probability ``skip_rate``
  and has its keys multiplied by ``skip_scale``; block 0 keeps scale 1.

The Llama-3.1-8B attention shape (32 query heads, 8 KV heads, d = 128) and the
long-context lengths follow the pages' benchmark settings; the pages' own
datasets (RULER, LongBench, needle-in-a-haystack) are not reproduced -- these
generated tensors stand in for them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

_STREAM_Q, _STREAM_K, _STREAM_V, _STREAM_NEEDLE, _STREAM_SCALE = range(5)


def _gen(seed: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + stream * 7919) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def gaussian(shape, seed: int, stream: int, device="cpu") -> torch.Tensor:
    return torch.randn(shape, generator=_gen(seed, stream, device), device=device,
                       dtype=torch.float32)


@dataclass
class LayerInputs:
    q: torch.Tensor  # bf16 or fp16 [Hq, L, d]
    k: torch.Tensor  # [Hkv, L, d], same type
    v: torch.Tensor | None  # [Hkv, L, d], same type
    needle_blocks: list = field(default_factory=list)  # per KV head
    skip_tier: torch.Tensor | None = None  # bool [Hkv, nk]


def layer_inputs(Hq: int, Hkv: int, L: int, d: int, seed: int, device="cpu", *,
                 with_v: bool = True, sink_tokens: int = 0, sink_scale: float = 4.0,
                 needles: int = 0, needle_scale: float = 4.0, block: int = 128,
                 skip_rate: float = 0.0, skip_scale: float = 0.01,
                 dtype: torch.dtype = torch.bfloat16) -> LayerInputs:
    """One attention layer's Q/K/V for a single sequence of length L, drawn
    in fp32 and rounded once to ``dtype`` (bf16 or fp16)."""
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    q = gaussian((Hq, L, d), seed, _STREAM_Q, device)
    k = gaussian((Hkv, L, d), seed, _STREAM_K, device)
    v = gaussian((Hkv, L, d), seed, _STREAM_V, device) if with_v else None
    nk = (L + block - 1) // block
    g = Hq // Hkv
    needle_blocks = []
    if needles:
        first = (sink_tokens + block - 1) // block
        eligible = torch.arange(first, max(nk - 1, first), device="cpu")
        gen = _gen(seed, _STREAM_NEEDLE, "cpu")
        qmean = q.view(Hkv, g, L, d).mean(dim=(1, 2))
        u = qmean / qmean.norm(dim=-1, keepdim=True)
        for kh in range(Hkv):
            n = min(needles, eligible.numel())
            pick = eligible[torch.randperm(eligible.numel(), generator=gen)[:n]].sort().values
            needle_blocks.append(pick.tolist())
            for j in pick.tolist():
                k[kh, j * block:(j + 1) * block] += needle_scale * math.sqrt(d) * u[kh]
    if sink_tokens:
        k[:, :sink_tokens] *= sink_scale
    skip_tier = None
    if skip_rate > 0.0:
        gen = _gen(seed, _STREAM_SCALE, "cpu")
        uni = torch.rand((Hkv, nk), generator=gen)
        skip_tier = uni < skip_rate
        skip_tier[:, :1] = False  # block 0 keeps scale 1 (no blocks when L = 0)
        scale = torch.where(skip_tier, torch.tensor(skip_scale), torch.tensor(1.0))
        scale_tok = scale.repeat_interleave(block, dim=1)[:, :L].to(device)
        k *= scale_tok[:, :, None]
    return LayerInputs(q.to(dtype), k.to(dtype), v.to(dtype) if v is not None else None,
                       needle_blocks, skip_tier)


def pack_varlen(parts):
    """Concatenate per-sequence [H, L_b, d] tensors along tokens.
    Returns (packed [H, T, d], cu_seqlens int32 [nseq+1] on CPU)."""
    lens = [p.shape[1] for p in parts]
    cu = torch.zeros(len(parts) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    return torch.cat(parts, dim=1), cu


# ---------------------------------------------------------------------------
# The five workloads.  Each is named by what it is; ``index`` keeps the seed
# plan stable (eval seeds 1000 + 10*index + rep, calibration seeds
# 2000 + 10*index + sample, + 100*layer for per-layer tables).
# ---------------------------------------------------------------------------
WORKLOADS = {
    "tiny-h2-d64-L1024": dict(
        index=0, Hq=2, Hkv=2, d=64, L=1024, Bq=64, Bk=64, sink_tokens=0,
        needles=3, ks=[4], n_cal=4, cal_L=1024, cal_needles=3),
    "llama8b-L32768": dict(
        index=1, Hq=32, Hkv=8, d=128, L=32768, Bq=128, Bk=128, sink_tokens=256,
        needles=16, ks=[64], n_cal=4, cal_L=32768, cal_needles=16),
    "llama8b-L131072": dict(
        index=2, Hq=32, Hkv=8, d=128, L=131072, Bq=128, Bk=128, sink_tokens=256,
        needles=64, ks=[32, 128, 512], n_cal=4, cal_L=65536, cal_needles=32),
    "lambda-sweep-L65536": dict(
        index=3, Hq=32, Hkv=8, d=128, L=65536, Bq=128, Bk=128, sink_tokens=0,
        needles=0, skip_rates=[0.0, 0.25, 0.5, 0.75, 0.9], log_lambda=-1.0),
    "varlen-8seq-32layer": dict(
        index=4, Hq=32, Hkv=8, d=128, Bq=128, Bk=128, sink_tokens=256,
        lens=[4096, 8192, 12288, 16384, 24576, 32768, 49152, 65536],
        needles_per_64k=32, ks=[128], n_cal=4, cal_L=65536, cal_needles=32,
        layers=32),
}


def eval_seed(index: int, rep: int = 0) -> int:
    return 1000 + 10 * index + rep


def cal_seed(index: int, sample: int, layer: int = 0) -> int:
    return 2000 + 10 * index + sample + 100 * layer
