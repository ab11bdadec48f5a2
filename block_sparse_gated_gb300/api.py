"""torch-facing wrappers over the C ABI: argument marshalling only.

Every step of the computation runs in libbsfa.so's CUDA kernels; torch
provides device memory and the current stream.
"""
from __future__ import annotations

import ctypes

import torch

from . import _native

GATE_THRESHOLD, GATE_LAMBDA, GATE_NONE = 0, 1, 2
_MODES = {"threshold": GATE_THRESHOLD, "lambda": GATE_LAMBDA, "none": GATE_NONE,
          "dense": GATE_NONE}


class BsfaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        msg = _native.lib().bsfa_status_string(status).decode()
        super().__init__(f"bsfa status {status} ({msg}){': ' + what if what else ''}")
        self.status = status


def _check(status: int, what: str = ""):
    if status != 0:
        raise BsfaError(status, what)


def _stream(stream, device=None):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _on_device(device, **tensors):
    """Every tensor the library dereferences must live on ``device`` (a CUDA
    device): a host pointer reaching a kernel is a fault, not an error code."""
    if device.type != "cuda":
        raise ValueError("q must be a CUDA tensor")
    for name, t in tensors.items():
        if t is not None and t.device != device:
            raise ValueError(f"{name} is on {t.device}, expected {device}")


def _nbytes(t) -> int:
    return t.numel() * t.element_size()


def _user_workspace(workspace, need: int, device):
    """The caller's workspace if it is a contiguous buffer of at least ``need``
    bytes on ``device``, else a fresh byte buffer."""
    if workspace is not None:
        if not workspace.is_contiguous():
            raise ValueError("the workspace must be contiguous")
        _on_device(device, workspace=workspace)
        if _nbytes(workspace) >= need:
            return workspace
    return torch.empty(max(need, 256), dtype=torch.uint8, device=device)


_DTYPES = {torch.bfloat16: _native.DTYPE_BF16, torch.float16: _native.DTYPE_F16}


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise TypeError("expected a bfloat16 or float16 tensor")
    return _DTYPES[t.dtype]


def _strides_bhtd(t: torch.Tensor, layout: str, varlen: bool):
    """Element strides {batch, head, token} of a bf16/fp16 tensor with d contiguous."""
    _dtype_code(t)
    if t.stride(-1) != 1:
        raise ValueError("the head dimension must be contiguous")
    s = t.stride()
    if varlen:
        if t.dim() != 3:
            raise ValueError("varlen tensors are 3-D")
        if layout == "htd":
            return (0, s[0], s[1]), t.shape[0], t.shape[1]
        if layout == "thd":
            return (0, s[1], s[0]), t.shape[1], t.shape[0]
        raise ValueError(layout)
    if t.dim() == 3:  # [H, L, d] single sequence
        return (t.shape[0] * s[0], s[0], s[1]), t.shape[0], t.shape[1]
    if t.dim() != 4:
        raise ValueError("batched tensors are 4-D")
    if layout == "bhld":
        return (s[0], s[1], s[2]), t.shape[1], t.shape[2]
    if layout == "blhd":
        return (s[0], s[2], s[1]), t.shape[2], t.shape[1]
    raise ValueError(layout)


def _pool_strides(t: torch.Tensor, kv_layout: str):
    """Element strides {page, head, token}, heads and page size of a K or V
    page pool: [pages, page_size, Hkv, d] ("pthd") or [pages, Hkv, page_size, d]
    ("phtd"), d contiguous."""
    _dtype_code(t)
    if t.dim() != 4 or t.stride(-1) != 1:
        raise ValueError("page pools are 4-D with the head dimension contiguous")
    s = t.stride()
    if kv_layout == "pthd":
        return (s[0], s[2], s[1]), t.shape[2], t.shape[1]
    if kv_layout == "phtd":
        return (s[0], s[1], s[2]), t.shape[1], t.shape[2]
    raise ValueError(kv_layout)


def _params(q, k, v, o, *, layout, cu_seqlens, max_seqlen, block_q, block_k, softmax_scale,
            mode, thresholds, log_lambda, v_always=False, block_table=None, kv_layout="pthd",
            mean_correction=False, schedule="auto"):
    varlen = cu_seqlens is not None
    if layout is None:
        layout = "htd" if varlen else "bhld"
    qs, Hq, Lq = _strides_bhtd(q, layout, varlen)
    os_, Ho, Lo = _strides_bhtd(o, layout, varlen)
    paged = block_table is not None
    if paged:
        ks, Hkv, page = _pool_strides(k, kv_layout)
        vs, Hv, page_v = _pool_strides(v, kv_layout)
        if page_v != page or v.shape[0] != k.shape[0]:
            raise ValueError("K and V pools disagree")
        if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.stride(1) != 1:
            raise ValueError("block_table must be an int32 [batch, pages_per_sequence] tensor")
        Lk = Lv = Lq
    else:
        ks, Hkv, Lk = _strides_bhtd(k, layout, varlen)
        vs, Hv, Lv = _strides_bhtd(v, layout, varlen)
    if not (Lq == Lk == Lv == Lo) or Hv != Hkv or Ho != Hq:
        raise ValueError("Q/K/V/O shapes disagree")
    if not (q.dtype == k.dtype == v.dtype == o.dtype):
        raise TypeError("Q, K, V and O must share one element type")
    d = q.shape[-1]
    if not (k.shape[-1] == v.shape[-1] == o.shape[-1] == d):
        raise ValueError("Q/K/V/O head dimensions disagree")
    # The library takes the batch size from q: o (and k, v unless they are
    # page pools) must have the same rank and batch extent.
    same_batch = [o] if paged else [k, v, o]
    if any(t.dim() != q.dim() or (q.dim() == 4 and t.shape[0] != q.shape[0])
           for t in same_batch):
        raise ValueError("Q/K/V/O batch shapes disagree")
    if varlen:
        if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or \
                not cu_seqlens.is_contiguous() or cu_seqlens.numel() < 1:
            raise ValueError("cu_seqlens must be a contiguous int32 [batch + 1] tensor")
        if max_seqlen is None:
            raise ValueError("varlen calls need max_seqlen")
    if paged:
        nb = cu_seqlens.numel() - 1 if varlen else (1 if q.dim() == 3 else q.shape[0])
        longest = int(max_seqlen) if varlen else Lq
        if block_table.shape[0] < nb or block_table.shape[1] * page < longest:
            raise ValueError("block_table has fewer rows than sequences or too few pages per row")
    p = _native.FwdParams()
    p.q, p.k, p.v, p.o = q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr()
    p.q_stride[:], p.k_stride[:], p.v_stride[:], p.o_stride[:] = qs, ks, vs, os_
    if varlen:
        p.batch = cu_seqlens.numel() - 1
        p.cu_seqlens = cu_seqlens.data_ptr()
        p.max_seqlen = int(max_seqlen)
    else:
        p.batch = 1 if q.dim() == 3 else q.shape[0]
        p.cu_seqlens = None
        p.max_seqlen = 0
    p.num_heads_q, p.num_heads_kv, p.seqlen, p.head_dim = Hq, Hkv, Lq, d
    p.block_q, p.block_k = block_q, block_k
    p.softmax_scale = float(softmax_scale) if softmax_scale else 0.0
    p.mode = _MODES[mode] if isinstance(mode, str) else int(mode)
    if thresholds is not None:
        if thresholds.dtype != torch.float32 or thresholds.dim() != 2 or \
                not thresholds.is_contiguous() or thresholds.shape[0] != Hq:
            raise ValueError("thresholds must be a contiguous float32 [Hq, nT] tensor")
        p.thresholds, p.thresholds_nq = thresholds.data_ptr(), thresholds.shape[1]
    else:
        p.thresholds, p.thresholds_nq = None, 0
    p.log_lambda = float(log_lambda) if log_lambda is not None else 0.0
    p.dtype = _dtype_code(q)
    schedule = resolve_schedule(schedule, mode=mode, block_q=block_q, block_k=block_k,
                                mean_correction=mean_correction)
    p.flags = (_native.FLAG_V_ALWAYS if v_always else 0) | \
        (_native.FLAG_MEAN_CORRECTION if mean_correction else 0) | \
        (_native.FLAG_PIPELINED if schedule == "pipelined" else 0)
    if paged:
        p.block_table = block_table.data_ptr()
        p.block_table_stride = block_table.stride(0)
        p.page_size = page
        p.num_pages = k.shape[0]
    return p


def resolve_schedule(schedule="auto", *, mode="threshold", block_q=128, block_k=128,
                     mean_correction=False) -> str:
    """The kernel schedule a call runs.  "auto" takes "pipelined" (one query
    head per CTA, Q.K^T issued ahead of P.V by a warp of its own) for gated
    calls with 128 x 128 blocks, with or without mean correction -- it is the
    faster one there once tiles are skipped -- and "paired" (two query heads
    of a GQA group per CTA sharing every K/V tile) for everything else."""
    del mean_correction  # both kernels carry it; the choice does not depend on it
    if block_k == 224:  # the 128 x 224 tile has only the one-head kernel
        return "pipelined"
    if schedule == "auto":
        return ("pipelined" if mode in ("threshold", "lambda") and block_q == 128 and
                block_k == 128 else "paired")
    if schedule not in ("paired", "pipelined"):
        raise ValueError(f"unknown schedule {schedule!r}")
    return schedule


def bitmap_shape(num_heads_q: int, *, block_q: int, block_k: int, seqlens) -> tuple[int, int, int]:
    """(rows, Hq, words) of the kept-block bitmap for sequences of lengths
    ``seqlens``: rows = sum ceil(L_b/Bq), words = ceil(ceil(max L_b/Bk)/32)."""
    rows = sum((int(L) + block_q - 1) // block_q for L in seqlens)
    mx = max((int(L) for L in seqlens), default=0)
    words = ((mx + block_k - 1) // block_k + 31) // 32
    return rows, num_heads_q, words


def prefill(q, k, v, *, block_q=128, block_k=128, softmax_scale=None, mode="threshold",
            thresholds=None, log_lambda=None, cu_seqlens=None, max_seqlen=None, layout=None,
            out=None, return_bitmap=False, return_lse=False, return_counts=False,
            workspace=None, stream=None, v_always=False, block_table=None, kv_layout="pthd",
            mean_correction=False, schedule="auto"):
    """Gated causal prefill.  Batched: q [B, Hq, L, d] (layout "bhld") or
    [B, L, Hq, d] ("blhd"); varlen (cu_seqlens int32 on the device): q [Hq, T, d]
    ("htd") or [T, Hq, d] ("thd").  Returns a dict with "out" and, on request,
    "bitmap" (int32 [rows, Hq, words], bit j of word j//32 = keep), "lse"
    (float32 [Hq, rows_of_tokens]) and "counts" (int64 [3]: kept candidates,
    candidates, diagonal-region blocks).  ``v_always`` loads V for skipped
    tiles too (results unchanged; for measuring what the skipped load saves).

    cu_seqlens must be non-decreasing from 0 or more, end at no more than
    the packed token count, and no length may exceed ``max_seqlen``: the
    offsets stay on the device and are not checked (that would need a
    synchronisation per call).

    Paged K/V: with ``block_table`` (int32 [batch, pages_per_sequence] on the
    device), k and v are page pools [pages, page_size, Hkv, d] (``kv_layout``
    "pthd") or [pages, Hkv, page_size, d] ("phtd"), page_size a multiple of
    128; key position pos of sequence b is token pos % page_size of page
    block_table[b, pos // page_size].  q and out keep their layout.

    ``mean_correction``: every skipped candidate block enters the softmax
    through a stand-in built from its mean key and mean value, weighted by its
    key count (threshold and lambda modes, 128 x 128 blocks, contiguous K/V).

    ``schedule``: "paired" (two query heads of a GQA group per CTA, sharing
    each K/V tile), "pipelined" (one query head per CTA, Q.K^T of the next
    tiles issued ahead of the current P.V; Bq = 128, Bk = 128 or 224) or
    "auto" (``resolve_schedule``: pipelined for gated 128 x 128 calls, else
    paired).  The choice never changes the bitmap or the counts; outputs
    differ only in floating-point rounding order."""
    if out is None:
        out = torch.empty_like(q)
    dev = q.device
    _on_device(dev, k=k, v=v, out=out, thresholds=thresholds, cu_seqlens=cu_seqlens,
               block_table=block_table)
    p = _params(q, k, v, out, layout=layout, cu_seqlens=cu_seqlens, max_seqlen=max_seqlen,
                block_q=block_q, block_k=block_k, softmax_scale=softmax_scale, mode=mode,
                thresholds=thresholds, log_lambda=log_lambda, v_always=v_always,
                block_table=block_table, kv_layout=kv_layout, mean_correction=mean_correction,
                schedule=schedule)
    L = _native.lib()
    res = {"out": out}
    if return_bitmap:
        if cu_seqlens is not None:
            cu = cu_seqlens.cpu().tolist()
            lens = [b - a for a, b in zip(cu[:-1], cu[1:])]
        else:
            lens = [p.seqlen] * p.batch
        rows, H, _ = bitmap_shape(p.num_heads_q, block_q=block_q, block_k=block_k, seqlens=lens)
        w = ctypes.c_int(0)
        _check(L.bsfa_bitmap_words_per_row(ctypes.byref(p), ctypes.byref(w)), "bitmap words")
        words = w.value  # the kernel's row pitch (from max_seqlen in varlen mode)
        bm = torch.empty((max(rows, 1), H, max(words, 1)), dtype=torch.int32, device=dev)
        p.kept_bitmap = bm.data_ptr()
        res["bitmap"] = bm[:rows]
    if return_lse:
        rows_tok = p.seqlen if cu_seqlens is not None else p.batch * p.seqlen
        lse = torch.empty((p.num_heads_q, rows_tok), dtype=torch.float32, device=dev)
        p.lse = lse.data_ptr()
        res["lse"] = lse
    if return_counts:
        cnt = torch.empty(3, dtype=torch.int64, device=dev)
        p.block_counts = cnt.data_ptr()
        res["counts"] = cnt
    workspace = _user_workspace(workspace, L.bsfa_prefill_workspace_size(ctypes.byref(p)), dev)
    p.workspace, p.workspace_bytes = workspace.data_ptr(), _nbytes(workspace)
    _check(L.bsfa_prefill_fwd(ctypes.byref(p), _stream(stream, dev)), "bsfa_prefill_fwd")
    return res


def prefill_workspace_bytes(q, k, v, **kw) -> int:
    """Workspace bytes bsfa_prefill_fwd needs for this call's shapes."""
    out = kw.pop("out", None)
    p = _params(q, k, v, out if out is not None else q, layout=kw.get("layout"),
                cu_seqlens=kw.get("cu_seqlens"), max_seqlen=kw.get("max_seqlen"),
                block_q=kw.get("block_q", 128), block_k=kw.get("block_k", 128),
                softmax_scale=kw.get("softmax_scale"), mode=kw.get("mode", "threshold"),
                thresholds=kw.get("thresholds"), log_lambda=kw.get("log_lambda"),
                v_always=kw.get("v_always", False), block_table=kw.get("block_table"),
                kv_layout=kw.get("kv_layout", "pthd"),
                mean_correction=kw.get("mean_correction", False),
                schedule=kw.get("schedule", "auto"))
    return int(_native.lib().bsfa_prefill_workspace_size(ctypes.byref(p)))


def calibrate(q_samples, k_samples, ks, *, block_q=128, block_k=128, softmax_scale=None,
              out=None, workspace=None, stream=None):
    """Thresholds [len(ks), Hq, ceil(L/Bq)] (float32, device) from equal-length
    samples q [Hq, L, d] / k [Hkv, L, d] (bf16 or fp16, one type for all, d contiguous)."""
    n = len(q_samples)
    if n == 0 or n != len(k_samples):
        raise ValueError("need matching non-empty sample lists")
    q0, k0 = q_samples[0], k_samples[0]
    Hq, Ltok, d = q0.shape
    Hkv = k0.shape[0]
    for t in list(q_samples) + list(k_samples):
        if t.dtype != q0.dtype or t.stride(-1) != 1 or t.shape[1] != Ltok or t.shape[2] != d:
            raise ValueError("samples must be [H, L, d] of one type with d contiguous and equal L")
    dcode = _dtype_code(q0)
    dev = q0.device
    _on_device(dev, **{f"sample {i}": t for i, t in enumerate(list(q_samples) + list(k_samples))})
    for t in k_samples:
        if t.shape[0] != Hkv:
            raise ValueError("all k samples must have the same number of heads")
    nq = (Ltok + block_q - 1) // block_q
    if out is None:
        out = torch.empty((len(ks), Hq, nq), dtype=torch.float32, device=dev)
    elif out.dtype != torch.float32 or not out.is_contiguous() or \
            tuple(out.shape) != (len(ks), Hq, nq):
        raise ValueError(f"out must be a contiguous float32 [{len(ks)}, {Hq}, {nq}] tensor")
    _on_device(dev, out=out)
    L = _native.lib()
    workspace = _user_workspace(workspace, L.bsfa_calibrate_workspace_size(Hq, Ltok, block_q,
                                                                           block_k), dev)
    qp = (ctypes.c_void_p * n)(*[t.data_ptr() for t in q_samples])
    kp = (ctypes.c_void_p * n)(*[t.data_ptr() for t in k_samples])
    qst = (ctypes.c_int64 * 2)(q0.stride(0), q0.stride(1))
    kst = (ctypes.c_int64 * 2)(k0.stride(0), k0.stride(1))
    for t in q_samples[1:]:
        if t.stride()[:2] != q0.stride()[:2]:
            raise ValueError("all q samples must share strides")
    for t in k_samples[1:]:
        if t.stride()[:2] != k0.stride()[:2]:
            raise ValueError("all k samples must share strides")
    karr = (ctypes.c_int * len(ks))(*[int(x) for x in ks])
    scale = float(softmax_scale) if softmax_scale else 0.0
    _check(L.bsfa_calibrate(qp, kp, n, Hq, Hkv, Ltok, d, dcode, qst, kst, block_q, block_k, scale,
                            karr, len(ks), ctypes.c_void_p(out.data_ptr()),
                            ctypes.c_void_p(workspace.data_ptr()), _nbytes(workspace),
                            _stream(stream, dev)), "bsfa_calibrate")
    return out


def device_error(stream=None) -> int:
    """Synchronise and return (and clear) the device error word; 0 if clean."""
    code = ctypes.c_uint(0)
    st = _native.lib().bsfa_device_error(_stream(stream), ctypes.byref(code))
    if st not in (0, 4):
        _check(st, "bsfa_device_error")
    return int(code.value)

