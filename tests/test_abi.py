"""The C-ABI library loads and exports every function include/*.h declares,
and the binding's ctypes signatures cover the same set.  No GPU compute."""
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b(bsfa_[a-z_0-9]+)\s*\(", text):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def libpath():
    from block_sparse_gated_gb300 import build
    return build.build()


def test_header_declares_the_boundary():
    d = _declared()
    for name in ("bsfa_prefill_fwd", "bsfa_calibrate", "bsfa_prefill_workspace_size",
                 "bsfa_calibrate_workspace_size", "bsfa_device_error", "bsfa_status_string"):
        assert name in d


def test_library_exports_every_declared_symbol(libpath):
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = _declared() - exported
    assert not missing, f"declared but not exported: {sorted(missing)}"


def test_ctypes_binding_loads_every_symbol(libpath):
    from block_sparse_gated_gb300 import _native
    L = _native.lib()
    bound = {name for name, _, _ in _native.SIGNATURES}
    assert bound == _declared()
    for name in bound:
        assert getattr(L, name) is not None


def test_host_side_validation_without_gpu(libpath):
    """Calls that fail host validation return before touching the device."""
    import ctypes
    from block_sparse_gated_gb300 import _native
    L = _native.lib()
    assert L.bsfa_version() > 0
    assert L.bsfa_status_string(0) == b"ok"
    p = _native.FwdParams()
    p.batch, p.num_heads_q, p.num_heads_kv, p.seqlen, p.head_dim = 1, 4, 3, 128, 128
    p.block_q = p.block_k = 128
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 1  # Hq % Hkv != 0
    p.num_heads_kv, p.head_dim = 2, 96
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 2  # unsupported head_dim
    p.head_dim, p.block_k = 128, 96
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 2  # unsupported block size
    p.block_k, p.dtype = 128, 7
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 2  # unknown element type
    p.dtype, p.flags = _native.DTYPE_F16, 8
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 2  # unknown flag bit
    p.flags, p.block_k = _native.FLAG_PIPELINED, 64
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 2  # pipelined: 128 x 128 blocks only
    p.flags, p.block_k = _native.FLAG_PIPELINED | _native.FLAG_MEAN_CORRECTION, 128
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 1  # accepted up to the null tensors
    p.flags = _native.FLAG_PIPELINED
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 1  # accepted up to the null tensors
    # The 128 x 224 tile: accepted with 128-row query blocks only, contiguous
    # K/V and no mean correction.
    p.flags, p.block_q, p.block_k = 0, 128, 224
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 1  # accepted up to the null tensors
    p.block_q = 64
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 2
    p.block_q, p.flags = 128, _native.FLAG_MEAN_CORRECTION
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 2
    p.flags, p.block_table, p.block_table_stride, p.page_size, p.num_pages = 0, 1 << 12, 8, 256, 8
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 2
    p.block_table, p.block_table_stride, p.page_size, p.num_pages = None, 0, 0, 0
    p.block_k = 160
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 2  # no other key tile
    p.block_k = 128
    p.flags = _native.FLAG_V_ALWAYS
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 1  # null tensors
    p.flags = 0
    p.dtype = _native.DTYPE_BF16
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 1  # null tensors
    p.batch = 0
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 0  # empty batch is a no-op
    p.batch = 2
    assert L.bsfa_prefill_workspace_size(ctypes.byref(p)) > 0
    w = ctypes.c_int(0)
    assert L.bsfa_bitmap_words_per_row(ctypes.byref(p), ctypes.byref(w)) == 0 and w.value == 1


def test_params_struct_layout_matches_header(libpath):
    """The ctypes mirror ends with the same field the header's struct ends
    with, at the C compiler's offset (checked by compiling a tiny probe)."""
    import ctypes
    import tempfile
    from block_sparse_gated_gb300 import _native
    src = (
        '#include <stddef.h>\n#include <stdio.h>\n#include "bsfa.h"\n'
        'int main(void) { printf("%zu %zu %zu %zu %zu\\n", sizeof(bsfa_fwd_params), '
        'offsetof(bsfa_fwd_params, dtype), offsetof(bsfa_fwd_params, flags), '
        'offsetof(bsfa_fwd_params, block_table), offsetof(bsfa_fwd_params, num_pages)); '
        'return 0; }\n')
    with tempfile.TemporaryDirectory() as tmp:
        c = os.path.join(tmp, "probe.c")
        exe = os.path.join(tmp, "probe")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        got = tuple(map(int, subprocess.run([exe], capture_output=True, text=True,
                                            check=True).stdout.split()))
    F = _native.FwdParams
    assert (ctypes.sizeof(F), F.dtype.offset, F.flags.offset, F.block_table.offset,
            F.num_pages.offset) == got


def test_paged_parameters_are_validated_on_the_host(libpath):
    """Paged K/V: page size, pool size and table width are checked before any
    launch (the tensor pointers here are never dereferenced)."""
    import ctypes
    from block_sparse_gated_gb300 import _native
    L = _native.lib()
    p = _native.FwdParams()
    p.batch, p.num_heads_q, p.num_heads_kv, p.seqlen, p.head_dim = 2, 4, 2, 1000, 128
    p.block_q = p.block_k = 128
    p.mode = 2
    p.q = p.k = p.v = p.o = 1 << 20  # 16-byte aligned stand-ins, never read
    p.q_stride[:] = p.o_stride[:] = (4 * 1000 * 128, 1000 * 128, 128)
    p.k_stride[:] = p.v_stride[:] = (256 * 2 * 128, 128, 2 * 128)  # [pages, 256, Hkv, d]
    p.block_table, p.block_table_stride, p.page_size, p.num_pages = 1 << 12, 4, 200, 16
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 2  # page size not a multiple of 128
    p.page_size = 256
    p.num_pages = 0
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 1  # empty pool
    p.num_pages, p.block_table_stride = 16, 3
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 1  # 3 pages of 256 < 1000 tokens
    p.block_table_stride = 4
    p.k_stride[0] = 100  # page stride not a multiple of 8 elements
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 2
    p.k_stride[0] = 256 * 2 * 128
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 5  # all fine up to the missing workspace
    p.flags = _native.FLAG_V_ALWAYS
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 2  # no paged V-always kernels


def test_mean_correction_parameters_are_validated_on_the_host(libpath):
    import ctypes
    from block_sparse_gated_gb300 import _native
    L = _native.lib()
    p = _native.FwdParams()
    p.batch, p.num_heads_q, p.num_heads_kv, p.seqlen, p.head_dim = 1, 4, 2, 1000, 128
    p.block_q = p.block_k = 128
    p.mode = 1
    p.q = p.k = p.v = p.o = 1 << 20  # 16-byte aligned stand-ins, never read
    p.q_stride[:] = p.o_stride[:] = (4 * 1000 * 128, 1000 * 128, 128)
    p.k_stride[:] = p.v_stride[:] = (2 * 1000 * 128, 1000 * 128, 128)
    plain = L.bsfa_prefill_workspace_size(ctypes.byref(p))
    p.flags = _native.FLAG_MEAN_CORRECTION
    # the workspace grows by two block-mean tables: 2 KV heads x 8 blocks x 128 x 2 bytes each
    corr = L.bsfa_prefill_workspace_size(ctypes.byref(p))
    assert corr >= plain + 2 * 2 * 8 * 128 * 2
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 5  # fine up to the missing workspace
    # Both schedules carry the option, with the same workspace.
    p.flags = _native.FLAG_MEAN_CORRECTION | _native.FLAG_PIPELINED
    assert L.bsfa_prefill_workspace_size(ctypes.byref(p)) == corr
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 5
    p.flags = _native.FLAG_MEAN_CORRECTION
    p.mode = 2
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 2  # nothing is skipped without a gate
    p.mode, p.block_k = 0, 64
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 2  # 128 x 128 blocks only
    p.block_k = 128
    p.flags |= _native.FLAG_V_ALWAYS
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 2
    p.flags = _native.FLAG_MEAN_CORRECTION
    p.block_table, p.block_table_stride, p.page_size, p.num_pages = 1 << 12, 8, 128, 8
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 2  # contiguous K/V only
    # The block-mean pass's head limit (d * Hkv <= 1024) is part of the
    # validation too: it is refused here, with no workspace and no device.
    p.block_table, p.block_table_stride, p.page_size, p.num_pages = None, 0, 0, 0
    p.num_heads_q, p.num_heads_kv = 16, 16
    p.q_stride[:] = p.o_stride[:] = (16 * 1000 * 128, 1000 * 128, 128)
    p.k_stride[:] = p.v_stride[:] = (16 * 1000 * 128, 1000 * 128, 128)
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 2
    p.thresholds, p.thresholds_nq = 1 << 20, 1
    p.head_dim = 64  # 16 x 64 = 1024: within the limit, so only the workspace is missing
    p.q_stride[:] = p.o_stride[:] = (16 * 1000 * 64, 1000 * 64, 64)
    p.k_stride[:] = p.v_stride[:] = (16 * 1000 * 64, 1000 * 64, 64)
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 5


def test_size_limits_are_rejected_on_the_host(libpath):
    """The documented limits: 4096 sequences per call, 16384 query tiles of
    128 rows per sequence; calibration: 16 budgets, 8192 key blocks."""
    import ctypes
    from block_sparse_gated_gb300 import _native
    L = _native.lib()
    p = _native.FwdParams()
    p.batch, p.num_heads_q, p.num_heads_kv, p.head_dim = 1, 2, 2, 128
    p.block_q = p.block_k = 128
    p.mode = 2
    p.seqlen = 16384 * 128 + 1
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 2  # one tile too many
    p.seqlen, p.batch = 1024, 4097
    assert L.bsfa_prefill_fwd(ctypes.byref(p), None) == 2  # too many sequences
    assert L.bsfa_prefill_workspace_size(ctypes.byref(p)) == 0
    dummy = (ctypes.c_void_p * 1)(1 << 20)
    st = (ctypes.c_int64 * 2)(1024 * 128, 128)
    out = ctypes.c_void_p(1 << 20)
    ks = (ctypes.c_int * 17)(*range(1, 18))
    assert L.bsfa_calibrate(dummy, dummy, 1, 2, 2, 1024, 128, 0, st, st, 128, 128, 0.0, ks, 17,
                            out, out, 1 << 30, None) == 2  # 17 budgets
    assert L.bsfa_calibrate(dummy, dummy, 1, 2, 2, 8193 * 128, 128, 0, st, st, 128, 128, 0.0,
                            ks, 1, out, out, 1 << 30, None) == 2  # 8193 key blocks


def test_mixed_element_types_are_rejected_before_the_library():
    import torch
    from block_sparse_gated_gb300 import api
    q = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 2, 128, 64, dtype=torch.float16)
    with pytest.raises(TypeError):
        api._params(q, k, k, q, layout=None, cu_seqlens=None, max_seqlen=None, block_q=128,
                    block_k=128, softmax_scale=None, mode="none", thresholds=None,
                    log_lambda=None)
    with pytest.raises(TypeError):
        api._params(q.float(), q.float(), q.float(), q.float(), layout=None, cu_seqlens=None,
                    max_seqlen=None, block_q=128, block_k=128, softmax_scale=None, mode="none",
                    thresholds=None, log_lambda=None)


def test_binding_checks_paged_arguments():
    """The Python binding's own checks of page pools and block tables (before
    the library sees the call)."""
    import torch
    from block_sparse_gated_gb300 import api
    q = torch.zeros(1, 4, 300, 128, dtype=torch.bfloat16)
    pool = torch.zeros(3, 256, 2, 128, dtype=torch.bfloat16)  # [pages, page_size, Hkv, d]
    table = torch.zeros(1, 2, dtype=torch.int32)
    kw = dict(layout=None, cu_seqlens=None, max_seqlen=None, block_q=128, block_k=128,
              softmax_scale=None, mode="none", thresholds=None, log_lambda=None)
    p = api._params(q, pool, pool, q, block_table=table, **kw)
    assert (p.page_size, p.num_pages, p.block_table_stride) == (256, 3, 2)
    assert tuple(p.k_stride) == (256 * 2 * 128, 128, 2 * 128)
    p = api._params(q, pool.permute(0, 2, 1, 3).contiguous(), pool.permute(0, 2, 1, 3).contiguous(),
                    q, block_table=table, kv_layout="phtd", **kw)
    assert (p.page_size, tuple(p.k_stride)) == (256, (2 * 256 * 128, 256 * 128, 128))
    with pytest.raises(ValueError):
        api._params(q, pool, pool, q, block_table=table.long(), **kw)  # int32 table only
    with pytest.raises(ValueError):
        api._params(q, pool, pool[:, :128], q, block_table=table, **kw)  # pools disagree
    p = api._params(q, q[:, :2], q[:, :2], q, mean_correction=True, **kw)
    assert p.flags == 2


def test_binding_rejects_host_tensors_before_the_library():
    """Host tensors never reach a kernel: the binding refuses them."""
    import torch
    from block_sparse_gated_gb300 import api
    q = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        api.prefill(q, q, q, mode="none")
    with pytest.raises(ValueError, match="CUDA"):
        api.calibrate([q[0]], [q[0]], [1])
    with pytest.raises(ValueError, match="expected cuda:0"):
        api._on_device(torch.device("cuda", 0), thresholds=torch.zeros(2, 1))


def test_binding_checks_shapes_the_library_cannot_see():
    """Extents that the C ABI takes from q alone (batch, head dimension, the
    threshold table's rows, the block table's rows and columns) are checked
    against every other tensor before the call."""
    import torch
    from block_sparse_gated_gb300 import api
    bf = torch.bfloat16
    q = torch.zeros(2, 4, 300, 128, dtype=bf)
    kv = torch.zeros(2, 2, 300, 128, dtype=bf)
    kw = dict(layout=None, cu_seqlens=None, max_seqlen=None, block_q=128, block_k=128,
              softmax_scale=None, mode="none", thresholds=None, log_lambda=None)
    p = api._params(q, kv, kv, q, **kw)
    assert (p.batch, p.num_heads_q, p.num_heads_kv, p.seqlen, p.head_dim) == (2, 4, 2, 300, 128)
    with pytest.raises(ValueError, match="head dimensions"):
        api._params(q, kv[..., :64], kv[..., :64], q, **kw)
    with pytest.raises(ValueError, match="batch"):
        api._params(q, kv[:1], kv[:1], q, **kw)
    with pytest.raises(ValueError, match="batch"):
        api._params(q, kv, kv, q[:1], **kw)
    with pytest.raises(ValueError, match="batch"):
        api._params(q[0], kv, kv, q[0], **kw)  # one sequence with batched K/V
    thr = dict(kw, mode="threshold")
    api._params(q, kv, kv, q, **dict(thr, thresholds=torch.zeros(4, 3)))
    with pytest.raises(ValueError, match="thresholds"):
        api._params(q, kv, kv, q, **dict(thr, thresholds=torch.zeros(2, 3)))  # rows != Hq
    # varlen: int32 offsets and a max_seqlen
    qv, kvv = torch.zeros(4, 300, 128, dtype=bf), torch.zeros(2, 300, 128, dtype=bf)
    cu = torch.tensor([0, 100, 300], dtype=torch.int32)
    p = api._params(qv, kvv, kvv, qv, **dict(kw, cu_seqlens=cu, max_seqlen=200))
    assert (p.batch, p.max_seqlen) == (2, 200)
    with pytest.raises(ValueError, match="cu_seqlens"):
        api._params(qv, kvv, kvv, qv, **dict(kw, cu_seqlens=cu.long(), max_seqlen=200))
    with pytest.raises(ValueError, match="max_seqlen"):
        api._params(qv, kvv, kvv, qv, **dict(kw, cu_seqlens=cu))
    # paged: one table row per sequence, enough pages for the longest one
    pool = torch.zeros(6, 128, 2, 128, dtype=bf)
    api._params(q, pool, pool, q, block_table=torch.zeros(2, 3, dtype=torch.int32), **kw)
    with pytest.raises(ValueError, match="block_table"):
        api._params(q, pool, pool, q, block_table=torch.zeros(1, 3, dtype=torch.int32), **kw)
    with pytest.raises(ValueError, match="block_table"):
        api._params(q, pool, pool, q, block_table=torch.zeros(2, 2, dtype=torch.int32), **kw)
    api._params(qv, pool, pool, qv, block_table=torch.zeros(2, 2, dtype=torch.int32),
                **dict(kw, cu_seqlens=cu, max_seqlen=200))
    with pytest.raises(ValueError, match="block_table"):
        api._params(qv, pool, pool, qv, block_table=torch.zeros(2, 1, dtype=torch.int32),
                    **dict(kw, cu_seqlens=cu, max_seqlen=200))


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """No fallback: without the built library the first call raises."""
    import torch
    from block_sparse_gated_gb300 import _native, api
    monkeypatch.setattr(_native, "LIB_PATH", str(tmp_path / "libbsfa.so"))
    monkeypatch.setattr(_native, "_lib", None)
    with pytest.raises(RuntimeError, match="is not built"):
        _native.lib()
    with pytest.raises(RuntimeError, match="is not built"):
        api.prefill_workspace_bytes(*(torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16),) * 3,
                                    mode="none")


def test_plain_c_caller_links_and_gets_host_statuses(libpath):
    """The boundary is usable from C alone: a C program built with gcc against
    include/bsfa.h and linked to the library gets sizes, words per row and
    host-side statuses back (no device work)."""
    import tempfile
    src = r'''
#include <stdio.h>
#include <string.h>
#include "bsfa.h"
int main(void) {
  bsfa_fwd_params p;
  memset(&p, 0, sizeof p);
  p.batch = 2; p.num_heads_q = 4; p.num_heads_kv = 2; p.seqlen = 1000; p.head_dim = 128;
  p.block_q = 128; p.block_k = 64; p.mode = BSFA_GATE_NONE;
  int words = -1;
  int st_words = bsfa_bitmap_words_per_row(&p, &words);
  size_t ws = bsfa_prefill_workspace_size(&p);
  p.head_dim = 96;
  int st_d96 = bsfa_prefill_fwd(&p, NULL);
  p.head_dim = 128; p.batch = 0;
  int st_empty = bsfa_prefill_fwd(&p, NULL);
  printf("%d %d %d %zu %d %d %s\n", bsfa_version() > 0, st_words, words, ws, st_d96, st_empty,
         bsfa_status_string(BSFA_ERR_WORKSPACE));
  return 0;
}
'''
    libdir = os.path.dirname(libpath)
    with tempfile.TemporaryDirectory() as tmp:
        c = os.path.join(tmp, "caller.c")
        exe = os.path.join(tmp, "caller")
        open(c, "w").write(src)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), c, "-o", exe, libpath,
                        f"-Wl,-rpath,{libdir}"], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()
    ok, st_words, words, ws, st_d96, st_empty = map(int, out[:6])
    assert ok == 1 and st_words == 0 and words == 1  # ceil(ceil(1000 / 64) / 32) = 1
    assert ws > 0
    assert st_d96 == 2 and st_empty == 0  # unsupported head_dim; an empty batch is a no-op
    assert " ".join(out[6:]) == "workspace missing, misaligned or too small"
