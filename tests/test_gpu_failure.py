"""Failure detection on the GPU without a fault: a device-side wait that can
never complete gives up after its time bound, reports through the device
error word, and leaves the context usable for the next call."""
import ctypes

import pytest
import torch

import block_sparse_gated_gb300 as bsfa
from block_sparse_gated_gb300 import _native, api
from block_sparse_gated_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

BSFA_ERR_DEVICE_TIMEOUT = 4
SELFTEST_SITE = 0x1FF


def test_bounded_wait_reports_and_context_survives(cuda_device):
    L = _native.lib()
    assert api.device_error() == 0
    assert L.bsfa_selftest_wait_guard(50_000, api._stream(None)) == 0  # 50 ms bound
    code = ctypes.c_uint(0)
    assert L.bsfa_device_error(api._stream(None), ctypes.byref(code)) == BSFA_ERR_DEVICE_TIMEOUT
    assert code.value == SELFTEST_SITE
    assert api.device_error() == 0  # the word was cleared
    # The context is still usable: a normal call runs and matches itself.
    x = wl.layer_inputs(4, 2, 300, 128, 5, cuda_device)
    a = bsfa.prefill(x.q[None], x.k[None], x.v[None], mode="none")["out"]
    b = bsfa.prefill(x.q[None], x.k[None], x.v[None], mode="none")["out"]
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.isfinite(a.float()).all()
    assert api.device_error() == 0


def test_selftest_rejects_bad_bounds():
    L = _native.lib()
    assert L.bsfa_selftest_wait_guard(0, None) == 1
    assert L.bsfa_selftest_wait_guard(20_000_000, None) == 1
