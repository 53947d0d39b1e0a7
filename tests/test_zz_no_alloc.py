"""flce_forward_noalloc: the forward pass for callers that cannot allocate
device memory (a custom operator inside a runtime that owns every device
allocation, or a loop that must not stall on cudaMalloc/cudaFree).  Its scratch
is a fixed array inside the library, so the test calls it through the C-ABI
twice in a row on different problems — the second call must not see the
first call's leftovers — and compares each result with flce_forward's, at the
tolerances the other parity tests use.  This file is collected last."""
import ctypes
import math

import numpy as np
import pytest

import synth
from helpers import LOSS_RTOL, LSE_ATOL, to_device

torch = pytest.importorskip("torch")

import lm_head_cross_gb300 as flce  # noqa: E402
from lm_head_cross_gb300 import binding  # noqa: E402


def _noalloc(L, problem, X, W, y):
    n, h = X.shape
    v = W.shape[0]
    p = binding.Problem(n, h, v, problem.ignore_index, binding.REDUCTIONS[problem.reduction])
    loss = torch.empty(1, dtype=torch.float32, device=X.device)
    lse = torch.empty(n, dtype=torch.float32, device=X.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = L.flce_forward_noalloc(ctypes.byref(p), ctypes.c_void_p(X.data_ptr()), ctypes.c_void_p(W.data_ptr()),
                                ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(loss.data_ptr()),
                                ctypes.c_void_p(lse.data_ptr()), stream)
    return st, loss, lse


def _lib():
    L = flce.lib()
    L.flce_forward_noalloc.argtypes = [ctypes.POINTER(binding.Problem)] + [ctypes.c_void_p] * 6
    L.flce_forward_noalloc.restype = ctypes.c_int
    return L


@pytest.mark.gpu
def test_noalloc_forward_matches_forward_twice():
    L = _lib()
    problems = [
        synth.make_problem(4096, 512, 20000, seed=31, labels="zipf", ignore_frac=0.05, reduction="mean"),
        synth.make_problem(1000, 264, 3001, seed=32, labels="uniform", ignore_frac=0.2, reduction="sum"),
    ]
    for p in problems:
        X, W, y = to_device(p)
        st, loss, lse = _noalloc(L, p, X, W, y)
        assert st == 0, flce.status_string(st)
        ref_loss, ref_lse, ws = flce.forward(X, W, y, p.ignore_index, p.reduction)
        assert flce.read_device_status(ws) == 0
        torch.cuda.synchronize()
        a, b = float(loss.item()), float(ref_loss.item())
        assert abs(a - b) <= LOSS_RTOL * abs(b), (a, b)
        assert (lse - ref_lse).abs().max().item() <= LSE_ATOL


@pytest.mark.gpu
def test_noalloc_limits_and_error_reporting():
    L = _lib()
    # beyond the fixed maximum: rejected on the host, nothing launched
    big = binding.Problem(32769, 64, 100, -100, 0)
    z = ctypes.c_void_p(0x1000)
    assert L.flce_forward_noalloc(ctypes.byref(big), z, z, z, z, z, None) == 9
    # a label out of range shows up as a NaN loss
    p = synth.make_problem(256, 64, 300, seed=33)
    p.labels[5] = 300
    X, W, y = to_device(p)
    st, loss, _ = _noalloc(L, p, X, W, y)
    assert st == 0
    assert math.isnan(float(loss.item()))
    # and the next clean call is unaffected
    p.labels[5] = 1
    X, W, y = to_device(p)
    st, loss, _ = _noalloc(L, p, X, W, y)
    ref_loss, _, _ = flce.forward(X, W, y, p.ignore_index, p.reduction)
    assert st == 0 and abs(float(loss.item()) - float(ref_loss.item())) <= LOSS_RTOL * abs(float(ref_loss.item()))
