"""flce_forward_noalloc: the forward pass for callers that cannot allocate
device memory (a custom operator inside a runtime that owns every device
allocation, or a loop that must not stall on cudaMalloc/cudaFree).  Its scratch
is a fixed array inside the library, shared by every call, so the tests call it
through the C-ABI several times in a row on different problems — small after
large and large after small, up to the 32768-row maximum that fills the scratch
regions — and check every result against the fp64 oracle and against
flce_forward, at the tolerances the other parity tests use: a call that read a
previous call's leftovers would fail.  This file is collected last."""
import ctypes
import math

import numpy as np
import pytest

import oracle
import synth
from helpers import LOSS_RTOL, LSE_ATOL, assert_loss, assert_lse, to_device

torch = pytest.importorskip("torch")

import lm_head_cross_gb300 as flce  # noqa: E402
from lm_head_cross_gb300 import binding  # noqa: E402


def _noalloc(L, problem, X, W, y, reduction=None, shift=0, seq_len=0):
    n, h = X.shape
    v = W.shape[0]
    red = reduction or problem.reduction
    p = binding.Problem(n, h, v, problem.ignore_index, binding.REDUCTIONS[red], shift, seq_len if shift else 0)
    loss = torch.empty(n if red == "none" else 1, dtype=torch.float32, device=X.device)
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


def _check(L, p, reduction=None, shift=0, seq_len=0):
    red = reduction or p.reduction
    X, W, y = to_device(p)
    st, loss, lse = _noalloc(L, p, X, W, y, red, shift, seq_len)
    assert st == 0, flce.status_string(st)
    ref_loss, ref_lse, ws = flce.forward(X, W, y, p.ignore_index, red, shift=shift, seq_len=seq_len)
    assert flce.read_device_status(ws) == 0
    torch.cuda.synchronize()
    lab = oracle.shift_labels(p.labels, seq_len, p.ignore_index) if shift else p.labels
    f = oracle.forward(oracle.widen_bf16(p.X), oracle.widen_bf16(p.W), lab, p.ignore_index, red)
    assert_lse(lse.cpu().numpy(), f["lse"])
    assert (lse - ref_lse).abs().max().item() <= LSE_ATOL
    if red == "none":
        np.testing.assert_allclose(loss.cpu().numpy(), f["loss"], rtol=LOSS_RTOL, atol=LSE_ATOL)
        np.testing.assert_allclose(loss.cpu().numpy(), ref_loss.cpu().numpy(), rtol=LOSS_RTOL, atol=LSE_ATOL)
    else:
        assert_loss(float(loss.item()), f["loss"])
        a, b = float(loss.item()), float(ref_loss.item())
        assert abs(a - b) <= LOSS_RTOL * abs(b), (a, b)


PROBLEMS = {
    "large": lambda: synth.make_problem(4096, 512, 20000, seed=31, labels="zipf", ignore_frac=0.05, reduction="mean"),
    "small": lambda: synth.make_problem(1000, 264, 3001, seed=32, labels="uniform", ignore_frac=0.2, reduction="sum"),
    "max_rows": lambda: synth.make_problem(32768, 64, 300, seed=34, labels="uniform", ignore_frac=0.1,
                                           reduction="mean"),
}


@pytest.mark.gpu
@pytest.mark.parametrize("order", [("large", "small"), ("small", "large"), ("max_rows", "small", "max_rows")],
                         ids=["large-then-small", "small-then-large", "max-small-max"])
def test_noalloc_forward_calls_in_a_row(order):
    L = _lib()
    for name in order:
        _check(L, PROBLEMS[name]())


@pytest.mark.gpu
def test_noalloc_reduction_none_and_shift():
    L = _lib()
    p = synth.make_problem(1200, 136, 5001, seed=35, labels="zipf", ignore_frac=0.1, reduction="mean")
    _check(L, p, "none")
    _check(L, p, "mean", shift=1, seq_len=300)
    _check(L, p, "none", shift=1, seq_len=400)


@pytest.mark.gpu
def test_noalloc_limits_and_error_reporting():
    L = _lib()
    # beyond the fixed maximum: rejected on the host, nothing launched
    big = binding.Problem(32769, 64, 100, -100, 0)
    z = ctypes.c_void_p(0x1000)
    assert L.flce_forward_noalloc(ctypes.byref(big), z, z, z, z, z, None) == 9
    # a label out of range shows up as a NaN loss: the scalar, or every per-row loss
    p = synth.make_problem(256, 64, 300, seed=33)
    p.labels[5] = 300
    X, W, y = to_device(p)
    st, loss, _ = _noalloc(L, p, X, W, y)
    assert st == 0
    assert math.isnan(float(loss.item()))
    st, loss, _ = _noalloc(L, p, X, W, y, "none")
    assert st == 0
    assert torch.isnan(loss).all().item()
    # and the next clean call is unaffected
    p.labels[5] = 1
    _check(L, p)
