"""Shared helpers for the parity tests: moving synthetic problems to the GPU and
the tolerances the library promises (loss relative 1e-3; dX and dW max-abs
2e-2 x max|ref|; lse absolute 2e-3; integer handling exact)."""
import numpy as np

LOSS_RTOL = 1e-3
GRAD_FRAC = 2e-2
LSE_ATOL = 2e-3


def to_device(problem, device="cuda"):
    import torch
    X = torch.from_numpy(problem.X.view(np.int16)).view(torch.bfloat16).to(device)
    W = torch.from_numpy(problem.W.view(np.int16)).view(torch.bfloat16).to(device)
    y = torch.from_numpy(problem.labels.astype(np.int32)).to(device)
    return X, W, y


def assert_loss(got, want, rtol=LOSS_RTOL):
    tol = rtol * max(abs(want), 1e-30)
    assert abs(got - want) <= tol, f"loss {got} vs oracle {want} (tol {tol})"


def assert_lse(got, want, atol=LSE_ATOL):
    err = np.abs(np.asarray(got, np.float64) - np.asarray(want, np.float64)).max()
    assert err <= atol, f"lse max abs err {err} > {atol}"


def assert_grad(got, want, frac=GRAD_FRAC, name="grad"):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    scale = np.abs(want).max()
    err = np.abs(got - want).max()
    assert err <= frac * scale, f"{name} max abs err {err} > {frac} x max|ref| {scale}"


def golden_forward(name, problem=None):
    """The oracle's stored full-forward results of a large workload (per-row lse,
    loss, n_valid), written by tests/golden/make_workload_golden.py; checked
    against the problem's input bytes when it is given."""
    import importlib.util
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "make_workload_golden.py")
    spec = importlib.util.spec_from_file_location("make_workload_golden", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.load(name, problem)
