"""GPU parity sweep: seeded random problems that exercise every call on the same
inputs — fwd_bwd on both paths (shapes, label mix, ignore fraction up to every
row, reduction, causal shift, logit scale), the per-row top-k, and the
soft-target KL on both paths (random ids with repeats, rows without mass) —
each against the fp64 oracle, element by element."""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_grad, assert_loss, assert_lse, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import lm_head_cross_gb300 as flce  # noqa: E402


def _check_fwd_bwd(p, red, shift, s_len, rowchunk, what):
    X, W, y = to_device(p)
    loss, lse, dX, dW, ws = flce.fwd_bwd(X, W, y, p.ignore_index, red, rowchunk=rowchunk, shift=shift,
                                         seq_len=s_len if shift else 0)
    assert flce.read_device_status(ws) == 0, what
    labels = oracle.shift_labels(p.labels, s_len, p.ignore_index) if shift else p.labels
    ref = oracle.full(oracle.widen_bf16(p.X), oracle.widen_bf16(p.W), labels, p.ignore_index, red)
    got = loss.cpu().numpy().astype(np.float64)
    if red == "none":
        np.testing.assert_allclose(got, ref["loss"], rtol=1e-3, atol=2e-3, err_msg=what)
    else:
        assert abs(float(got[0]) - ref["loss"]) <= 1e-3 * max(abs(ref["loss"]), 1e-6), what
    assert_lse(lse.cpu().numpy(), ref["lse"])
    if np.abs(ref["dX"]).max() > 0:
        assert_grad(dX.float().cpu().numpy(), ref["dX"], name="dX " + what)
        assert_grad(dW.float().cpu().numpy(), ref["dW"], name="dW " + what)
    else:
        assert not dX.float().abs().max().item() and not dW.float().abs().max().item(), what
    return X, W


def _check_topk(p, X, W, k, what):
    idx, val, lse, ws = flce.topk(X, W, k)
    assert flce.read_device_status(ws) == 0, what
    Xd, Wd = oracle.widen_bf16(p.X), oracle.widen_bf16(p.W)
    _, rval, rlse = oracle.topk(Xd, Wd, k)
    assert_lse(lse.cpu().numpy(), rlse)
    tol = 2e-3 * max(1.0, float(np.abs(rval).max()))
    np.testing.assert_allclose(val.cpu().numpy(), rval, rtol=0, atol=tol, err_msg=what)
    got = np.take_along_axis(Xd @ Wd.T, idx.cpu().numpy().astype(np.int64), axis=1)
    np.testing.assert_allclose(got, val.cpu().numpy(), rtol=0, atol=tol, err_msg=what)


def _check_soft(p, X, W, rng, what):
    n, v = p.n, p.v
    k = int(rng.integers(1, 17))
    idx = rng.integers(0, v, size=(n, k)).astype(np.int32)
    q = rng.random((n, k)).astype(np.float32)
    q[rng.random((n, k)) < 0.2] = 0.0
    q = (q / np.maximum(q.sum(axis=1, keepdims=True), 1e-30)).astype(np.float32)
    red = ["mean", "sum", "none"][int(rng.integers(0, 3))]
    rowchunk = bool(rng.integers(0, 2))
    what = f"{what} soft k={k} {red} rowchunk={rowchunk}"
    loss, lse, dX, dW, ws = flce.soft_fwd_bwd(X, W, torch.from_numpy(idx).cuda(), torch.from_numpy(q).cuda(), red,
                                              rowchunk=rowchunk)
    assert flce.read_device_status(ws) == 0, what
    ref = oracle.soft_full(oracle.widen_bf16(p.X), oracle.widen_bf16(p.W), idx, q.astype(np.float64), red)
    if red == "none":
        assert np.abs(loss.cpu().numpy() - ref["loss"]).max() <= 2e-3 + 1e-3 * np.abs(ref["loss"]).max(), what
    else:
        assert_loss(float(loss.item()), ref["loss"])
    assert_lse(lse.cpu().numpy(), ref["lse"])
    if np.abs(ref["dX"]).max() > 0:
        assert_grad(dX.float().cpu().numpy(), ref["dX"], name="dX " + what)
        assert_grad(dW.float().cpu().numpy(), ref["dW"], name="dW " + what)


def test_sweep_every_call():
    """60 seeded random problems, each through fwd_bwd (one of the two paths), top-k
    and the soft-target KL."""
    rng = np.random.default_rng(4242)
    for case in range(60):
        seq = int(rng.integers(1, 6))
        s_len = int(rng.integers(1, 300))
        n = seq * s_len
        h = 8 * int(rng.integers(1, 80))
        v = int(rng.integers(1, 12000))
        red = ["mean", "sum", "none"][int(rng.integers(0, 3))]
        shift = int(rng.integers(0, 2)) if s_len > 1 else 0
        rowchunk = bool(rng.integers(0, 2))
        p = synth.make_problem(n, h, v, seed=70000 + case, labels=["uniform", "zipf"][int(rng.integers(0, 2))],
                               ignore_frac=float(rng.choice([0.0, 0.1, 0.5, 1.0])), reduction=red,
                               x_std=float(rng.choice([0.25, 1.0, 4.0])), w_std=float(rng.choice([0.02, 0.1, 0.3])))
        what = f"case {case}: n={n} h={h} v={v} {red} shift={shift} rowchunk={rowchunk}"
        X, W = _check_fwd_bwd(p, red, shift, s_len, rowchunk, what)
        _check_topk(p, X, W, min(int(rng.integers(1, 17)), v), what)
        _check_soft(p, X, W, rng, what)
