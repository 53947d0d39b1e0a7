"""Parity at the five workloads' full sizes, in the launch the benchmark times
(one flce_fwd_bwd with a caller workspace).

Every output the fp64 oracle can compute on its own terms is compared with it:
the whole problem for the two smaller workloads; for the others, per-row lse
and dX on sampled rows (each needs only that row).  dW needs every row's lse;
the oracle's own full forward provides it where that finishes in tens of
seconds (N=8192), and elsewhere dW is checked through properties that hold
at any size:

* sum_j dW_j = 0 (each row of G sums to zero over the vocabulary);
* X^T dX = dW^T W (both equal X^T G W), an H x H identity tying dW to the
  oracle-checked dX;
* the loss equals the reduction of (lse_i - z_{i,y_i}) over valid rows with the
  oracle's own target logits z.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import LOSS_RTOL, assert_grad, assert_loss, assert_lse, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import lm_head_cross_gb300 as flce  # noqa: E402


def sample_rows(p, k, rng):
    n = p.n
    base = set(rng.choice(n, size=min(n, k), replace=False).tolist())
    base |= {0, n - 1, n - 2, max(0, n - 128)}
    ign = np.nonzero(p.labels == p.ignore_index)[0]
    base |= set(ign[:4].tolist())
    if p.outlier_ids is not None:
        hit = np.nonzero(np.isin(p.labels, p.outlier_ids))[0]
        base |= set(hit[:16].tolist())
    return np.array(sorted(base), dtype=np.int64)


def sample_ids(p, k, rng):
    v = p.v
    ids = set(rng.choice(v, size=min(v, k), replace=False).tolist())
    lab = p.labels[p.labels != p.ignore_index]
    ids |= set(np.argsort(-np.bincount(lab, minlength=v))[:8].tolist())   # most frequent labels
    ids |= {0, v - 1}
    if p.outlier_ids is not None:
        ids |= set(p.outlier_ids[:16].tolist())
    return np.array(sorted(ids), dtype=np.int64)


def gpu_properties(p, X, W, dX, dW, valid):
    # ignored rows: exactly zero gradient rows
    assert torch.count_nonzero(dX[torch.from_numpy(~valid).to(dX.device)]).item() == 0
    # sum over the vocabulary of dW vanishes up to bf16 rounding of dW
    dWf = dW.float()
    resid = dWf.double().sum(0).abs().max().item()
    bound = 2 * 2.0 ** -8 * dWf.double().abs().sum(0).max().item()
    assert resid <= bound, ("vocab sum of dW", resid, bound)
    # X^T dX = dW^T W
    m1 = X.float().T @ dX.float()
    m2 = dWf.T @ W.float()
    err = (m1 - m2).abs().max().item()
    scale = m1.abs().max().item()
    assert err <= 2e-2 * scale, ("X^T dX vs dW^T W", err, scale)


@pytest.mark.parametrize("name", ["n8192_h2048_v32000", "n8192_h4096_v128256", "n32768_h4096_v151936",
                                  "n131072_h4096_v131072"])
def test_workload_full_size(name):
    p = synth.workload_problem(name)
    rng = np.random.default_rng(101 + synth.WORKLOADS[name]["seed"])
    X, W, y = to_device(p)
    # the recompute path (minimal workspace) must agree with the fused path
    loss_m, lse_m, dX_m, dW_m, ws = flce.fwd_bwd(X, W, y, p.ignore_index, p.reduction, minimal_workspace=True)
    assert flce.read_device_status(ws) == 0
    del ws
    loss, lse, dX, dW, ws = flce.fwd_bwd(X, W, y, p.ignore_index, p.reduction)
    assert flce.read_device_status(ws) == 0
    del ws
    assert abs(float(loss_m.item()) - float(loss.item())) <= 1e-4 * abs(float(loss.item()))
    assert (lse_m - lse).abs().max().item() <= 1e-3
    for a, b, name in ((dX, dX_m, "dX"), (dW, dW_m, "dW")):
        err = (a.float() - b.float()).abs().max().item()
        assert err <= 1e-2 * b.float().abs().max().item(), (name, err)
    del loss_m, lse_m, dX_m, dW_m
    loss = float(loss.item())
    lse_g = lse.cpu().numpy()
    valid = p.labels != p.ignore_index
    n_valid = int(valid.sum())
    s = oracle.grad_scale(n_valid, p.reduction)

    Xd = oracle.widen_bf16(p.X)
    Wd = oracle.widen_bf16(p.W)
    full_forward = p.n <= 32768   # the oracle's full forward: ~20 s (N=8192) to ~90 s (N=32768) on 16 cores
    if name == synth.DEFAULT_WORKLOAD:
        ref = oracle.full(Xd, Wd, p.labels, p.ignore_index, p.reduction)
        assert_loss(loss, ref["loss"])
        assert_lse(lse_g, ref["lse"])
        assert_grad(dX.float().cpu().numpy(), ref["dX"], name="dX")
        assert_grad(dW.float().cpu().numpy(), ref["dW"], name="dW")
    else:
        rows = sample_rows(p, 256 if p.n <= 32768 else 192, rng)
        lse_r, _ = oracle.lse_and_target(Xd, Wd, p.labels, p.ignore_index, rows)
        assert_lse(lse_g[rows], lse_r)
        dx_r = oracle.backward_dx_rows(Xd, Wd, p.labels, rows, s, p.ignore_index, lse_rows=lse_r)
        assert_grad(dX[torch.from_numpy(rows).cuda()].float().cpu().numpy(), dx_r, name="dX rows")
        # target logits of every valid row, from the oracle
        tgt = np.zeros(p.n)
        vi = np.nonzero(valid)[0]
        for s0 in range(0, vi.size, 8192):
            r = vi[s0:s0 + 8192]
            tgt[r] = np.einsum("ij,ij->i", Xd[r], Wd[p.labels[r]])
        total = float(np.sum((lse_g.astype(np.float64) - tgt)[valid]))
        want = total / n_valid if p.reduction == "mean" else total
        assert abs(loss - want) <= LOSS_RTOL * abs(want), (loss, want)
        if full_forward:
            f = oracle.forward(Xd, Wd, p.labels, p.ignore_index, p.reduction)
            assert_loss(loss, f["loss"])
            assert_lse(lse_g, f["lse"])
            ids = sample_ids(p, 64, rng)
            dw_r = oracle.backward_dw_ids(Xd, Wd, p.labels, f["lse"], ids, s, p.ignore_index)
            assert_grad(dW[torch.from_numpy(ids).cuda()].float().cpu().numpy(), dw_r, name="dW ids")
    gpu_properties(p, X, W, dX, dW, valid)
