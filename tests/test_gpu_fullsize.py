"""Parity at the five workloads' full sizes, on both fwd_bwd paths (the bounded
one the benchmark times, and the row-chunk one), against the fp64 oracle.

The N 8192 x V 32000 workload is compared in full.  For the three large ones the
oracle's full forward (every row's lse, the loss) was computed once by
tests/golden/make_workload_golden.py and is loaded after checking that it
belongs to these exact input bytes; from it the oracle computes, here, dX on
1024 sampled rows (each needs only its own lse) and dW on sampled vocabulary
ids (each needs every row's lse): the ids include the most frequent labels,
both ends of the vocabulary and, for the 32K x 152K workload, outlier rows.
Properties that hold at any size are checked as well:

* sum_j dW_j = 0 (each row of G sums to zero over the vocabulary);
* X^T dX = dW^T W (both equal X^T G W), an H x H identity tying dW to dX;
* ignored rows have exactly zero dX.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_grad, assert_loss, assert_lse, golden_forward, to_device

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


def gpu_properties(X, W, dX, dW, valid):
    assert torch.count_nonzero(dX[torch.from_numpy(~valid).to(dX.device)]).item() == 0
    dWf = dW.float()
    resid = dWf.double().sum(0).abs().max().item()
    bound = 2 * 2.0 ** -8 * dWf.double().abs().sum(0).max().item()
    assert resid <= bound, ("vocab sum of dW", resid, bound)
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
    valid = p.labels != p.ignore_index
    s = oracle.grad_scale(int(valid.sum()), p.reduction)
    Xd = oracle.widen_bf16(p.X)
    Wd = oracle.widen_bf16(p.W)
    if name == synth.DEFAULT_WORKLOAD:
        ref = oracle.full(Xd, Wd, p.labels, p.ignore_index, p.reduction)
        rows, ids = np.arange(p.n), np.arange(p.v)
        want = dict(loss=ref["loss"], lse=ref["lse"], dx=ref["dX"], dw=ref["dW"])
    else:
        g = golden_forward(name, p)
        assert int(g["n_valid"]) == int(valid.sum())
        rows, ids = sample_rows(p, 1024, rng), sample_ids(p, 64, rng)
        want = dict(loss=float(g["loss"]), lse=g["lse"],
                    dx=oracle.backward_dx_rows(Xd, Wd, p.labels, rows, s, p.ignore_index, lse_rows=g["lse"][rows]),
                    dw=oracle.backward_dw_ids(Xd, Wd, p.labels, g["lse"], ids, s, p.ignore_index))
    del Xd, Wd
    X, W, y = to_device(p)
    rows_t, ids_t = torch.from_numpy(rows).cuda(), torch.from_numpy(ids).cuda()
    for rowchunk in (False, True):
        loss, lse, dX, dW, ws = flce.fwd_bwd(X, W, y, p.ignore_index, p.reduction, rowchunk=rowchunk)
        assert flce.read_device_status(ws) == 0, rowchunk
        del ws
        assert_loss(float(loss.item()), want["loss"])
        assert_lse(lse.cpu().numpy(), want["lse"])
        assert_grad(dX[rows_t].float().cpu().numpy(), want["dx"], name=f"dX rows (rowchunk={rowchunk})")
        assert_grad(dW[ids_t].float().cpu().numpy(), want["dw"], name=f"dW ids (rowchunk={rowchunk})")
        gpu_properties(X, W, dX, dW, valid)
        del loss, lse, dX, dW
        torch.cuda.empty_cache()


def test_largest_workload_extra_memory():
    """The 128K-token x 128K-vocabulary workload on the bounded path: the device
    memory allocated beyond inputs and outputs is the workspace alone, under 4 GB
    (the materialised logits would take 32 GiB in bf16)."""
    n, h, v = synth.workload_shape("n131072_h4096_v131072")
    ws_bytes = flce.workspace_bytes(n, h, v)
    assert ws_bytes < 4e9
    g = torch.Generator(device="cuda").manual_seed(3)
    X = (torch.randn(n, h, device="cuda", generator=g)).to(torch.bfloat16)
    W = (torch.randn(v, h, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
    y = torch.randint(0, v, (n,), device="cuda", generator=g, dtype=torch.int32)
    out = (torch.empty(1, device="cuda"), torch.empty(n, device="cuda"), torch.empty_like(X), torch.empty_like(W))
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    _, _, _, _, ws = flce.fwd_bwd(X, W, y, -100, "mean", out=out)
    assert flce.read_device_status(ws) == 0
    peak = torch.cuda.max_memory_allocated() - base
    # the caching allocator rounds sizes to 512 bytes and may hand out a cached block with up to
    # 1 MiB of unsplit slack per allocation (five per call)
    assert ws.numel() == ws_bytes and ws_bytes <= peak <= ws_bytes + (5 << 20) + 4096, (peak, ws_bytes)
