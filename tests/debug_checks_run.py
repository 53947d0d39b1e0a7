"""Runs small problems on every entry point through the library named by
FLCE_LIB (the debug build, whose kernels check every computed index and TMA
coordinate before use) and checks each result against the fp64 oracle and each
status word for FLCE_OK.  Started in its own process by
tests/test_gpu_debug_checks.py, because a process loads the library once.
Prints "ok" on success."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import torch  # noqa: E402

import lm_head_cross_gb300 as flce  # noqa: E402
import oracle  # noqa: E402
import synth  # noqa: E402
from helpers import assert_grad, assert_loss, assert_lse, to_device  # noqa: E402


def main():
    assert flce.lib().flce_debug_checks() == 1, "FLCE_LIB is not the debug build"
    problems = [synth.workload_problem(synth.TINY),
                synth.make_problem(300, 136, 1000, seed=71, labels="zipf", ignore_frac=0.1, reduction="sum",
                                   w_std=0.05),
                synth.make_problem(1500, 128, 4001, seed=72, labels="uniform", ignore_frac=0.1, w_std=0.05)]
    for p in problems:
        ref = oracle.full_bf16(p)
        X, W, y = to_device(p)
        for rowchunk in (False, True):
            loss, lse, dX, dW, ws = flce.fwd_bwd(X, W, y, p.ignore_index, p.reduction, rowchunk=rowchunk)
            assert flce.read_device_status(ws) == 0, (p.n, rowchunk)
            assert_loss(float(loss.item()), ref["loss"])
            assert_lse(lse.cpu().numpy(), ref["lse"])
            assert_grad(dX.float().cpu().numpy(), ref["dX"], name="dX")
            assert_grad(dW.float().cpu().numpy(), ref["dW"], name="dW")
        rng = np.random.default_rng(p.n)
        sidx = rng.integers(0, p.v, size=(p.n, 4)).astype(np.int32)
        sq = rng.random((p.n, 4)).astype(np.float32)
        sq /= sq.sum(axis=1, keepdims=True)
        sref = oracle.soft_full(oracle.widen_bf16(p.X), oracle.widen_bf16(p.W), sidx, sq.astype(np.float64), "mean")
        for rowchunk in (False, True):
            loss, lse_s, dX, dW, ws = flce.soft_fwd_bwd(X, W, torch.from_numpy(sidx).cuda(), torch.from_numpy(sq).cuda(),
                                                        "mean", rowchunk=rowchunk)
            assert flce.read_device_status(ws) == 0, ("soft", p.n, rowchunk)
            assert_loss(float(loss.item()), sref["loss"])
            assert_grad(dX.float().cpu().numpy(), sref["dX"], name="soft dX")
            assert_grad(dW.float().cpu().numpy(), sref["dW"], name="soft dW")
        idx, val, lse_t, ws = flce.topk(X, W, 8)
        assert flce.read_device_status(ws) == 0
        oi, ov, _ = oracle.topk(oracle.widen_bf16(p.X), oracle.widen_bf16(p.W), 8)
        np.testing.assert_allclose(val.cpu().numpy(), ov, rtol=0, atol=2e-3)
        half = p.v // 2
        lp, tp, ws = flce.shard_forward(X, W[:half].contiguous(), y, 0, p.v, p.ignore_index)
        assert flce.read_device_status(ws) == 0
        dxp, dws, ws = flce.shard_backward(X, W[half:].contiguous(), y, lse, half, p.v, None, p.ignore_index,
                                           p.reduction)
        assert flce.read_device_status(ws) == 0
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    import ctypes
    assert flce.lib().flce_selftest_bounds(ctypes.c_void_p(ws.data_ptr()), 256, None) == 0
    assert flce.read_device_status(ws) == 10   # the check fired and recorded itself
    print("ok")


if __name__ == "__main__":
    main()
