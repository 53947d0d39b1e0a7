"""The vocabulary-shard calls on the GPU against the fp64 oracle.

One process stands in for the ranks of a vocabulary split
("What-Each-Parallelism-Actually-Shards" §7.2): W is cut into shards (uneven,
one of them a single row), each shard's forward runs on its own, the parts are
stacked as the all-gather would stack them, combined, and each shard's backward
runs with the global lse; the fp32 dX parts are summed as the all-reduce would
sum them.  The whole must equal the oracle on the unsplit problem, and each
shard's own (lse, target logit) must equal the oracle's on that shard.  A last
test runs lm_head_cross_gb300.sharded itself on two gloo processes that share
the GPU (host-staged collectives; no kernel waits on another process).
"""
import os
import socket

import numpy as np
import pytest

import oracle
import synth
from helpers import assert_grad, assert_loss, assert_lse, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import lm_head_cross_gb300 as flce  # noqa: E402


def run_shards(p, bounds, reduction, shift=0, seq_len=0, grad=None):
    X, W, y = to_device(p)
    kw = dict(ignore_index=p.ignore_index, shift=shift, seq_len=seq_len)
    parts = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        lp, tp, ws = flce.shard_forward(X, W[a:b].contiguous(), y, a, p.v, **kw)
        assert flce.read_device_status(ws) == 0
        parts.append((lp, tp))
    lse_parts = torch.stack([q[0] for q in parts]).contiguous()
    tgt_parts = torch.stack([q[1] for q in parts]).contiguous()
    loss, lse, ws = flce.shard_combine(lse_parts, tgt_parts, y, p.v, p.h, reduction=reduction, **kw)
    assert flce.read_device_status(ws) == 0
    dX32 = torch.zeros(p.n, p.h, dtype=torch.float32, device="cuda")
    dWs = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        dXp, dW, ws = flce.shard_backward(X, W[a:b].contiguous(), y, lse, a, p.v, grad, reduction=reduction, **kw)
        assert flce.read_device_status(ws) == 0
        dX32 += dXp
        dWs.append(dW)
    dX = flce.f32_to_bf16(dX32)
    return dict(loss=loss.cpu().numpy().astype(np.float64), lse=lse.cpu().numpy(), dX=dX.float().cpu().numpy(),
                dW=torch.cat(dWs).float().cpu().numpy(), lse_parts=lse_parts.cpu().numpy(),
                tgt_parts=tgt_parts.cpu().numpy())


@pytest.mark.parametrize("bounds_frac,reduction,shift", [
    ((0, 0.5, 1), "mean", 0),
    ((0, 0.13, None, 1), "sum", 0),          # None: a shard of one row
    ((0, 0.3, 0.31, 0.8, 1), "mean", 1),
    ((0, 0.6, 1), "none", 0),
])
def test_vocab_shards_match_oracle(bounds_frac, reduction, shift):
    p = synth.make_problem(600, 136, 3001, seed=61, labels="zipf", ignore_frac=0.1, reduction=reduction,
                           w_std=0.05)
    bounds = []
    for f in bounds_frac:
        bounds.append(bounds[-1] + 1 if f is None else int(round(f * p.v)))
    seq = 150 if shift else 0
    grad = None
    g_np = 1.0
    if reduction == "none":
        g_np = np.random.default_rng(3).standard_normal(p.n)
        grad = torch.from_numpy(g_np.astype(np.float32)).cuda()
    got = run_shards(p, bounds, reduction, shift, seq, grad)
    lab = oracle.shift_labels(p.labels, seq, p.ignore_index) if shift else p.labels
    Xd, Wd = oracle.widen_bf16(p.X), oracle.widen_bf16(p.W)
    ref = oracle.full(Xd, Wd, lab, p.ignore_index, reduction,
                      grad_output=g_np.astype(np.float32).astype(np.float64) if reduction == "none" else 1.0)
    if reduction == "none":
        np.testing.assert_allclose(got["loss"], ref["loss"], rtol=1e-3, atol=2e-3)
    else:
        assert_loss(float(got["loss"][0]), ref["loss"])
    assert_lse(got["lse"], ref["lse"])
    assert_grad(got["dX"], ref["dX"], name="dX")
    assert_grad(got["dW"], ref["dW"], name="dW")
    # each shard's own part: lse over its ids, the target logit where it holds the label
    for r, (a, b) in enumerate(zip(bounds[:-1], bounds[1:])):
        own = (lab != p.ignore_index) & (lab >= a) & (lab < b)
        local = np.where(own, lab - a, p.ignore_index)
        lse_r, tgt_r = oracle.lse_and_target(Xd, Wd[a:b], local, p.ignore_index)
        assert_lse(got["lse_parts"][r], lse_r)
        np.testing.assert_allclose(got["tgt_parts"][r], tgt_r, rtol=0, atol=2e-3)
        assert np.all(got["tgt_parts"][r][~own] == 0.0)


def test_vocab_shards_random_shapes():
    """12 seeded random problems (rows, hidden size, vocabulary, 2-5 uneven shards,
    reduction, shift, ignore fraction) through the shard calls against the oracle."""
    rng = np.random.default_rng(65)
    for case in range(12):
        seq = int(rng.integers(1, 4))
        s_len = int(rng.integers(2, 160))
        n = seq * s_len
        h = 8 * int(rng.integers(1, 40))
        v = int(rng.integers(8, 5000))
        parts = int(rng.integers(2, 6))
        cuts = np.sort(rng.choice(np.arange(1, v), size=min(parts - 1, v - 1), replace=False)).tolist()
        bounds = [0] + cuts + [v]
        red = ["mean", "sum"][case % 2]
        shift = int(rng.integers(0, 2))
        p = synth.make_problem(n, h, v, seed=2000 + case, labels=["uniform", "zipf"][case % 2],
                               ignore_frac=float(rng.choice([0.0, 0.1, 0.4])), reduction=red,
                               w_std=float(rng.choice([0.02, 0.1])))
        got = run_shards(p, bounds, red, shift, s_len if shift else 0)
        lab = oracle.shift_labels(p.labels, s_len, p.ignore_index) if shift else p.labels
        ref = oracle.full(oracle.widen_bf16(p.X), oracle.widen_bf16(p.W), lab, p.ignore_index, red)
        what = f"case {case}: n={n} h={h} v={v} bounds={bounds} {red} shift={shift}"
        assert abs(float(got["loss"][0]) - ref["loss"]) <= 1e-3 * max(abs(ref["loss"]), 1e-6), what
        assert_lse(got["lse"], ref["lse"])
        if np.abs(ref["dX"]).max() > 0:
            assert_grad(got["dX"], ref["dX"], name="dX " + what)
            assert_grad(got["dW"], ref["dW"], name="dW " + what)


def test_shard_label_out_of_range_sets_status():
    p = synth.make_problem(300, 64, 1000, seed=62)
    p.labels[7] = 1000
    X, W, y = to_device(p)
    _, _, ws = flce.shard_forward(X, W[:500].contiguous(), y, 0, p.v)
    assert flce.read_device_status(ws) == 5
    _, _, ws = flce.shard_forward(X, W[500:].contiguous(), y, 500, p.v)
    assert flce.read_device_status(ws) == 5


def test_valid_count_and_f32_to_bf16():
    p = synth.make_problem(1000, 64, 500, seed=63, ignore_frac=0.3)
    _, _, y = to_device(p)
    c, ws = flce.valid_count(y, p.v)
    assert flce.read_device_status(ws) == 0
    assert int(c.item()) == int((p.labels != p.ignore_index).sum())
    c, _ = flce.valid_count(y, p.v, shift=1, seq_len=100)
    assert int(c.item()) == int((oracle.shift_labels(p.labels, 100, p.ignore_index) != p.ignore_index).sum())
    g = torch.Generator(device="cuda").manual_seed(1)
    for count in (0, 1, 7, 8, 9, 1 << 20, (1 << 20) + 5):
        src = torch.randn(count, device="cuda", generator=g) * 100
        got = flce.f32_to_bf16(src)
        assert torch.equal(got.view(torch.int16), src.to(torch.bfloat16).view(torch.int16)), count


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    sys.path.insert(0, os.path.join(root, "tests"))
    import torch.distributed as dist
    import lm_head_cross_gb300 as f
    from helpers import to_device as dev
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        p = synth.make_problem(400, 128, 2001, seed=64, labels="zipf", ignore_frac=0.1, w_std=0.05)
        X, W, y = dev(p)
        bounds = [0, 900, p.v]
        a, b = bounds[rank], bounds[rank + 1]
        loss, lse, dX, dW = f.sharded_cross_entropy(X, W[a:b].contiguous(), y, v_offset=a, v_total=p.v,
                                                    vocab_group=dist.group.WORLD, check=True)
        torch.cuda.synchronize()
        ref = oracle.full_bf16(p)
        assert abs(float(loss.item()) - ref["loss"]) <= 1e-3 * abs(ref["loss"])
        assert np.abs(lse.cpu().numpy() - ref["lse"]).max() <= 2e-3
        scale_x = np.abs(ref["dX"]).max()
        assert np.abs(dX.float().cpu().numpy() - ref["dX"]).max() <= 2e-2 * scale_x
        scale_w = np.abs(ref["dW"]).max()
        assert np.abs(dW.float().cpu().numpy() - ref["dW"][a:b]).max() <= 2e-2 * scale_w
        out[rank] = "ok"
    except Exception as e:  # noqa: BLE001 — reported to the parent
        out[rank] = f"{type(e).__name__}: {e}"
        raise
    finally:
        dist.destroy_process_group()


def test_sharded_cross_entropy_two_processes_one_gpu():
    import torch.multiprocessing as mp
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    try:
        mp.spawn(_worker, args=(2, _free_port(), out), nprocs=2, join=True)
    finally:
        results = dict(out)
    assert results == {0: "ok", 1: "ok"}, results
