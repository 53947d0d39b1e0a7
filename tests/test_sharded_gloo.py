"""The exchange of the sharded loss (lm_head_cross_gb300.sharded), on gloo ranks on
the CPU: vocabulary split ("What-Each-Parallelism-Actually-Shards" §7.2), sequence
split (§7.3) and both at once (§4.1's [B, S/SP, V/TP]).  The per-rank steps run
on a stand-in written here in float64 numpy (the GPU tests check the CUDA steps
themselves against the oracle); what is checked is that the collectives put the
pieces together into exactly the whole problem's loss, lse, dX and dW, as the
fp64 oracle computes them on one process."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

IGN = -100


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _labels(labels, ignore_index, shift, seq_len):
    import oracle
    lab = labels.numpy().astype(np.int64)
    return oracle.shift_labels(lab, seq_len, ignore_index) if shift else lab


class Float64Ops:
    """The per-rank steps in float64 on CPU tensors: what the library's calls compute."""

    @staticmethod
    def shard_forward(x, w, labels, v_offset, v_total, ignore_index, shift, seq_len, ws=None):
        X, Wd = x.numpy(), w.numpy()
        y = _labels(labels, ignore_index, shift, seq_len)
        z = X @ Wd.T
        m = z.max(axis=1)
        lse = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
        own = (y != ignore_index) & (y >= v_offset) & (y < v_offset + w.shape[0])
        tgt = np.zeros(X.shape[0])
        tgt[own] = z[np.nonzero(own)[0], y[own] - v_offset]
        return torch.from_numpy(lse), torch.from_numpy(tgt), "ws"

    @staticmethod
    def shard_combine(lse_parts, tgt_parts, labels, v_total, h, ignore_index, shift, seq_len, ws=None):
        lp, tp = lse_parts.numpy(), tgt_parts.numpy()
        m = lp.max(axis=0)
        lse = m + np.log(np.exp(lp - m).sum(axis=0))
        z = tp.sum(axis=0)
        y = _labels(labels, ignore_index, shift, seq_len)
        valid = y != ignore_index
        return torch.tensor([np.where(valid, lse - z, 0.0).sum()]), torch.from_numpy(lse), ws

    @staticmethod
    def shard_backward(x, w, labels, lse, v_offset, v_total, scale, ignore_index, shift, seq_len, ws=None):
        X, Wd = x.numpy(), w.numpy()
        y = _labels(labels, ignore_index, shift, seq_len)
        valid = y != ignore_index
        G = np.exp(X @ Wd.T - lse.numpy()[:, None])
        own = valid & (y >= v_offset) & (y < v_offset + w.shape[0])
        G[np.nonzero(own)[0], y[own] - v_offset] -= 1.0
        G[~valid] = 0.0
        G *= float(scale.item())
        return torch.from_numpy(G @ Wd), torch.from_numpy(G.T @ X), ws

    @staticmethod
    def fwd_bwd(x, w, labels, ignore_index, shift, seq_len, ws=None):
        import oracle
        f = oracle.full(x.numpy(), w.numpy(), _labels(labels, ignore_index, shift, seq_len), ignore_index, "sum")
        return (torch.tensor([f["loss"]]), torch.from_numpy(f["lse"]), torch.from_numpy(f["dX"]),
                torch.from_numpy(f["dW"]), "ws")

    @staticmethod
    def valid_count(labels, v_total, ignore_index, shift, seq_len, ws=None):
        return torch.tensor([int((_labels(labels, ignore_index, shift, seq_len) != ignore_index).sum())],
                            dtype=torch.int32), ws

    @staticmethod
    def scale_grads(dX, dW, scale):
        dX.mul_(float(scale.item()))
        dW.mul_(float(scale.item()))

    @staticmethod
    def f32_to_bf16(t):
        return t.clone()


def _problem(n, h, v, seed, ignore_frac):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((n, h))
    W = rng.standard_normal((v, h)) * 0.3
    y = rng.integers(0, v, size=n)
    y[rng.permutation(n)[:int(round(ignore_frac * n))]] = IGN
    return X, W, y.astype(np.int32)


def _worker(rank, world, port, layout, reduction, shift, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import oracle
    from lm_head_cross_gb300 import sharded
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        n, h, v, seq_len = 96, 12, 701, 24
        X, W, y = _problem(n, h, v, 7, 0.2)
        vocab_parts, seq_parts = layout
        # rank = s * vocab_parts + t: sequence slice s, vocabulary shard t (uneven bounds)
        s, t = divmod(rank, vocab_parts)
        vb = [0, 300, v] if vocab_parts == 2 else [0, v]
        rb = [0, 40, n] if seq_parts == 2 else [0, n]
        vocab_groups = [dist.new_group([s_ * vocab_parts + t_ for t_ in range(vocab_parts)])
                        for s_ in range(seq_parts)]
        seq_groups = [dist.new_group([s_ * vocab_parts + t_ for s_ in range(seq_parts)])
                      for t_ in range(vocab_parts)]
        vg = vocab_groups[s] if vocab_parts > 1 else None
        sg = seq_groups[t] if seq_parts > 1 else None
        r0, r1, v0, v1 = rb[s], rb[s + 1], vb[t], vb[t + 1]
        loss, lse, dX, dW = sharded.sharded_cross_entropy(
            torch.from_numpy(X[r0:r1]), torch.from_numpy(W[v0:v1]), torch.from_numpy(y[r0:r1]), v_offset=v0,
            v_total=v, vocab_group=vg, seq_group=sg, ignore_index=IGN, reduction=reduction, shift=shift,
            seq_len=seq_len if shift else 0, ops=Float64Ops)
        lab = oracle.shift_labels(y, seq_len, IGN) if shift else y
        ref = oracle.full(X, W, lab, IGN, reduction)
        tol = 1e-6   # fp32 on the wire for dW of the sequence split
        assert abs(float(loss.item()) - ref["loss"]) <= 1e-6 * abs(ref["loss"]), (float(loss.item()), ref["loss"])
        np.testing.assert_allclose(lse.numpy(), ref["lse"][r0:r1], rtol=0, atol=1e-9)
        np.testing.assert_allclose(dX.numpy(), ref["dX"][r0:r1], rtol=0, atol=tol * np.abs(ref["dX"]).max())
        np.testing.assert_allclose(dW.numpy(), ref["dW"][v0:v1], rtol=0, atol=tol * np.abs(ref["dW"]).max())
        out[rank] = "ok"
    except Exception as e:  # noqa: BLE001 — reported to the parent
        out[rank] = f"{type(e).__name__}: {e}"
        raise
    finally:
        dist.destroy_process_group()


def _run(layout, reduction, shift):
    world = layout[0] * layout[1]
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    try:
        mp.spawn(_worker, args=(world, _free_port(), layout, reduction, shift, out), nprocs=world, join=True)
    finally:
        results = dict(out)
    assert results == {r: "ok" for r in range(world)}, results


@pytest.mark.parametrize("reduction", ["mean", "sum"])
@pytest.mark.parametrize("shift", [0, 1])
def test_vocab_split_two_ranks(reduction, shift):
    _run((2, 1), reduction, shift)


@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_sequence_split_two_ranks(reduction):
    _run((1, 2), reduction, 0)


def test_vocab_and_sequence_split_four_ranks():
    _run((2, 2), "mean", 0)


def test_shift_with_sequence_group_is_refused():
    from lm_head_cross_gb300 import sharded

    class G:  # a stand-in group of two ranks
        pass

    import unittest.mock as um
    with um.patch.object(sharded, "_world", lambda g: 2 if g is not None else 1):
        with pytest.raises(ValueError):
            sharded.sharded_cross_entropy(torch.zeros(4, 8), torch.zeros(5, 8), torch.zeros(4, dtype=torch.int32),
                                          seq_group=G(), shift=1, seq_len=4, ops=Float64Ops)
