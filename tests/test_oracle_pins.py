"""Pins for the fp64 oracle: results fixed by mathematics, not by the oracle itself.

The pages print no loss or gradient value for this method, so every numeric
pin here is a closed form, an invariant, a special case that reduces to a
textbook formula, brute force, finite differences, or torch's own CPU
cross-entropy (the library routine the naive step of
"What-Each-Parallelism-Actually-Shards" §1.4 calls).  ``test_oracle_mutants``
plants plausible mistakes in a copy of the oracle and checks these pins catch
each one.
"""
import math
import types

import numpy as np
import pytest

import oracle
import synth

IGN = -100


def _rand_problem(rng, n, h, v, ignore_frac=0.25, x_std=1.0, w_std=0.5):
    X = rng.standard_normal((n, h)) * x_std
    W = rng.standard_normal((v, h)) * w_std
    y = rng.integers(0, v, size=n)
    k = int(round(ignore_frac * n))
    if k:
        y[rng.permutation(n)[:k]] = IGN
    return X, W, y


# ---------------------------------------------------------------- pins (reusable)

def pin_w_zero(orc):
    """W = 0: every logit is 0, so lse = ln V, loss = ln V (mean) / n_valid ln V (sum),
    dX = 0 and dW_j = s((1/V) sum_valid X_i - sum_{y_i = j} X_i)."""
    rng = np.random.default_rng(11)
    n, h, v = 9, 5, 7
    X, _, y = _rand_problem(rng, n, h, v)
    W = np.zeros((v, h))
    valid = y != IGN
    nv = int(valid.sum())
    for red in ("mean", "sum"):
        f = orc.full(X, W, y, IGN, red)
        s = 1.0 / nv if red == "mean" else 1.0
        want = math.log(v) if red == "mean" else nv * math.log(v)
        assert abs(f["loss"] - want) <= 1e-12 * max(1.0, abs(want))
        np.testing.assert_allclose(f["lse"], np.full(n, math.log(v)), rtol=0, atol=1e-13)
        assert np.all(f["dX"] == 0.0)
        dW = np.empty((v, h))
        for j in range(v):
            dW[j] = s * (X[valid].sum(axis=0) / v - X[y == j].sum(axis=0))
        np.testing.assert_allclose(f["dW"], dW, rtol=0, atol=1e-13)


def pin_equal_rows(orc):
    """All W rows equal to u: lse_i = x_i.u + ln V, loss = ln V, dX = 0."""
    rng = np.random.default_rng(12)
    n, h, v = 8, 6, 5
    X, _, y = _rand_problem(rng, n, h, v)
    u = rng.standard_normal(h)
    W = np.tile(u, (v, 1))
    f = orc.full(X, W, y, IGN, "mean")
    np.testing.assert_allclose(f["lse"], X @ u + math.log(v), rtol=0, atol=1e-12)
    assert abs(f["loss"] - math.log(v)) < 1e-12
    np.testing.assert_allclose(f["dX"], 0.0, atol=1e-14)


def pin_x_zero(orc):
    """X = 0: loss = ln V, dW = 0, dX_i = s (mean_j W_j - W_{y_i}) on valid rows, 0 otherwise."""
    rng = np.random.default_rng(13)
    n, h, v = 10, 4, 6
    _, W, y = _rand_problem(rng, n, h, v)
    X = np.zeros((n, h))
    valid = y != IGN
    nv = int(valid.sum())
    f = orc.full(X, W, y, IGN, "mean")
    assert abs(f["loss"] - math.log(v)) < 1e-12
    assert np.all(f["dW"] == 0.0)
    want = np.zeros((n, h))
    for i in range(n):
        if valid[i]:
            want[i] = (W.mean(axis=0) - W[y[i]]) / nv
    np.testing.assert_allclose(f["dX"], want, rtol=0, atol=1e-14)


def pin_dw_vocab_sum(orc):
    """Each row of G sums to zero over the vocabulary, so sum_j dW_j = 0."""
    rng = np.random.default_rng(14)
    X, W, y = _rand_problem(rng, 12, 7, 9)
    f = orc.full(X, W, y, IGN, "sum")
    assert np.abs(f["dW"].sum(axis=0)).max() < 1e-12 * max(1.0, np.abs(f["dW"]).max())


def pin_translation(orc):
    """Adding one vector u to every W row shifts each row's logits by x_i.u:
    loss, softmax and dX do not change."""
    rng = np.random.default_rng(15)
    X, W, y = _rand_problem(rng, 7, 5, 6)
    u = rng.standard_normal(5)
    a = orc.full(X, W, y, IGN, "mean")
    b = orc.full(X, W + u[None, :], y, IGN, "mean")
    assert abs(a["loss"] - b["loss"]) < 1e-12
    np.testing.assert_allclose(a["dX"], b["dX"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(b["lse"] - a["lse"], X @ u, rtol=0, atol=1e-12)


def pin_ignored_rows(orc):
    """Ignored rows: loss 0, dX row exactly 0, no dW contribution (equal to the
    problem with those rows removed, at the same scale)."""
    rng = np.random.default_rng(16)
    X, W, y = _rand_problem(rng, 11, 5, 6, ignore_frac=0.4)
    valid = y != IGN
    f = orc.full(X, W, y, IGN, "sum")
    assert np.all(f["dX"][~valid] == 0.0)
    assert np.all(f["loss_rows"][~valid] == 0.0)
    g = orc.full(X[valid], W, y[valid], IGN, "sum")
    np.testing.assert_allclose(f["dW"], g["dW"], rtol=0, atol=1e-13)
    assert abs(f["loss"] - g["loss"]) < 1e-12
    m = orc.full(X, W, y, IGN, "mean")
    assert abs(m["loss"] - g["loss"] / valid.sum()) < 1e-12


def pin_v1_v2(orc):
    """V = 1: loss 0 and zero gradients.  V = 2: the loss is the logistic loss
    softplus(z_other - z_label) and dX_i = sigma(z_o - z_l) (W_o - W_l)."""
    rng = np.random.default_rng(17)
    n, h = 6, 4
    X = rng.standard_normal((n, h))
    W1 = rng.standard_normal((1, h))
    f = orc.full(X, W1, np.zeros(n, dtype=np.int64), IGN, "mean")
    assert abs(f["loss"]) < 1e-15 and np.all(np.abs(f["dX"]) < 1e-15) and np.all(np.abs(f["dW"]) < 1e-15)
    W2 = rng.standard_normal((2, h))
    y = rng.integers(0, 2, size=n)
    f = orc.full(X, W2, y, IGN, "sum")
    loss = 0.0
    dX = np.zeros((n, h))
    for i in range(n):
        zl = float(X[i] @ W2[y[i]])
        zo = float(X[i] @ W2[1 - y[i]])
        loss += math.log1p(math.exp(zo - zl))
        sig = 1.0 / (1.0 + math.exp(-(zo - zl)))
        dX[i] = sig * (W2[1 - y[i]] - W2[y[i]])
    assert abs(f["loss"] - loss) < 1e-12
    np.testing.assert_allclose(f["dX"], dX, rtol=0, atol=1e-12)


def pin_bruteforce(orc):
    """V <= 8, every label enumerated for one row: sum_y exp(-loss(y)) = 1 and
    the loss is smallest at the largest logit."""
    rng = np.random.default_rng(18)
    for v in (2, 3, 5, 8):
        x = rng.standard_normal((1, 4))
        W = rng.standard_normal((v, 4))
        losses = [orc.full(x, W, np.array([y]), IGN, "sum")["loss"] for y in range(v)]
        assert abs(sum(math.exp(-l) for l in losses) - 1.0) < 1e-12
        z = [sum(x[0, k] * W[j, k] for k in range(4)) for j in range(v)]
        assert int(np.argmin(losses)) == int(np.argmax(z))


def pin_python_loops(orc):
    """Tiny case written out with scalar Python loops and math.exp/log only."""
    rng = np.random.default_rng(19)
    n, h, v = 5, 3, 4
    X, W, y = _rand_problem(rng, n, h, v, ignore_frac=0.2)
    total, nv = 0.0, 0
    lse_ref = []
    for i in range(n):
        z = [sum(X[i, k] * W[j, k] for k in range(h)) for j in range(v)]
        lse = math.log(sum(math.exp(t) for t in z))
        lse_ref.append(lse)
        if y[i] != IGN:
            total += lse - z[y[i]]
            nv += 1
    f = orc.full(X, W, y, IGN, "mean")
    assert abs(f["loss"] - total / nv) < 1e-12
    np.testing.assert_allclose(f["lse"], lse_ref, rtol=0, atol=1e-12)


def pin_finite_differences(orc):
    """Central differences of the fp64 loss agree with dX and dW."""
    rng = np.random.default_rng(20)
    for red in ("mean", "sum"):
        X, W, y = _rand_problem(rng, 4, 5, 6, ignore_frac=0.25)
        f = orc.full(X, W, y, IGN, red)
        eps = 1e-6

        def L(Xa, Wa):
            return orc.forward(Xa, Wa, y, IGN, red)["loss"]

        num_dX = np.zeros_like(X)
        for idx in np.ndindex(*X.shape):
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += eps
            Xm[idx] -= eps
            num_dX[idx] = (L(Xp, W) - L(Xm, W)) / (2 * eps)
        num_dW = np.zeros_like(W)
        for idx in np.ndindex(*W.shape):
            Wp, Wm = W.copy(), W.copy()
            Wp[idx] += eps
            Wm[idx] -= eps
            num_dW[idx] = (L(X, Wp) - L(X, Wm)) / (2 * eps)
        np.testing.assert_allclose(f["dX"], num_dX, rtol=1e-7, atol=1e-8)
        np.testing.assert_allclose(f["dW"], num_dW, rtol=1e-7, atol=1e-8)


def pin_torch(orc):
    """torch's CPU cross-entropy in float64 with autograd (the library routine of
    the naive step), both reductions, with ignored rows."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    rng = np.random.default_rng(21)
    for (n, h, v, red) in ((33, 16, 50, "mean"), (40, 8, 17, "sum")):
        X, W, y = _rand_problem(rng, n, h, v, ignore_frac=0.2, w_std=0.7)
        f = orc.full(X, W, y, IGN, red)
        tX = torch.tensor(X, dtype=torch.float64, requires_grad=True)
        tW = torch.tensor(W, dtype=torch.float64, requires_grad=True)
        loss = F.cross_entropy(tX @ tW.T, torch.tensor(y), ignore_index=IGN, reduction=red)
        loss.backward()
        assert abs(f["loss"] - loss.item()) < 1e-12 * max(1.0, abs(loss.item()))
        np.testing.assert_allclose(f["dX"], tX.grad.numpy(), rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(f["dW"], tW.grad.numpy(), rtol=1e-10, atol=1e-13)
        lse = torch.logsumexp(tX.detach() @ tW.detach().T, dim=1).numpy()
        np.testing.assert_allclose(f["lse"], lse, rtol=0, atol=1e-12)


def pin_subsets(orc):
    """The sampled-row and sampled-id entry points agree with the whole problem."""
    rng = np.random.default_rng(22)
    X, W, y = _rand_problem(rng, 20, 6, 13)
    f = orc.full(X, W, y, IGN, "mean")
    rows = np.array([0, 3, 7, 19])
    lse, tgt = orc.lse_and_target(X, W, y, IGN, rows)
    np.testing.assert_allclose(lse, f["lse"][rows], rtol=0, atol=1e-13)
    dx = orc.backward_dx_rows(X, W, y, rows, f["scale"], IGN)
    np.testing.assert_allclose(dx, f["dX"][rows], rtol=0, atol=1e-13)
    ids = np.array([1, 5, 12])
    dw = orc.backward_dw_ids(X, W, y, f["lse"], ids, f["scale"], IGN)
    np.testing.assert_allclose(dw, f["dW"][ids], rtol=0, atol=1e-13)


PINS = [pin_w_zero, pin_equal_rows, pin_x_zero, pin_dw_vocab_sum, pin_translation,
        pin_ignored_rows, pin_v1_v2, pin_bruteforce, pin_python_loops, pin_finite_differences,
        pin_torch, pin_subsets]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle)


def test_reduction_none_matches_torch():
    """Per-row losses and the gradient of sum_i g_i loss_i against torch's reduction='none'."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    rng = np.random.default_rng(31)
    X, W, y = _rand_problem(rng, 23, 9, 14, ignore_frac=0.2)
    g = rng.standard_normal(23)
    f = oracle.full(X, W, y, IGN, "none", grad_output=g)
    tX = torch.tensor(X, requires_grad=True)
    tW = torch.tensor(W, requires_grad=True)
    rows = F.cross_entropy(tX @ tW.T, torch.tensor(y), ignore_index=IGN, reduction="none")
    (rows * torch.tensor(g)).sum().backward()
    np.testing.assert_allclose(f["loss"], rows.detach().numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(f["dX"], tX.grad.numpy(), rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(f["dW"], tW.grad.numpy(), rtol=1e-10, atol=1e-13)


def test_shift_matches_causal_lm_loss():
    """shift=1 on flattened [B, S] rows equals the usual causal-LM loss: logits of
    positions 0..S-2 against labels of positions 1..S-1 (torch, float64)."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    rng = np.random.default_rng(32)
    B, S, H, V = 3, 7, 6, 11
    X = rng.standard_normal((B * S, H))
    W = rng.standard_normal((V, H)) * 0.5
    lab = rng.integers(0, V, size=(B, S))
    lab[0, 3] = IGN
    y = oracle.shift_labels(lab, S, IGN)
    assert list(y[:S]) == list(lab[0, 1:]) + [IGN]
    f = oracle.full(X, W, y, IGN, "mean")
    tX = torch.tensor(X.reshape(B, S, H), requires_grad=True)
    tW = torch.tensor(W, requires_grad=True)
    logits = tX @ tW.T
    loss = F.cross_entropy(logits[:, :-1].reshape(-1, V), torch.tensor(lab[:, 1:]).reshape(-1), ignore_index=IGN)
    loss.backward()
    assert abs(f["loss"] - loss.item()) < 1e-12
    np.testing.assert_allclose(f["dX"], tX.grad.numpy().reshape(B * S, H), rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(f["dW"], tW.grad.numpy(), rtol=1e-10, atol=1e-13)


def test_soft_targets_k1_equals_hard_labels():
    """One target id with probability 1 per row is the hard-label cross-entropy."""
    rng = np.random.default_rng(33)
    X, W, y = _rand_problem(rng, 19, 6, 13, ignore_frac=0.0)
    for red in ("mean", "sum"):
        a = oracle.full(X, W, y, IGN, red)
        b = oracle.soft_full(X, W, y[:, None], np.ones((19, 1)), red)
        assert abs(a["loss"] - b["loss"]) < 1e-12
        np.testing.assert_allclose(a["dX"], b["dX"], rtol=0, atol=1e-13)
        np.testing.assert_allclose(a["dW"], b["dW"], rtol=0, atol=1e-13)


def test_soft_targets_match_torch_kl_div():
    """Sparse soft targets against torch's KL divergence on dense targets (float64, autograd);
    a row with no positive mass contributes nothing."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    rng = np.random.default_rng(34)
    n, h, v, k = 17, 8, 21, 5
    X, W, _ = _rand_problem(rng, n, h, v, ignore_frac=0.0)
    idx = np.stack([rng.permutation(v)[:k] for _ in range(n)])
    q = rng.random((n, k))
    q[:, -1] = 0.0
    q /= q.sum(axis=1, keepdims=True)
    q[3] = 0.0                                    # no mass: ignored
    dense = np.zeros((n, v))
    np.put_along_axis(dense, idx, q, axis=1)
    f = oracle.soft_full(X, W, idx, q, "mean")
    tX = torch.tensor(X, requires_grad=True)
    tW = torch.tensor(W, requires_grad=True)
    logp = F.log_softmax(tX @ tW.T, dim=1)
    total = F.kl_div(logp, torch.tensor(dense), reduction="sum")
    (total / (n - 1)).backward()
    assert abs(f["loss"] - total.item() / (n - 1)) < 1e-12
    np.testing.assert_allclose(f["dX"], tX.grad.numpy(), rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(f["dW"], tW.grad.numpy(), rtol=1e-10, atol=1e-13)
    assert np.all(f["dX"][3] == 0.0) and f["n_valid"] == n - 1


def test_topk_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(35)
    X, W, _ = _rand_problem(rng, 12, 7, 40, ignore_frac=0.0)
    idx, val, lse = oracle.topk(X, W, 6)
    z = torch.tensor(X) @ torch.tensor(W).T
    tv, ti = torch.topk(z, 6, dim=1)
    np.testing.assert_allclose(val, tv.numpy(), rtol=0, atol=1e-13)
    assert np.array_equal(idx, ti.numpy())
    np.testing.assert_allclose(lse, torch.logsumexp(z, dim=1).numpy(), rtol=0, atol=1e-12)
    assert np.array_equal(oracle.topk(X, W, 1)[0][:, 0], np.argmax(X @ W.T, axis=1))


def _multi_block_pin(orc, monkeypatch):
    """Row blocking (the large workloads run through hundreds of blocks): with ten rows
    per block, 103 rows make eleven blocks, the last one ragged (3 rows).  Every row's
    lse and target logit, the loss, the top-k and a row subset must equal torch's fp64
    logsumexp / gather / cross_entropy / topk on the whole problem."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    rng = np.random.default_rng(36)
    n, h, v = 103, 16, 37
    X, W, y = _rand_problem(rng, n, h, v, ignore_frac=0.2, w_std=1.0)
    monkeypatch.setattr(orc, "_BLOCK_BYTES", 8 * v * 10)
    z = torch.tensor(X) @ torch.tensor(W).T
    want_lse = torch.logsumexp(z, dim=1).numpy()
    valid = y != IGN
    want_tgt = np.where(valid, z.numpy()[np.arange(n), np.where(valid, y, 0)], 0.0)
    lse, tgt = orc.lse_and_target(X, W, y, IGN)
    np.testing.assert_allclose(lse, want_lse, rtol=0, atol=1e-12)
    np.testing.assert_allclose(tgt, want_tgt, rtol=0, atol=1e-12)
    rows = rng.permutation(n)[:47]
    lse_r, tgt_r = orc.lse_and_target(X, W, y, IGN, rows)
    np.testing.assert_allclose(lse_r, want_lse[rows], rtol=0, atol=1e-12)
    np.testing.assert_allclose(tgt_r, want_tgt[rows], rtol=0, atol=1e-12)
    f = orc.forward(X, W, y, IGN, "mean")
    ref = F.cross_entropy(z, torch.tensor(y.astype(np.int64)), ignore_index=IGN).item()
    assert abs(f["loss"] - ref) <= 1e-12 * abs(ref)
    idx, val, lse_k = orc.topk(X, W, 5)
    tv, ti = torch.topk(z, 5, dim=1)
    assert np.array_equal(idx, ti.numpy())
    np.testing.assert_allclose(val, tv.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_k, want_lse, rtol=0, atol=1e-12)


def test_multi_block_rows_match_torch(monkeypatch):
    assert [b.size for b in _blocks_with(monkeypatch, 103, 37, 10)] == [10] * 10 + [3]
    _multi_block_pin(oracle, monkeypatch)


def _blocks_with(monkeypatch, n, v, rows_per_block):
    monkeypatch.setattr(oracle, "_BLOCK_BYTES", 8 * v * rows_per_block)
    return list(oracle._row_blocks(n, v))


def _drop_ragged_block(n, v):
    step = max(1, oracle._BLOCK_BYTES // max(1, 8 * v))
    for s in range(0, n - n % step, step):
        yield np.arange(s, s + step)


def _end_off_by_one(n, v):
    step = max(1, oracle._BLOCK_BYTES // max(1, 8 * v))
    for s in range(0, n, step):
        yield np.arange(s, min(n - 1, s + step))


@pytest.mark.parametrize("bad", [_drop_ragged_block, _end_off_by_one], ids=["ragged tail dropped", "last row dropped"])
def test_multi_block_pin_catches_blocking_mistakes(monkeypatch, bad):
    """A row-blocking mistake planted in the oracle fails the multi-block pin."""
    monkeypatch.setattr(oracle, "_row_blocks", bad)
    with pytest.raises(AssertionError):
        _multi_block_pin(oracle, monkeypatch)


def test_mean_with_no_valid_row():
    """Reading taken where the pages are silent: no valid row under mean gives 0, not NaN."""
    rng = np.random.default_rng(23)
    X, W, _ = _rand_problem(rng, 4, 3, 5)
    f = oracle.full(X, W, np.full(4, IGN), IGN, "mean")
    assert f["loss"] == 0.0 and np.all(f["dX"] == 0) and np.all(f["dW"] == 0)


def test_label_out_of_range_is_an_error():
    rng = np.random.default_rng(24)
    X, W, y = _rand_problem(rng, 4, 3, 5)
    for bad in (5, -1, 1 << 30):
        yb = y.copy()
        yb[1] = bad
        with pytest.raises(ValueError):
            oracle.forward(X, W, yb, IGN, "mean")


def test_widen_bf16_exact():
    b = np.array([0x0000, 0x3F80, 0xBF80, 0x4049, 0x0001, 0x7F7F], dtype=np.uint16)
    want = np.array([0.0, 1.0, -1.0, 3.140625, 2.0 ** -133, 3.3895313892515355e38])
    np.testing.assert_array_equal(oracle.widen_bf16(b), want)


def test_synth_rounding_and_recipe():
    """The generator's bf16 rounding is nearest-even and its counts follow the recipe."""
    a = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e-39], dtype=np.float32)
    bits = synth.f32_to_bf16_bits(a)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: goes to the even mantissa (1.0)
    # 1 + 3*2^-8 is a tie between 1 + 2^-7 and 1 + 2^-6: goes to even (1 + 2^-6)
    np.testing.assert_array_equal(synth.bf16_bits_to_f32(bits)[:4],
                                  np.array([1.0, 1.0, 1.015625, -2.5], dtype=np.float32))
    p = synth.workload_problem(synth.TINY)
    assert p.X.shape == (256, 128) and p.W.shape == (1024, 128)
    assert int((p.labels == IGN).sum()) == 26
    assert p.labels[p.labels != IGN].min() >= 0 and p.labels.max() < 1024
    q = synth.workload_problem(synth.TINY)
    assert np.array_equal(p.X, q.X) and np.array_equal(p.W, q.W) and np.array_equal(p.labels, q.labels)
    z = synth.make_problem(4000, 8, 100, seed=5, labels="zipf", ignore_frac=0.05)
    lab = z.labels[z.labels != IGN]
    counts = np.bincount(lab, minlength=100)
    assert counts[0] > counts[1] > counts[5] and int((z.labels == IGN).sum()) == 200
    o = synth.make_problem(64, 8, 300, seed=6, outlier_rows=10)
    Wf = synth.bf16_bits_to_f32(o.W)
    norms = np.linalg.norm(Wf, axis=1)
    assert set(np.argsort(norms)[-10:]) == set(o.outlier_ids.tolist())


def test_oracle_full_on_tiny_workload_matches_torch():
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    p = synth.workload_problem(synth.TINY)
    f = oracle.full_bf16(p)
    X = torch.tensor(oracle.widen_bf16(p.X), requires_grad=True)
    W = torch.tensor(oracle.widen_bf16(p.W), requires_grad=True)
    loss = F.cross_entropy(X @ W.T, torch.tensor(p.labels.astype(np.int64)), ignore_index=IGN)
    loss.backward()
    assert abs(f["loss"] - loss.item()) < 1e-12
    np.testing.assert_allclose(f["dX"], X.grad.numpy(), rtol=1e-9, atol=1e-15)
    np.testing.assert_allclose(f["dW"], W.grad.numpy(), rtol=1e-9, atol=1e-15)


def test_oracle_full_on_workload_8k_32k_matches_torch():
    """The library special case at a benchmark size: the first 2500 rows of the
    N 8192 x V 32000 workload (three row blocks of the oracle, the last one
    ragged) against torch's fp64 cross_entropy and autograd on the CPU."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    p = synth.workload_problem(synth.DEFAULT_WORKLOAD)
    rows = 2500
    X = oracle.widen_bf16(p.X[:rows])
    W = oracle.widen_bf16(p.W)
    lab = p.labels[:rows]
    blocks = list(oracle._row_blocks(rows, p.v))
    assert len(blocks) == 3 and blocks[-1].size < blocks[0].size
    f = oracle.full(X, W, lab, p.ignore_index, p.reduction)
    Xt = torch.tensor(X, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    z = Xt @ Wt.T
    loss = F.cross_entropy(z, torch.tensor(lab.astype(np.int64)), ignore_index=p.ignore_index)
    loss.backward()
    assert abs(f["loss"] - loss.item()) <= 1e-12 * abs(loss.item())
    np.testing.assert_allclose(f["lse"], torch.logsumexp(z.detach(), dim=1).numpy(), rtol=0, atol=1e-10)
    np.testing.assert_allclose(f["dX"], Xt.grad.numpy(), rtol=0, atol=1e-12 * np.abs(Xt.grad.numpy()).max())
    np.testing.assert_allclose(f["dW"], Wt.grad.numpy(), rtol=0, atol=1e-12 * np.abs(Wt.grad.numpy()).max())


# ---------------------------------------------------------------- planted mistakes

def _mutant(**overrides):
    ns = types.SimpleNamespace(**{k: getattr(oracle, k) for k in dir(oracle) if not k.startswith("__")})
    for k, fn in overrides.items():
        setattr(ns, k, fn)
    # rebind 'full' and 'forward' so they call the overridden pieces
    def forward(X, W, labels, ignore_index=-100, reduction="mean"):
        lse, tgt = ns.lse_and_target(X, W, labels, ignore_index)
        valid = oracle.valid_rows(labels, ignore_index)
        if not oracle.labels_in_range(labels, np.shape(W)[0], ignore_index):
            raise ValueError("label out of range")
        loss_rows = np.where(valid, lse - tgt, 0.0)
        nv = int(valid.sum())
        total = float(loss_rows.sum())
        loss = ns.reduce(total, nv, reduction)
        return dict(loss=loss, lse=lse, loss_rows=loss_rows, n_valid=nv)

    def full(X, W, labels, ignore_index=-100, reduction="mean", grad_output=1.0):
        X = np.asarray(X, np.float64)
        W = np.asarray(W, np.float64)
        f = forward(X, W, labels, ignore_index, reduction)
        s = ns.grad_scale(f["n_valid"], reduction, grad_output)
        G = ns.grad_logits_rows(X, W, labels, np.arange(X.shape[0]), f["lse"], s, ignore_index)
        f["dX"] = ns.dx_from_g(G, X, W)
        f["dW"] = ns.dw_from_g(G, X, W)
        f["scale"] = s
        return f

    if not hasattr(ns, "reduce"):
        ns.reduce = lambda total, nv, red: (0.0 if nv == 0 else total / nv) if red == "mean" else total
    if not hasattr(ns, "dx_from_g"):
        ns.dx_from_g = lambda G, X, W: G @ W
    if not hasattr(ns, "dw_from_g"):
        ns.dw_from_g = lambda G, X, W: G.T @ X
    ns.forward = forward
    ns.full = full
    return ns


def _bad_grad_sign(X, W, labels, rows, lse_rows, scale, ignore_index=-100):
    return -oracle.grad_logits_rows(X, W, labels, rows, lse_rows, scale, ignore_index)


def _bad_grad_no_onehot(X, W, labels, rows, lse_rows, scale, ignore_index=-100):
    X = np.asarray(X, np.float64)
    z = X[np.asarray(rows)] @ np.asarray(W, np.float64).T
    p = np.exp(z - np.asarray(lse_rows)[:, None])
    p[np.asarray(labels)[np.asarray(rows)] == ignore_index] = 0.0
    return scale * p


def _bad_grad_no_mask(X, W, labels, rows, lse_rows, scale, ignore_index=-100):
    X = np.asarray(X, np.float64)
    lab = np.asarray(labels, dtype=np.int64)[np.asarray(rows)]
    z = X[np.asarray(rows)] @ np.asarray(W, np.float64).T
    p = np.exp(z - np.asarray(lse_rows)[:, None])
    ok = lab != ignore_index
    p[np.nonzero(ok)[0], lab[ok]] -= 1.0
    return scale * p


def _bad_lse_no_max(X, W, labels, ignore_index, rows=None):
    lse, tgt = oracle.lse_and_target(X, W, labels, ignore_index, rows)
    X = np.asarray(X, np.float64)
    r = np.arange(X.shape[0]) if rows is None else np.asarray(rows)
    m = (X[r] @ np.asarray(W, np.float64).T).max(axis=1)
    return lse - m, tgt


MUTANTS = {
    "grad sign flipped": dict(grad_logits_rows=_bad_grad_sign),
    "onehot term dropped": dict(grad_logits_rows=_bad_grad_no_onehot),
    "ignored rows not masked in G": dict(grad_logits_rows=_bad_grad_no_mask),
    "max dropped from lse": dict(lse_and_target=_bad_lse_no_max),
    "mean over all rows": dict(reduce=lambda t, nv, red: t / 9.0 if red == "mean" else t,
                              grad_scale=lambda nv, red, g=1.0: g / 9.0 if red == "mean" else g),
    "dW transposed operand": dict(dw_from_g=lambda G, X, W: (G.T @ X)[::-1]),
    "dX with a wrong vocab index": dict(dx_from_g=lambda G, X, W: G @ W[::-1]),
    "sum scale 1/n": dict(grad_scale=lambda nv, red, g=1.0: (0.0 if nv == 0 else g / nv)),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_oracle_mutants(name):
    """Each planted mistake must fail at least one pin."""
    orc = _mutant(**MUTANTS[name])
    caught = []
    for pin in PINS:
        if pin in (pin_subsets,):
            continue
        try:
            pin(orc)
        except AssertionError:
            caught.append(pin.__name__)
        except (ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"mutant '{name}' passed every pin"


def test_unmutated_copy_passes_every_pin():
    orc = _mutant()
    for pin in PINS:
        if pin in (pin_subsets,):
            continue
        pin(orc)
