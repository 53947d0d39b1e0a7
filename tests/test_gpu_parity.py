"""GPU parity: the CUDA path through the C-ABI against the fp64 oracle, element
by element, on the same seeded inputs.  Sizes span several tiles with ragged
tails in every dimension (rows vs 128-row tiles, vocabulary vs 256-wide tiles
and the backward's vocabulary chunks, hidden vs 64-wide K steps)."""
import math

import numpy as np
import pytest

import oracle
import synth
from helpers import assert_grad, assert_loss, assert_lse, to_device

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import lm_head_cross_gb300 as flce  # noqa: E402


def run(problem, **kw):
    X, W, y = to_device(problem)
    loss, lse, dX, dW, ws = flce.fwd_bwd(X, W, y, problem.ignore_index, problem.reduction, **kw)
    st = flce.read_device_status(ws)
    return dict(loss=float(loss.item()), lse=lse.cpu().numpy(), dX=dX.float().cpu().numpy(),
                dW=dW.float().cpu().numpy(), status=st)


def check_full(problem, rowchunk=False):
    got = run(problem, rowchunk=rowchunk)
    assert got["status"] == 0, flce.status_string(got["status"])
    ref = oracle.full_bf16(problem)
    assert_loss(got["loss"], ref["loss"])
    assert_lse(got["lse"], ref["lse"])
    assert_grad(got["dX"], ref["dX"], name="dX")
    assert_grad(got["dW"], ref["dW"], name="dW")
    valid = problem.labels != problem.ignore_index
    assert np.all(got["dX"][~valid] == 0.0), "ignored rows must give exactly zero dX"
    return got, ref


# the bounded path (flce_fwd_bwd: logits recomputed, V-independent workspace) and the
# row-chunk path (flce_fwd_bwd_rowchunk: logits computed once, a row chunk kept)
PATHS = pytest.mark.parametrize("rowchunk", [False, True], ids=["bounded", "rowchunk"])


@PATHS
def test_tiny_workload_full(rowchunk):
    check_full(synth.workload_problem(synth.TINY), rowchunk)


@pytest.mark.parametrize("n,h,v,red,labels", [
    (300, 136, 1000, "mean", "uniform"),      # ragged N, H (K tail), V
    (129, 64, 257, "sum", "zipf"),            # one row past a tile, one column past a tile
    (1, 8, 1, "mean", "uniform"),             # smallest shape; V = 1
    (77, 72, 2, "sum", "uniform"),            # V = 2
    (640, 256, 17000, "mean", "zipf"),        # three backward vocabulary chunks, ragged last chunk
    (1000, 520, 8200, "sum", "uniform"),      # chunk boundary + 8 past it; H not a tile multiple
    (1500, 128, 4001, "mean", "zipf"),        # fused path: two row chunks, the last one ragged; odd V
    (70, 64, 262147, "mean", "uniform"),      # 2^18 + 3 ids: 1025 vocabulary tiles, 33 backward chunks
])
@PATHS
def test_ragged_shapes(n, h, v, red, labels, rowchunk):
    p = synth.make_problem(n, h, v, seed=n + h + v, labels=labels, ignore_frac=0.1, reduction=red,
                           w_std=0.05)
    check_full(p, rowchunk)


@PATHS
def test_outlier_rows_sum_reduction(rowchunk):
    p = synth.make_problem(512, 256, 3000, seed=44, labels="zipf", ignore_frac=0.05, reduction="sum",
                           outlier_rows=16, outlier_scale=10.0)
    check_full(p, rowchunk)


def test_fused_and_recompute_paths_agree():
    p = synth.make_problem(2048, 256, 6000, seed=45, labels="zipf", ignore_frac=0.05)
    a = run(p, rowchunk=True)
    b = run(p)
    assert abs(a["loss"] - b["loss"]) <= 1e-4 * abs(b["loss"])
    assert np.abs(a["lse"] - b["lse"]).max() <= 1e-4
    assert_grad(a["dX"], b["dX"], frac=1e-2, name="dX")
    assert_grad(a["dW"], b["dW"], frac=1e-2, name="dW")


@PATHS
def test_all_rows_ignored_mean_gives_zero(rowchunk):
    p = synth.make_problem(200, 64, 500, seed=3, ignore_frac=1.0, reduction="mean")
    got = run(p, rowchunk=rowchunk)
    assert got["status"] == 0
    assert got["loss"] == 0.0
    assert np.all(got["dX"] == 0) and np.all(got["dW"] == 0)
    ref = oracle.full_bf16(p)
    assert_lse(got["lse"], ref["lse"])


@PATHS
def test_w_zero_closed_form(rowchunk):
    """W = 0: loss = ln V exactly in the definition; dX = 0; dW from its closed form."""
    p = synth.make_problem(384, 128, 3000, seed=5, ignore_frac=0.1)
    p.W[:] = 0
    got = run(p, rowchunk=rowchunk)
    assert abs(got["loss"] - math.log(3000)) <= 1e-3 * math.log(3000)
    assert np.all(got["dX"] == 0)
    X = oracle.widen_bf16(p.X)
    valid = p.labels != p.ignore_index
    nv = valid.sum()
    dW = np.tile(X[valid].sum(axis=0) / 3000, (3000, 1))
    for i in np.nonzero(valid)[0]:
        dW[p.labels[i]] -= X[i]
    assert_grad(got["dW"], dW / nv, name="dW")


@PATHS
def test_equal_rows_give_zero_dx_and_log_v(rowchunk):
    p = synth.make_problem(256, 128, 700, seed=6, ignore_frac=0.0)
    p.W[:] = p.W[3]
    got = run(p, rowchunk=rowchunk)
    assert abs(got["loss"] - math.log(700)) <= 1e-3 * math.log(700)
    # every softmax row is uniform: dX_i = s (mean_j W_j - W_{y_i}) = 0
    assert np.abs(got["dX"]).max() <= 1e-6


@PATHS
def test_dw_vocab_sum_is_zero(rowchunk):
    p = synth.make_problem(512, 256, 5000, seed=8, ignore_frac=0.05, reduction="sum")
    got = run(p, rowchunk=rowchunk)
    dW = got["dW"]
    # each row of G sums to zero, so the vocabulary sum of dW vanishes up to bf16 rounding of dW
    resid = np.abs(dW.astype(np.float64).sum(axis=0)).max()
    bound = 2 * 2.0 ** -8 * np.abs(dW.astype(np.float64)).sum(axis=0).max()
    assert resid <= bound, (resid, bound)


def test_label_out_of_range_sets_status():
    p = synth.make_problem(256, 64, 300, seed=9)
    p.labels[17] = 300
    X, W, y = to_device(p)
    _, _, _, _, ws = flce.fwd_bwd(X, W, y, p.ignore_index, p.reduction)
    assert flce.read_device_status(ws) == 5
    p.labels[17] = -5
    X, W, y = to_device(p)
    _, _, ws = flce.forward(X, W, y, p.ignore_index, p.reduction)
    assert flce.read_device_status(ws) == 5
    # a clean call clears the word
    p.labels[17] = 0
    X, W, y = to_device(p)
    _, _, ws = flce.forward(X, W, y, p.ignore_index, p.reduction, ws=ws)
    assert flce.read_device_status(ws) == 0


def test_separate_forward_backward_with_upstream_gradient():
    p = synth.make_problem(700, 192, 2500, seed=10, labels="zipf", ignore_frac=0.1, reduction="mean")
    X, W, y = to_device(p)
    loss, lse, ws = flce.forward(X, W, y, p.ignore_index, p.reduction)
    g = torch.tensor([0.37], dtype=torch.float32, device="cuda")
    dX, dW, _ = flce.backward(X, W, y, lse, g, p.ignore_index, p.reduction, ws=ws)
    assert flce.read_device_status(ws) == 0
    ref = oracle.full_bf16(p, grad_output=0.37)
    assert_loss(float(loss.item()), ref["loss"])
    assert_grad(dX.float().cpu().numpy(), ref["dX"], name="dX")
    assert_grad(dW.float().cpu().numpy(), ref["dW"], name="dW")


@pytest.mark.parametrize("upstream", [1.0, 2.5])
@PATHS
def test_autograd_wrapper(upstream, rowchunk):
    p = synth.make_problem(2 * 150, 128, 1500, seed=12, labels="zipf", ignore_frac=0.1)
    X, W, y = to_device(p)
    x3 = X.reshape(2, 150, 128).clone().requires_grad_(True)
    w = W.clone().requires_grad_(True)
    loss = flce.linear_cross_entropy(x3, w, y.reshape(2, 150).long(), rowchunk=rowchunk)
    (loss * upstream).backward()
    ref = oracle.full_bf16(p, grad_output=upstream)
    assert_loss(float(loss.item()), ref["loss"])
    assert_grad(x3.grad.reshape(300, 128).float().cpu().numpy(), ref["dX"], name="dX")
    assert_grad(w.grad.float().cpu().numpy(), ref["dW"], name="dW")
    with torch.no_grad():
        l2 = flce.linear_cross_entropy(X.reshape(2, 150, 128), W, y.reshape(2, 150).long())
    assert_loss(float(l2.item()), ref["loss"])


@PATHS
def test_repeat_calls_are_deterministic(rowchunk):
    p = synth.make_problem(512, 256, 9000, seed=13, ignore_frac=0.05)
    a = run(p, rowchunk=rowchunk)
    b = run(p, rowchunk=rowchunk)
    assert a["loss"] == b["loss"]
    assert np.array_equal(a["lse"], b["lse"])
    assert np.array_equal(a["dW"], b["dW"])


def test_timeout_path_returns_status():
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    L = flce.lib()
    import ctypes
    assert L.flce_selftest_timeout(ctypes.c_void_p(ws.data_ptr()), 1024, 20_000_000, None) == 0
    assert flce.read_device_status(ws) == 6
    # the context is still usable
    p = synth.make_problem(128, 64, 256, seed=1)
    got = run(p)
    assert got["status"] == 0


@PATHS
def test_reduction_none_fwd_bwd(rowchunk):
    """Per-row losses; the fused call's gradients are those of their sum."""
    p = synth.make_problem(600, 128, 3000, seed=61, labels="zipf", ignore_frac=0.1, reduction="none")
    X, W, y = to_device(p)
    loss, lse, dX, dW, ws = flce.fwd_bwd(X, W, y, p.ignore_index, "none", rowchunk=rowchunk)
    assert flce.read_device_status(ws) == 0
    ref = oracle.full_bf16(p)
    rows = loss.cpu().numpy()
    assert rows.shape == (600,)
    assert np.abs(rows - ref["loss"]).max() <= 2e-3 + 1e-3 * np.abs(ref["loss"]).max()
    valid = p.labels != p.ignore_index
    assert np.all(rows[~valid] == 0.0)
    assert_grad(dX.float().cpu().numpy(), ref["dX"], name="dX")
    assert_grad(dW.float().cpu().numpy(), ref["dW"], name="dW")


def test_reduction_none_backward_per_row_gradients():
    p = synth.make_problem(500, 136, 2200, seed=62, labels="uniform", ignore_frac=0.1, reduction="none")
    X, W, y = to_device(p)
    loss, lse, ws = flce.forward(X, W, y, p.ignore_index, "none")
    g = np.random.default_rng(5).standard_normal(500).astype(np.float32)
    dX, dW, _ = flce.backward(X, W, y, lse, torch.from_numpy(g).cuda(), p.ignore_index, "none", ws=ws)
    assert flce.read_device_status(ws) == 0
    ref = oracle.full_bf16(p, grad_output=g.astype(np.float64))
    assert_grad(dX.float().cpu().numpy(), ref["dX"], name="dX")
    assert_grad(dW.float().cpu().numpy(), ref["dW"], name="dW")


@PATHS
@pytest.mark.parametrize("red", ["mean", "sum"])
def test_shift_one(rowchunk, red):
    """Causal next-token shift inside the kernels: row i is scored against labels[i + 1]."""
    B, S = 3, 200
    p = synth.make_problem(B * S, 128, 2500, seed=63, labels="zipf", ignore_frac=0.05, reduction=red)
    X, W, y = to_device(p)
    loss, lse, dX, dW, ws = flce.fwd_bwd(X, W, y, p.ignore_index, red, rowchunk=rowchunk, shift=1, seq_len=S)
    assert flce.read_device_status(ws) == 0
    shifted = oracle.shift_labels(p.labels, S, p.ignore_index)
    ref = oracle.full(oracle.widen_bf16(p.X), oracle.widen_bf16(p.W), shifted, p.ignore_index, red)
    assert_loss(float(loss.item()), ref["loss"])
    assert_lse(lse.cpu().numpy(), ref["lse"])
    assert_grad(dX.float().cpu().numpy(), ref["dX"], name="dX")
    assert_grad(dW.float().cpu().numpy(), ref["dW"], name="dW")


def test_autograd_none_and_shift():
    B, S, H, V = 2, 160, 128, 1800
    p = synth.make_problem(B * S, H, V, seed=64, labels="zipf", ignore_frac=0.1)
    X, W, y = to_device(p)
    x3 = X.reshape(B, S, H).clone().requires_grad_(True)
    w = W.clone().requires_grad_(True)
    rows = flce.linear_cross_entropy(x3, w, y.reshape(B, S).long(), reduction="none", shift=1)
    assert rows.shape == (B, S)
    g = torch.linspace(0.5, 1.5, B * S, device="cuda").reshape(B, S)
    (rows * g).sum().backward()
    shifted = oracle.shift_labels(p.labels, S, p.ignore_index)
    ref = oracle.full(oracle.widen_bf16(p.X), oracle.widen_bf16(p.W), shifted, p.ignore_index, "none",
                      grad_output=g.reshape(-1).cpu().numpy().astype(np.float64))
    assert np.abs(rows.detach().reshape(-1).cpu().numpy() - ref["loss"]).max() <= 2e-3 + 1e-3 * np.abs(ref["loss"]).max()
    assert_grad(x3.grad.reshape(B * S, H).float().cpu().numpy(), ref["dX"], name="dX")
    assert_grad(w.grad.float().cpu().numpy(), ref["dW"], name="dW")


@pytest.mark.parametrize("red", ["mean", "sum"])
@PATHS
def test_wide_logit_range_rows(red, rowchunk):
    """Rows whose target logit lies far below the row's max (some tiles, or the
    whole row, stored relative to the tiles' own maxima) next to ordinary rows,
    over two row chunks.  The ordinary rows' dX is checked against its own
    scale, so the large rows cannot hide an error there."""
    p = synth.make_problem(1500, 128, 4001, seed=46, labels="uniform", ignore_frac=0.1, reduction=red,
                           w_std=0.05)
    xf = synth.bf16_bits_to_f32(p.X)
    group = np.arange(p.n) % 3           # 0: x1, 1: x16, 2: x64 (powers of two: exact in bf16)
    xf = xf * np.array([1.0, 16.0, 64.0], np.float32)[group][:, None]
    p.X = synth.f32_to_bf16_bits(xf)
    got, ref = check_full(p, rowchunk)
    for g in range(3):
        rows = group == g
        assert_grad(got["dX"][rows], ref["dX"][rows], name=f"dX rows x{[1, 16, 64][g]}")
    # the x64 rows do have logits spread far past the reference span
    z = xf[group == 2].astype(np.float64) @ synth.bf16_bits_to_f32(p.W).astype(np.float64).T
    assert (z.max(axis=1) - z.min(axis=1)).max() > 64 / math.log2(math.e)


def test_fwd_bwd_host_matches_device_call():
    """The host-memory entry point runs the same pass: results equal the device
    call's bit for bit, and its device status is read from the buffer's start."""
    p = synth.make_problem(700, 136, 3001, seed=47, labels="zipf", ignore_frac=0.1, w_std=0.05)
    a = run(p)
    X, W, y = to_device(p)
    xh, wh, yh = X.cpu().pin_memory(), W.cpu().pin_memory(), y.cpu().pin_memory()
    out = (torch.empty(1, dtype=torch.float32).pin_memory(), torch.empty(p.n, dtype=torch.float32).pin_memory(),
           torch.empty(xh.shape, dtype=torch.bfloat16).pin_memory(),
           torch.empty(wh.shape, dtype=torch.bfloat16).pin_memory())
    dev = torch.empty(flce.host_buffer_bytes(p.n, p.h, p.v), dtype=torch.uint8, device="cuda")
    flce.fwd_bwd_host(xh, wh, yh, out, dev, p.ignore_index, p.reduction)
    assert flce.read_device_status(dev) == 0
    torch.cuda.synchronize()
    assert float(out[0].item()) == a["loss"]
    assert np.array_equal(out[1].numpy(), a["lse"])
    assert np.array_equal(out[2].float().numpy(), a["dX"])
    assert np.array_equal(out[3].float().numpy(), a["dW"])
    with pytest.raises(flce.FlceError):
        flce.fwd_bwd_host(xh, wh, yh, out, dev[:1024], p.ignore_index, p.reduction)


def test_profile_mask_times_only_the_selected_kinds():
    """flce_profile_enable(mask): only launches of the selected kinds are bracketed."""
    p = synth.make_problem(600, 128, 3000, seed=48, labels="zipf", ignore_frac=0.05)
    X, W, y = to_device(p)
    flce.fwd_bwd(X, W, y, p.ignore_index, p.reduction)
    torch.cuda.synchronize()
    flce.profile_enable(True, kinds=["dxdw"])
    flce.fwd_bwd(X, W, y, p.ignore_index, p.reduction)
    only = flce.profile_read()
    flce.profile_enable(True)
    flce.fwd_bwd(X, W, y, p.ignore_index, p.reduction)
    every = flce.profile_read()
    flce.profile_enable(False)
    assert only["dxdw"][0] == every["dxdw"][0] > 0
    assert only["forward"][0] == only["small"][0] == 0
    assert every["forward"][0] > 0 and every["small"][0] > 0
    assert every["dxdw"][2] == pytest.approx(4.0 * p.n * p.h * p.v)   # the credited flops of the contraction


def test_fwd_bwd_host_on_copy_streams_pipelined():
    """Four pipelined calls on two device buffers with the copies on their own
    streams give every step the device call's results exactly."""
    p = synth.make_problem(520, 128, 2100, seed=49, labels="zipf", ignore_frac=0.05, w_std=0.05)
    a = run(p)
    X, W, y = to_device(p)
    xh, wh, yh = X.cpu().pin_memory(), W.cpu().pin_memory(), y.cpu().pin_memory()
    hb = flce.host_buffer_bytes(p.n, p.h, p.v)
    comp, cin, cout = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    slots = []
    for _ in range(2):
        outs = (torch.empty(1, dtype=torch.float32).pin_memory(), torch.empty(p.n, dtype=torch.float32).pin_memory(),
                torch.empty(xh.shape, dtype=torch.bfloat16).pin_memory(),
                torch.empty(wh.shape, dtype=torch.bfloat16).pin_memory())
        slots.append((outs, torch.empty(hb, dtype=torch.uint8, device="cuda"), torch.cuda.Event()))
    results = []
    for i in range(4):
        outs, buf, done = slots[i % 2]
        if i >= 2:
            cin.wait_event(done)
            cout.synchronize()
            results.append(tuple(t.clone() for t in outs))
        flce.fwd_bwd_host(xh, wh, yh, outs, buf, p.ignore_index, p.reduction, stream=comp, in_stream=cin,
                          out_stream=cout)
        done.record(cout)
    torch.cuda.synchronize()
    results += [tuple(t.clone() for t in slots[i % 2][0]) for i in (2, 3)]
    for loss, lse, dx, dw in results:
        assert float(loss.item()) == a["loss"]
        assert np.array_equal(lse.numpy(), a["lse"])
        assert np.array_equal(dx.float().numpy(), a["dX"])
        assert np.array_equal(dw.float().numpy(), a["dW"])


@pytest.mark.parametrize("red", ["mean", "sum", "none"])
def test_empty_batch(red):
    """n = 0: no valid row, so the loss is 0 (mean reads as n_valid = 0), dW = 0,
    and every per-row output is empty, on every entry point."""
    h, v = 64, 300
    g = torch.Generator().manual_seed(5)
    w = (torch.randn(v, h, generator=g) * 0.05).to(torch.bfloat16).cuda()
    x = torch.empty(0, h, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(0, dtype=torch.int32, device="cuda")
    dW = torch.full_like(w, 3.0)
    out = (torch.full((0 if red == "none" else 1,), 7.0, device="cuda"), torch.empty(0, device="cuda"),
           torch.empty_like(x), dW)
    loss, lse, dX, dW, ws = flce.fwd_bwd(x, w, y, -100, red, out=out)
    assert flce.read_device_status(ws) == 0
    assert lse.numel() == 0 and dX.numel() == 0
    assert torch.count_nonzero(dW).item() == 0
    if red != "none":
        assert float(loss.item()) == 0.0
    loss_f, lse_f, ws = flce.forward(x, w, y, -100, red)
    assert flce.read_device_status(ws) == 0 and lse_f.numel() == 0
    if red != "none":
        assert float(loss_f.item()) == 0.0
    gl = torch.empty(0, device="cuda") if red == "none" else torch.ones(1, device="cuda")
    dX_b, dW_b, ws = flce.backward(x, w, y, lse_f, gl, -100, red)
    assert flce.read_device_status(ws) == 0 and torch.count_nonzero(dW_b).item() == 0 and dX_b.numel() == 0
    idx, val, lse_t, ws = flce.topk(x, w, 4)
    assert flce.read_device_status(ws) == 0 and idx.shape == (0, 4) and val.shape == (0, 4)
    ti = torch.empty(0, 2, dtype=torch.int32, device="cuda")
    tq = torch.empty(0, 2, dtype=torch.float32, device="cuda")
    loss_s, _, _, dW_s, ws = flce.soft_fwd_bwd(x, w, ti, tq, red)
    assert flce.read_device_status(ws) == 0 and torch.count_nonzero(dW_s).item() == 0
    if red != "none":
        assert float(loss_s.item()) == 0.0
        xr = x.clone().requires_grad_(True)
        wr = w.clone().requires_grad_(True)
        l = flce.linear_cross_entropy(xr, wr, y.long(), reduction=red)
        l.backward()
        assert float(l.item()) == 0.0 and torch.count_nonzero(wr.grad).item() == 0
    # host-memory entry point
    hb = flce.host_buffer_bytes(0, h, v, -100, red)
    dev = torch.empty(hb, dtype=torch.uint8, device="cuda")
    outs = (torch.full((0 if red == "none" else 1,), 7.0).pin_memory(), torch.empty(0).pin_memory(),
            torch.empty(0, h, dtype=torch.bfloat16).pin_memory(), torch.full((v, h), 3.0, dtype=torch.bfloat16).pin_memory())
    flce.fwd_bwd_host(x.cpu(), w.cpu().pin_memory(), y.cpu(), outs, dev, -100, red)
    torch.cuda.synchronize()
    assert flce.read_device_status(dev) == 0 and torch.count_nonzero(outs[3]).item() == 0
    if red != "none":
        assert float(outs[0].item()) == 0.0


@PATHS
def test_row_tile_groups_and_wide_hidden(rowchunk):
    """Forward launches whose row tiles span several unit groups (H = 4096: 24 row
    tiles of 256 per group, 28 here, the last group short), and a wide hidden size."""
    p = synth.make_problem(7000, 4096, 1500, seed=31, labels="zipf", ignore_frac=0.05, reduction="sum",
                           x_std=4.0 / 64.0)
    check_full(p, rowchunk)
    X, W, y = to_device(p)
    loss, lse, ws = flce.forward(X, W, y, p.ignore_index, p.reduction)
    assert flce.read_device_status(ws) == 0
    f = oracle.forward(oracle.widen_bf16(p.X), oracle.widen_bf16(p.W), p.labels, p.ignore_index, p.reduction)
    assert_loss(float(loss.item()), f["loss"])
    assert_lse(lse.cpu().numpy(), f["lse"])
    q = synth.make_problem(600, 8192, 3000, seed=32, labels="uniform", ignore_frac=0.1, x_std=1.0 / 16)
    check_full(q, rowchunk)


def test_random_shapes_and_options():
    """48 seeded random problems (shapes, label mix, ignore fraction, reduction,
    shift, workspace size, logit scale) against the oracle, element by element."""
    rng = np.random.default_rng(2024)
    for case in range(48):
        seq = int(rng.integers(1, 5))
        s_len = int(rng.integers(1, 200))
        n = seq * s_len
        h = 8 * int(rng.integers(1, 80))
        v = int(rng.integers(1, 6000))
        red = ["mean", "sum", "none"][case % 3]
        shift = int(rng.integers(0, 2)) if s_len > 1 else 0
        rowchunk = bool(rng.integers(0, 2))
        p = synth.make_problem(n, h, v, seed=1000 + case, labels=["uniform", "zipf"][case % 2],
                               ignore_frac=float(rng.choice([0.0, 0.1, 0.5])), reduction=red,
                               x_std=float(rng.choice([0.25, 1.0, 4.0])), w_std=float(rng.choice([0.02, 0.1])))
        X, W, y = to_device(p)
        loss, lse, dX, dW, ws = flce.fwd_bwd(X, W, y, p.ignore_index, red, rowchunk=rowchunk, shift=shift,
                                             seq_len=s_len if shift else 0)
        assert flce.read_device_status(ws) == 0, case
        labels = oracle.shift_labels(p.labels, s_len, p.ignore_index) if shift else p.labels
        ref = oracle.full(oracle.widen_bf16(p.X), oracle.widen_bf16(p.W), labels, p.ignore_index, red)
        what = f"case {case}: n={n} h={h} v={v} {red} shift={shift} rowchunk={rowchunk}"
        got_loss = loss.cpu().numpy().astype(np.float64)
        if red == "none":
            np.testing.assert_allclose(got_loss, ref["loss"], rtol=1e-3, atol=2e-3, err_msg=what)
        else:
            assert abs(float(got_loss[0]) - ref["loss"]) <= 1e-3 * max(abs(ref["loss"]), 1e-6), what
        assert_lse(lse.cpu().numpy(), ref["lse"])
        if np.abs(ref["dX"]).max() > 0:
            assert_grad(dX.float().cpu().numpy(), ref["dX"], name="dX " + what)
            assert_grad(dW.float().cpu().numpy(), ref["dW"], name="dW " + what)
        else:
            assert not dX.float().abs().max().item() and not dW.float().abs().max().item(), what


def test_concurrent_calls_on_two_streams():
    """Two calls with their own workspaces on two streams at once give the same
    bits as the same calls one after the other (no state outside the workspace)."""
    p1 = synth.make_problem(1200, 256, 7000, seed=51, labels="zipf", ignore_frac=0.05)
    p2 = synth.make_problem(900, 192, 5001, seed=52, labels="uniform", ignore_frac=0.1, reduction="sum")
    a1, a2 = run(p1), run(p2)
    X1, W1, y1 = to_device(p1)
    X2, W2, y2 = to_device(p2)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    for _ in range(3):
        r1 = flce.fwd_bwd(X1, W1, y1, p1.ignore_index, p1.reduction, stream=s1)
        r2 = flce.fwd_bwd(X2, W2, y2, p2.ignore_index, p2.reduction, stream=s2)
        torch.cuda.synchronize()
        for r, a in ((r1, a1), (r2, a2)):
            assert flce.read_device_status(r[4]) == 0
            assert float(r[0].item()) == a["loss"]
            assert np.array_equal(r[1].cpu().numpy(), a["lse"])
            assert np.array_equal(r[2].float().cpu().numpy(), a["dX"])
            assert np.array_equal(r[3].float().cpu().numpy(), a["dW"])
