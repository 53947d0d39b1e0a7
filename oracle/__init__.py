"""fp64 CPU oracle for the fused LM-head projection + cross-entropy.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
(``cpu_baseline`` / ``--impl reference``) may use it.  It shares no code with
the CUDA library; both are fed from the seeded generators in ``synth``.

What it computes is the plain definition the fused method must reproduce.
"What-Each-Parallelism-Actually-Shards" §1.4 prints the naive step: project the
hidden states with the LM head into ``[B,S,V]`` logits, upcast, and take
``F.cross_entropy`` over the flattened rows; §7.4 passes ``ignore_index=-100`` to
the fused call and says the fused operator keeps the same autograd semantics
while never storing the logits.  So, for rows ``i`` and vocabulary ids ``j``:

* logits ``z[i, j] = sum_h X[i, h] W[j, h]``  (W is ``[V, H]``, as in §7.4's call)
* ``lse[i] = log sum_j exp(z[i, j])``, evaluated as ``m + log sum exp(z - m)``
  with ``m = max_j z[i, j]`` (the same number, written to avoid overflow)
* ``loss_i = (lse[i] - z[i, y_i]) * valid_i``, ``valid_i = [y_i != ignore_index]``
* ``loss = sum_i loss_i / n_valid`` (``mean``) or ``sum_i loss_i`` (``sum``)
* the gradient of ``g * loss``: ``G = s * (softmax(z) - onehot(y)) * valid`` with
  ``s = g / n_valid`` (mean) or ``g`` (sum); ``dX = G W``, ``dW = G^T X``.

Readings where the pages are silent: under ``mean`` with no valid row the loss
is 0 and both gradients are 0; ``lse`` is reported for ignored rows too; a label
that is neither ``ignore_index`` nor in ``[0, V)`` is an error.  ``none``
returns the per-row losses, and the gradient then takes one upstream value per
row.  §7.4's call passes ``shift=1`` (causal next-token shift): position t of a
sequence is scored against the token at t + 1, and the last position has no
target; ``shift_labels`` writes that out.

Everything is float64.  bf16 inputs widen exactly.  Matrix products use numpy's
``matmul`` (a library primitive); rows are processed in blocks only to bound
memory, each row's arithmetic happening wholly inside one block.
"""
from __future__ import annotations

import numpy as np

_BLOCK_BYTES = 256 << 20   # cap on one block of fp64 logits


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exact."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def labels_in_range(labels: np.ndarray, v: int, ignore_index: int) -> bool:
    """True when every label is ``ignore_index`` or an id in ``[0, V)``."""
    lab = np.asarray(labels, dtype=np.int64)
    ok = (lab == ignore_index) | ((lab >= 0) & (lab < v))
    return bool(ok.all())


def valid_rows(labels: np.ndarray, ignore_index: int) -> np.ndarray:
    return np.asarray(labels, dtype=np.int64) != ignore_index


def shift_labels(labels: np.ndarray, seq_len: int, ignore_index: int) -> np.ndarray:
    """Next-token targets: row i of a flattened [B, S] batch takes labels[i + 1];
    the last position of each sequence gets ``ignore_index``."""
    lab = np.asarray(labels).reshape(-1, seq_len)
    out = np.full_like(lab, ignore_index)
    out[:, :-1] = lab[:, 1:]
    return out.reshape(-1)


def grad_scale(n_valid: int, reduction: str, grad_output=1.0):
    """``s``: d(loss)/d(loss_i) times the upstream gradient (per row for ``none``)."""
    if reduction == "mean":
        return 0.0 if n_valid == 0 else grad_output / n_valid
    if reduction in ("sum", "none"):
        return grad_output
    raise ValueError(reduction)


def _row_blocks(n: int, v: int):
    step = max(1, _BLOCK_BYTES // max(1, 8 * v))
    for s in range(0, n, step):
        yield np.arange(s, min(n, s + step))


def lse_and_target(X: np.ndarray, W: np.ndarray, labels: np.ndarray, ignore_index: int,
                   rows: np.ndarray | None = None):
    """Per-row ``lse`` and target logit ``z[i, y_i]`` (0 for ignored rows).

    ``rows`` selects a subset; each selected row is computed on its own terms.
    """
    X = np.asarray(X, np.float64)
    W = np.asarray(W, np.float64)
    lab = np.asarray(labels, dtype=np.int64)
    rows = np.arange(X.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    v = W.shape[0]
    lse = np.full(rows.size, np.nan)       # a row no block reaches stays NaN
    tgt = np.zeros(rows.size, np.float64)
    for blk in _row_blocks(rows.size, v):
        r = rows[blk]
        z = X[r] @ W.T
        m = z.max(axis=1)
        lse[blk] = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
        y = lab[r]
        ok = y != ignore_index
        tgt[blk[ok]] = z[np.nonzero(ok)[0], y[ok]]
    return lse, tgt


def forward(X, W, labels, ignore_index: int = -100, reduction: str = "mean"):
    """Loss, per-row lse, per-row loss and the valid count over all rows."""
    if not labels_in_range(labels, np.shape(W)[0], ignore_index):
        raise ValueError("label out of range")
    lse, tgt = lse_and_target(X, W, labels, ignore_index)
    valid = valid_rows(labels, ignore_index)
    loss_rows = np.where(valid, lse - tgt, 0.0)
    n_valid = int(valid.sum())
    total = float(np.sum(loss_rows))
    if reduction == "mean":
        loss = 0.0 if n_valid == 0 else total / n_valid
    elif reduction == "sum":
        loss = total
    elif reduction == "none":
        loss = loss_rows.copy()
    else:
        raise ValueError(reduction)
    return dict(loss=loss, lse=lse, loss_rows=loss_rows, n_valid=n_valid)


def grad_logits_rows(X, W, labels, rows, lse_rows, scale, ignore_index: int = -100):
    """``G[rows, :] = s * (exp(z - lse) - onehot(y)) * valid`` for selected rows
    (``scale``: a number, or one value per selected row)."""
    X = np.asarray(X, np.float64)
    W = np.asarray(W, np.float64)
    rows = np.asarray(rows, dtype=np.int64)
    lab = np.asarray(labels, dtype=np.int64)[rows]
    z = X[rows] @ W.T
    p = np.exp(z - np.asarray(lse_rows, np.float64)[:, None])
    ok = lab != ignore_index
    p[np.nonzero(ok)[0], lab[ok]] -= 1.0
    p[~ok, :] = 0.0
    return np.reshape(scale, (-1, 1)) * p if np.ndim(scale) else scale * p


def backward_dx_rows(X, W, labels, rows, scale: float, ignore_index: int = -100, lse_rows=None):
    """``dX[rows] = G[rows] W``; needs only the selected rows' own lse."""
    rows = np.asarray(rows, dtype=np.int64)
    if lse_rows is None:
        lse_rows, _ = lse_and_target(X, W, labels, ignore_index, rows)
    G = grad_logits_rows(X, W, labels, rows, lse_rows, scale, ignore_index)
    return G @ np.asarray(W, np.float64)


def backward_dw_ids(X, W, labels, lse_all, ids, scale, ignore_index: int = -100):
    """``dW[ids] = G[:, ids]^T X``; needs every row's lse (``scale``: number or per row)."""
    X = np.asarray(X, np.float64)
    W = np.asarray(W, np.float64)
    ids = np.asarray(ids, dtype=np.int64)
    lab = np.asarray(labels, dtype=np.int64)
    z = X @ W[ids].T                                    # [N, k]
    p = np.exp(z - np.asarray(lse_all, np.float64)[:, None])
    p -= (lab[:, None] == ids[None, :]).astype(np.float64)
    p[lab == ignore_index, :] = 0.0
    if np.ndim(scale):
        p = p * np.reshape(scale, (-1, 1))
        return p.T @ X
    return scale * (p.T @ X)


def full(X, W, labels, ignore_index: int = -100, reduction: str = "mean", grad_output=1.0):
    """Loss, lse, dX and dW for a whole (small) problem, in float64
    (``grad_output``: one number, or one per row for ``none``)."""
    X = np.asarray(X, np.float64)
    W = np.asarray(W, np.float64)
    f = forward(X, W, labels, ignore_index, reduction)
    s = grad_scale(f["n_valid"], reduction, grad_output)
    rows = np.arange(X.shape[0])
    G = grad_logits_rows(X, W, labels, rows, f["lse"], s, ignore_index)
    f["dX"] = G @ W
    f["dW"] = G.T @ X
    f["scale"] = s
    return f


def full_bf16(problem, grad_output: float = 1.0):
    """``full`` on a ``synth.Problem`` (bf16 bits widened exactly)."""
    return full(widen_bf16(problem.X), widen_bf16(problem.W), problem.labels,
                problem.ignore_index, problem.reduction, grad_output)


# ----------------------------------------------------------------------------- distillation without full logits
# "What-Each-Parallelism-Actually-Shards" §7.6 suggests keeping only top-k logits
# (or a chunked KL) for distillation instead of returning [B,S,V] logits.

def topk(X, W, k: int):
    """Per row: the k largest logits (high to low; ties keep the lower id first),
    their ids, and the row's lse."""
    X = np.asarray(X, np.float64)
    W = np.asarray(W, np.float64)
    n = X.shape[0]
    idx = np.full((n, k), -1, dtype=np.int64)     # a row no block reaches stays -1 / NaN
    val = np.full((n, k), np.nan)
    lse = np.full(n, np.nan)
    for blk in _row_blocks(n, W.shape[0]):
        z = X[blk] @ W.T
        order = np.argsort(-z, axis=1, kind="stable")[:, :k]
        idx[blk] = order
        val[blk] = np.take_along_axis(z, order, axis=1)
        m = z.max(axis=1)
        lse[blk] = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
    return idx, val, lse


def soft_full(X, W, tgt_idx, tgt_prob, reduction: str = "mean", grad_output=1.0):
    """KL(q || p) of sparse soft targets per row against p = softmax(X W^T):
    loss_i = sum_k q_k log q_k - sum_k q_k log p_{id_k} (entries with q <= 0 unused;
    a row with no positive mass is ignored), and the gradients of g * loss."""
    X = np.asarray(X, np.float64)
    W = np.asarray(W, np.float64)
    idx = np.asarray(tgt_idx, dtype=np.int64)
    q = np.where(np.asarray(tgt_prob, np.float64) > 0, np.asarray(tgt_prob, np.float64), 0.0)
    n = X.shape[0]
    z = X @ W.T
    m = z.max(axis=1)
    lse = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
    logp = z - lse[:, None]
    Q = q.sum(axis=1)
    valid = Q > 0
    ent = np.where(q > 0, q * np.log(np.where(q > 0, q, 1.0)), 0.0).sum(axis=1)
    cross = (q * np.take_along_axis(logp, idx, axis=1)).sum(axis=1)
    loss_rows = np.where(valid, ent - cross, 0.0)
    n_valid = int(valid.sum())
    if reduction == "mean":
        loss = 0.0 if n_valid == 0 else float(loss_rows.sum()) / n_valid
    elif reduction == "sum":
        loss = float(loss_rows.sum())
    elif reduction == "none":
        loss = loss_rows.copy()
    else:
        raise ValueError(reduction)
    s = grad_scale(n_valid, reduction, grad_output)
    G = np.exp(logp) * Q[:, None]
    np.add.at(G, (np.repeat(np.arange(n), idx.shape[1]), idx.reshape(-1)), -q.reshape(-1))
    G[~valid] = 0.0
    G = (np.reshape(s, (-1, 1)) if np.ndim(s) else s) * G
    return dict(loss=loss, lse=lse, loss_rows=loss_rows, n_valid=n_valid, dX=G @ W, dW=G.T @ X)
