"""Sharded LM-head cross-entropy: vocabulary split, sequence split, or both.

"What-Each-Parallelism-Actually-Shards" §3.2 and §7.2 split the LM head's
vocabulary across ranks (vocab-parallel cross-entropy), §7.3 splits the tokens
(sequence-sharded loss), and §4.1 combines the two into [B, S/SP, V/TP] logits
per rank.  None of them ever forms the full logits.  This module runs the
exchange between ranks with ``torch.distributed`` (NCCL on GPUs, gloo on CPU);
every step of arithmetic on either side of it is a call into the library
(``binding``): per-shard log-sum-exp and target logit, their combination, the
shard backward, valid counts, scaling and the fp32 -> bf16 cast.

Exchange per call (P ranks in the vocabulary group, Q in the sequence group):

* vocabulary split: one all-gather of [2, N] fp32 (each shard's lse and target
  logit), then, after the backward, an all-reduce of the [N, H] fp32 dX parts;
  each rank's dW rows are complete without any exchange.
* sequence split: an all-reduce of two fp64 numbers (the loss sum and the valid
  count, so that a mean divides by the global count) and an all-reduce of dW in
  fp32 (every rank's rows add to every row of dW, as under data parallelism).

Returns the loss and the gradients of upstream gradient 1 (like
``binding.fwd_bwd``); scale them for another upstream gradient.
"""
from __future__ import annotations

from . import binding


class LibraryOps:
    """The per-rank steps, on the CUDA library.  One workspace serves every step
    of a call (``ws``: allocated by the first step, passed to the rest)."""

    @staticmethod
    def shard_forward(x, w_shard, labels, v_offset, v_total, ignore_index, shift, seq_len, ws=None):
        lse_p, tgt_p, ws = binding.shard_forward(x, w_shard, labels, v_offset, v_total, ignore_index, shift,
                                                 seq_len, ws=ws)
        return lse_p, tgt_p, ws

    @staticmethod
    def shard_combine(lse_parts, tgt_parts, labels, v_total, h, ignore_index, shift, seq_len, ws=None):
        loss, lse, ws = binding.shard_combine(lse_parts, tgt_parts, labels, v_total, h, ignore_index, "sum", shift,
                                              seq_len, ws=ws)
        return loss, lse, ws

    @staticmethod
    def shard_backward(x, w_shard, labels, lse, v_offset, v_total, scale, ignore_index, shift, seq_len, ws=None):
        dXp, dWs, ws = binding.shard_backward(x, w_shard, labels, lse, v_offset, v_total, scale, ignore_index, "sum",
                                              shift, seq_len, ws=ws)
        return dXp, dWs, ws

    @staticmethod
    def fwd_bwd(x, w, labels, ignore_index, shift, seq_len, ws=None):
        loss, lse, dX, dW, ws = binding.fwd_bwd(x, w, labels, ignore_index, "sum", ws=ws, shift=shift,
                                                seq_len=seq_len)
        return loss, lse, dX, dW, ws

    @staticmethod
    def valid_count(labels, v_total, ignore_index, shift, seq_len, ws=None):
        count, ws = binding.valid_count(labels, v_total, 8, ignore_index, shift, seq_len, ws=ws)
        return count, ws

    @staticmethod
    def scale_grads(dX, dW, scale):
        binding.scale_grads(dX, dW, scale)

    @staticmethod
    def f32_to_bf16(t):
        return binding.f32_to_bf16(t)


def _world(group):
    import torch.distributed as dist
    return 1 if group is None else dist.get_world_size(group)


def sharded_cross_entropy(x, w, labels, *, v_offset=0, v_total=None, vocab_group=None, seq_group=None,
                          ignore_index=-100, reduction="mean", shift=0, seq_len=0, ops=None, check=False):
    """Loss, lse and gradients of this rank's piece of a sharded LM-head cross-entropy.

    x: [N_r, H] bf16, this rank's rows (its slice of the sequence when
    ``seq_group`` is given, else all rows); w: [V_r, H] bf16, the rows
    [v_offset, v_offset + V_r) of the LM head (all V rows when ``vocab_group`` is
    None); labels: [N_r] int32 global vocabulary ids (or ignore_index).
    ``v_total``: the whole vocabulary (default: w's rows).  ``reduction``:
    'mean' (over the valid rows of every rank) or 'sum'.  shift=1 (the causal
    next-token shift within sequences of seq_len rows) needs complete sequences
    on the rank, so it is taken only without a sequence group.

    Returns (loss [1] fp32, lse [N_r] fp32 over the whole vocabulary,
    dX [N_r, H] bf16, dW [V_r, H] bf16): the loss is the same on every rank, dX
    covers this rank's rows, dW this rank's vocabulary rows summed over the
    sequence group.  ``check=True`` reads the device status word after each
    library step (a stream synchronisation each) and raises on a device error
    (a label outside the vocabulary, a bounded wait that ran out).
    """
    import torch
    import torch.distributed as dist

    ops = ops or LibraryOps

    def status(ws, step):
        if check and ops is LibraryOps:
            code = binding.read_device_status(ws)
            if code != binding.FLCE_OK:
                raise binding.FlceError(code, step)
    if reduction not in ("mean", "sum"):
        raise ValueError("sharded_cross_entropy takes reduction 'mean' or 'sum'")
    if shift and seq_group is not None and _world(seq_group) > 1:
        raise ValueError("shift=1 with a sequence group: shift the labels before splitting the rows")
    n, h = x.shape
    v_total = int(v_total if v_total is not None else w.shape[0])
    vocab_split = _world(vocab_group) > 1 or w.shape[0] != v_total
    if vocab_split and vocab_group is None and w.shape[0] != v_total:
        raise ValueError("a vocabulary shard needs the vocab_group it is part of")

    if vocab_split:
        lse_p, tgt_p, ws = ops.shard_forward(x, w, labels, v_offset, v_total, ignore_index, shift, seq_len)
        status(ws, "shard_forward")
        mine = torch.stack([lse_p, tgt_p])                      # [2, N]
        parts = [torch.empty_like(mine) for _ in range(_world(vocab_group))]
        dist.all_gather(parts, mine, group=vocab_group)
        lse_parts = torch.stack([t[0] for t in parts]).contiguous()
        tgt_parts = torch.stack([t[1] for t in parts]).contiguous()
        loss_sum, lse, ws = ops.shard_combine(lse_parts, tgt_parts, labels, v_total, h, ignore_index, shift,
                                              seq_len, ws=ws)
        status(ws, "shard_combine")
    else:
        loss_sum, lse, dX, dW, ws = ops.fwd_bwd(x, w, labels, ignore_index, shift, seq_len)
        status(ws, "fwd_bwd")
    count, ws = ops.valid_count(labels, v_total, ignore_index, shift, seq_len, ws=ws)
    status(ws, "valid_count")

    # the loss sum and the valid count of the whole sequence
    totals = torch.cat([loss_sum.reshape(1).to(torch.float64), count.reshape(1).to(torch.float64)])
    if seq_group is not None and _world(seq_group) > 1:
        dist.all_reduce(totals, group=seq_group)
    if reduction == "mean":
        scale = torch.where(totals[1] > 0, 1.0 / totals[1].clamp(min=1.0), torch.zeros_like(totals[1]))
    else:
        scale = torch.ones_like(totals[1])
    loss = (totals[0] * scale).to(torch.float32).reshape(1)
    scale32 = scale.to(torch.float32).reshape(1).contiguous()

    if vocab_split:
        dXp, dW, ws = ops.shard_backward(x, w, labels, lse, v_offset, v_total, scale32, ignore_index, shift,
                                         seq_len, ws=ws)
        status(ws, "shard_backward")
        dist.all_reduce(dXp, group=vocab_group)
        dX = ops.f32_to_bf16(dXp)
    else:
        ops.scale_grads(dX, dW, scale32)
    if seq_group is not None and _world(seq_group) > 1:
        dW32 = dW.to(torch.float32)
        dist.all_reduce(dW32, group=seq_group)
        dW = ops.f32_to_bf16(dW32)
    return loss, lse, dX, dW
