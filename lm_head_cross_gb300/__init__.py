"""Fused LM-head projection + cross-entropy for GB300 (sm_103a).

Python binding over the C-ABI library ``libflce.so`` (declared in
``include/flce.h``).  Every step of the computation runs in the library's CUDA
kernels; this module only marshals arguments.  See ``binding`` for the calls
and ``sharded`` for the vocabulary- and sequence-sharded loss across ranks.
"""
from .binding import (  # noqa: F401
    FlceError, Problem, VocabShard, lib, lib_path, workspace_bytes, workspace_bytes_rowchunk, forward, backward,
    fwd_bwd, read_device_status, status_string, linear_cross_entropy, logits_footprint_bytes,
    profile_enable, profile_read, KERNEL_KINDS, scale_grads, topk, topk_workspace_bytes, soft_fwd_bwd,
    host_buffer_bytes, fwd_bwd_host, sparse_kl_divergence, shard_workspace_bytes, shard_forward, shard_combine,
    shard_backward, valid_count, f32_to_bf16,
)
from .sharded import sharded_cross_entropy  # noqa: F401
