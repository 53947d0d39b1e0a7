"""Fused LM-head projection + cross-entropy for GB300 (sm_103a).

Python binding over the C-ABI library ``libflce.so`` (declared in
``include/flce.h``).  Every step of the computation runs in the library's CUDA
kernels; this module only marshals arguments.  See ``binding`` for the calls.
"""
from .binding import (  # noqa: F401
    FlceError, Problem, lib, lib_path, workspace_bytes, workspace_bytes_min, forward, backward, fwd_bwd,
    read_device_status, status_string, linear_cross_entropy, logits_footprint_bytes,
    profile_enable, profile_read, KERNEL_KINDS, scale_grads, topk, topk_workspace_bytes, soft_fwd_bwd,
    host_buffer_bytes, fwd_bwd_host, sparse_kl_divergence,
)
