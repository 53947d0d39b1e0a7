"""ctypes binding over ``libflce.so`` (C-ABI declared in ``include/flce.h``).

Argument marshalling only: shapes, dtypes and device pointers are checked and
passed through; every step of the computation runs in the library's kernels.
PyTorch is used for device memory and the current stream.  There is no CPU
fallback: if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None

FLCE_OK = 0
FLCE_ERR_LABEL_OUT_OF_RANGE = 5
FLCE_ERR_TIMEOUT = 6
REDUCTIONS = {"mean": 0, "sum": 1, "none": 2}

EXPORTED = ("flce_workspace_bytes", "flce_workspace_bytes_rowchunk", "flce_forward", "flce_backward", "flce_fwd_bwd",
            "flce_fwd_bwd_rowchunk", "flce_read_device_status", "flce_selftest_timeout", "flce_profile_enable",
            "flce_profile_read", "flce_forward_noalloc", "flce_scale_grads", "flce_topk_workspace_bytes", "flce_topk",
            "flce_soft_fwd_bwd", "flce_soft_fwd_bwd_rowchunk", "flce_host_buffer_bytes", "flce_fwd_bwd_host", "flce_shard_workspace_bytes",
            "flce_shard_forward", "flce_shard_combine", "flce_shard_backward", "flce_valid_count",
            "flce_f32_to_bf16", "flce_debug_checks", "flce_selftest_bounds", "flce_status_string")
KERNEL_KINDS = ("forward", "grad", "dxdw", "small")


class FlceError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        self.code = int(code)
        msg = status_string(code) if _LIB is not None else f"status {code}"
        super().__init__(f"{where}: {msg} (status {code})" if where else f"{msg} (status {code})")


class Problem(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int64), ("h", ctypes.c_int64), ("v", ctypes.c_int64),
                ("ignore_index", ctypes.c_int32), ("reduction", ctypes.c_int32),
                ("shift", ctypes.c_int32), ("seq_len", ctypes.c_int32)]


class VocabShard(ctypes.Structure):
    _fields_ = [("v_offset", ctypes.c_int64), ("v_rows", ctypes.c_int64)]


def lib_path() -> str:
    return os.environ.get("FLCE_LIB", os.path.join(HERE, "libflce.so"))


def lib():
    """Load the C-ABI library (once).  Raises if it is not built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        raise FlceError(-1, f"{path} is not built; run __graft_entry__.build() or "
                            "python -m lm_head_cross_gb300.build")
    L = ctypes.CDLL(path)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    P = ctypes.POINTER(Problem)
    L.flce_workspace_bytes.argtypes = [P]
    L.flce_workspace_bytes.restype = sz
    L.flce_workspace_bytes_rowchunk.argtypes = [P]
    L.flce_workspace_bytes_rowchunk.restype = sz
    S = ctypes.POINTER(VocabShard)
    L.flce_shard_workspace_bytes.argtypes = [P, S]
    L.flce_shard_workspace_bytes.restype = sz
    L.flce_shard_forward.argtypes = [P, S, vp, vp, vp, vp, vp, vp, sz, vp]
    L.flce_shard_forward.restype = ctypes.c_int
    L.flce_shard_combine.argtypes = [P, ctypes.c_int32, vp, vp, vp, vp, vp, vp, sz, vp]
    L.flce_shard_combine.restype = ctypes.c_int
    L.flce_shard_backward.argtypes = [P, S, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.flce_shard_backward.restype = ctypes.c_int
    L.flce_valid_count.argtypes = [P, vp, vp, vp, sz, vp]
    L.flce_valid_count.restype = ctypes.c_int
    L.flce_f32_to_bf16.argtypes = [vp, vp, ctypes.c_int64, vp]
    L.flce_f32_to_bf16.restype = ctypes.c_int
    L.flce_forward_noalloc.argtypes = [P, vp, vp, vp, vp, vp, vp]
    L.flce_forward_noalloc.restype = ctypes.c_int
    L.flce_forward.argtypes = [P, vp, vp, vp, vp, vp, vp, sz, vp]
    L.flce_forward.restype = ctypes.c_int
    L.flce_backward.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.flce_backward.restype = ctypes.c_int
    L.flce_fwd_bwd.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.flce_fwd_bwd.restype = ctypes.c_int
    L.flce_fwd_bwd_rowchunk.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.flce_fwd_bwd_rowchunk.restype = ctypes.c_int
    L.flce_topk_workspace_bytes.argtypes = [P, ctypes.c_int32]
    L.flce_topk_workspace_bytes.restype = sz
    L.flce_topk.argtypes = [P, ctypes.c_int32, vp, vp, vp, vp, vp, vp, sz, vp]
    L.flce_topk.restype = ctypes.c_int
    L.flce_soft_fwd_bwd.argtypes = [P, ctypes.c_int32, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.flce_soft_fwd_bwd.restype = ctypes.c_int
    L.flce_soft_fwd_bwd_rowchunk.argtypes = [P, ctypes.c_int32, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.flce_soft_fwd_bwd_rowchunk.restype = ctypes.c_int
    L.flce_host_buffer_bytes.argtypes = [P]
    L.flce_host_buffer_bytes.restype = sz
    L.flce_fwd_bwd_host.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp, vp]
    L.flce_fwd_bwd_host.restype = ctypes.c_int
    L.flce_scale_grads.argtypes = [P, vp, vp, vp, vp]
    L.flce_scale_grads.restype = ctypes.c_int
    L.flce_read_device_status.argtypes = [vp, vp]
    L.flce_read_device_status.restype = ctypes.c_int
    L.flce_selftest_timeout.argtypes = [vp, sz, ctypes.c_uint64, vp]
    L.flce_selftest_timeout.restype = ctypes.c_int
    L.flce_profile_enable.argtypes = [ctypes.c_int]
    L.flce_profile_enable.restype = ctypes.c_int
    L.flce_profile_read.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double),
                                    ctypes.POINTER(ctypes.c_double)]
    L.flce_profile_read.restype = ctypes.c_int
    L.flce_debug_checks.argtypes = []
    L.flce_debug_checks.restype = ctypes.c_int
    L.flce_selftest_bounds.argtypes = [vp, sz, vp]
    L.flce_selftest_bounds.restype = ctypes.c_int
    L.flce_status_string.argtypes = [ctypes.c_int]
    L.flce_status_string.restype = ctypes.c_char_p
    _LIB = L
    return L


def status_string(code: int) -> str:
    return lib().flce_status_string(int(code)).decode()


def logits_footprint_bytes(n_rows: int, v: int, elem_bytes: int) -> int:
    """Bytes of a materialised [N, V] logits tensor (what the fused path never allocates)."""
    return int(n_rows) * int(v) * int(elem_bytes)


def _problem(n, h, v, ignore_index, reduction, shift=0, seq_len=0) -> Problem:
    if reduction not in REDUCTIONS:
        raise ValueError(f"reduction must be 'mean', 'sum' or 'none', got {reduction!r}")
    if shift not in (0, 1):
        raise ValueError("shift must be 0 or 1")
    if shift and (seq_len < 1 or n % seq_len):
        raise ValueError("shift=1 needs seq_len dividing the number of rows")
    return Problem(int(n), int(h), int(v), int(ignore_index), REDUCTIONS[reduction], int(shift),
                   int(seq_len) if shift else 0)


def workspace_bytes(n, h, v, ignore_index=-100, reduction="mean") -> int:
    """Workspace of forward, backward and fwd_bwd: bounded, independent of V."""
    p = _problem(n, h, v, ignore_index, reduction)
    return int(lib().flce_workspace_bytes(ctypes.byref(p)))


def workspace_bytes_rowchunk(n, h, v, ignore_index=-100, reduction="mean") -> int:
    """Workspace of the row-chunk calls (fwd_bwd(rowchunk=True), soft_fwd_bwd); grows with V."""
    p = _problem(n, h, v, ignore_index, reduction)
    return int(lib().flce_workspace_bytes_rowchunk(ctypes.byref(p)))


def _torch():
    import torch
    return torch


def _stream_ptr(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check_inputs(x, w, labels):
    torch = _torch()
    if x.dim() != 2 or w.dim() != 2 or labels.dim() != 1:
        raise ValueError("x must be [N, H], w [V, H], labels [N]")
    if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16:
        raise TypeError("x and w must be bfloat16")
    if labels.dtype != torch.int32:
        raise TypeError("labels must be int32")
    if not (x.is_cuda and w.is_cuda and labels.is_cuda):
        raise ValueError("x, w and labels must be CUDA tensors")
    if not (x.is_contiguous() and w.is_contiguous() and labels.is_contiguous()):
        raise ValueError("x, w and labels must be contiguous")
    if x.shape[1] != w.shape[1] or labels.shape[0] != x.shape[0]:
        raise ValueError(f"shape mismatch: x {tuple(x.shape)}, w {tuple(w.shape)}, labels {tuple(labels.shape)}")


def _alloc_ws(n, h, v, ignore_index, reduction, device, rowchunk=False):
    torch = _torch()
    nbytes = (workspace_bytes_rowchunk if rowchunk else workspace_bytes)(n, h, v, ignore_index, reduction)
    if nbytes == 0:
        raise FlceError(1, "workspace_bytes")
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def _call(name, code):
    if code != FLCE_OK:
        raise FlceError(code, name)


def forward(x, w, labels, ignore_index=-100, reduction="mean", ws=None, stream=None, check=False, shift=0,
            seq_len=0):
    """Returns (loss fp32 ([1], or [N] per row for reduction 'none'), lse [N] fp32, ws)."""
    torch = _torch()
    _check_inputs(x, w, labels)
    n, h = x.shape
    v = w.shape[0]
    p = _problem(n, h, v, ignore_index, reduction, shift, seq_len)
    if ws is None:
        ws = _alloc_ws(n, h, v, ignore_index, reduction, x.device)
    loss = torch.empty(n if reduction == "none" else 1, dtype=torch.float32, device=x.device)
    lse = torch.empty(n, dtype=torch.float32, device=x.device)
    s = _stream_ptr(stream)
    _call("flce_forward", lib().flce_forward(ctypes.byref(p), x.data_ptr(), w.data_ptr(), labels.data_ptr(),
                                             loss.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(), s))
    if check:
        _call("device", read_device_status(ws, stream))
    return loss, lse, ws


def backward(x, w, labels, lse, grad_loss=None, ignore_index=-100, reduction="mean", ws=None, stream=None,
             check=False, shift=0, seq_len=0):
    """Returns (dX [N,H] bf16, dW [V,H] bf16, ws).  grad_loss: None or a 1-element fp32 CUDA
    tensor; for reduction 'none', an [N] fp32 CUDA tensor of per-row gradients (required)."""
    torch = _torch()
    _check_inputs(x, w, labels)
    n, h = x.shape
    v = w.shape[0]
    if lse.dtype != torch.float32 or lse.shape != (n,) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [N]")
    want = n if reduction == "none" else 1
    if reduction == "none" and grad_loss is None:
        raise ValueError("reduction 'none' needs per-row gradients")
    if grad_loss is not None and (grad_loss.dtype != torch.float32 or grad_loss.numel() != want or not grad_loss.is_cuda
                                  or not grad_loss.is_contiguous()):
        raise ValueError(f"grad_loss must be a contiguous {want}-element fp32 CUDA tensor")
    p = _problem(n, h, v, ignore_index, reduction, shift, seq_len)
    if ws is None:
        ws = _alloc_ws(n, h, v, ignore_index, reduction, x.device)
    dX = torch.empty_like(x)
    dW = torch.empty_like(w)
    s = _stream_ptr(stream)
    g = None if grad_loss is None else grad_loss.data_ptr()
    _call("flce_backward", lib().flce_backward(ctypes.byref(p), x.data_ptr(), w.data_ptr(), labels.data_ptr(),
                                               lse.data_ptr(), g, dX.data_ptr(), dW.data_ptr(), ws.data_ptr(),
                                               ws.numel(), s))
    if check:
        _call("device", read_device_status(ws, stream))
    return dX, dW, ws


def fwd_bwd(x, w, labels, ignore_index=-100, reduction="mean", ws=None, stream=None, out=None, check=False,
            rowchunk=False, shift=0, seq_len=0):
    """Returns (loss, lse, dX, dW, ws).  ``out`` may pass preallocated (loss, lse, dX, dW).
    Default: flce_fwd_bwd on the bounded, V-independent workspace (logits recomputed in
    the backward pass).  ``rowchunk=True``: flce_fwd_bwd_rowchunk (logits computed once,
    a row chunk of the vocabulary gradient kept in a workspace that grows with V).  For
    reduction 'none' the loss is per row and the gradients are those of its sum."""
    torch = _torch()
    _check_inputs(x, w, labels)
    n, h = x.shape
    v = w.shape[0]
    p = _problem(n, h, v, ignore_index, reduction, shift, seq_len)
    if ws is None:
        ws = _alloc_ws(n, h, v, ignore_index, reduction, x.device, rowchunk=rowchunk)
    if out is None:
        out = (torch.empty(n if reduction == "none" else 1, dtype=torch.float32, device=x.device),
               torch.empty(n, dtype=torch.float32, device=x.device), torch.empty_like(x), torch.empty_like(w))
    loss, lse, dX, dW = out
    s = _stream_ptr(stream)
    name = "flce_fwd_bwd_rowchunk" if rowchunk else "flce_fwd_bwd"
    _call(name, getattr(lib(), name)(ctypes.byref(p), x.data_ptr(), w.data_ptr(), labels.data_ptr(),
                                     loss.data_ptr(), lse.data_ptr(), dX.data_ptr(), dW.data_ptr(),
                                     ws.data_ptr(), ws.numel(), s))
    if check:
        _call("device", read_device_status(ws, stream))
    return loss, lse, dX, dW, ws


def host_buffer_bytes(n, h, v, ignore_index=-100, reduction="mean") -> int:
    """Device buffer of fwd_bwd_host: the workspace, then device copies of inputs and results."""
    p = _problem(n, h, v, ignore_index, reduction)
    return int(lib().flce_host_buffer_bytes(ctypes.byref(p)))


def fwd_bwd_host(x, w, labels, out, dev, ignore_index=-100, reduction="mean", stream=None, shift=0, seq_len=0,
                 in_stream=None, out_stream=None):
    """flce_fwd_bwd_host: x, w, labels and out = (loss, lse, dX, dW) are CPU tensors (pinned for
    asynchronous copies), dev a CUDA uint8 tensor of host_buffer_bytes.  Input copies on
    `in_stream`, the pass on `stream`, result copies on `out_stream` (each defaults to `stream`);
    synchronise before reading `out`.  Device status: read_device_status(dev)."""
    torch = _torch()
    if x.is_cuda or w.is_cuda or labels.is_cuda or any(t.is_cuda for t in out):
        raise ValueError("fwd_bwd_host takes host tensors")
    if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16 or labels.dtype != torch.int32:
        raise TypeError("x and w must be bfloat16, labels int32")
    if not (x.is_contiguous() and w.is_contiguous() and labels.is_contiguous()):
        raise ValueError("inputs must be contiguous")
    n, h = x.shape
    v = w.shape[0]
    p = _problem(n, h, v, ignore_index, reduction, shift, seq_len)
    loss, lse, dX, dW = out
    s = _stream_ptr(stream)
    si = _stream_ptr(in_stream) if in_stream is not None else s
    so = _stream_ptr(out_stream) if out_stream is not None else s
    _call("flce_fwd_bwd_host", lib().flce_fwd_bwd_host(ctypes.byref(p), x.data_ptr(), w.data_ptr(), labels.data_ptr(),
                                                       loss.data_ptr(), lse.data_ptr(), dX.data_ptr(), dW.data_ptr(),
                                                       dev.data_ptr(), dev.numel(), s, si, so))
    return out


def topk_workspace_bytes(n, h, v, k) -> int:
    p = _problem(n, h, v, -100, "mean")
    return int(lib().flce_topk_workspace_bytes(ctypes.byref(p), int(k)))


def topk(x, w, k, ws=None, stream=None):
    """Per row, the k largest logits of x @ w.T (high to low), their ids and the row's lse.
    Returns (idx [N,k] int32, logit [N,k] fp32, lse [N] fp32, ws)."""
    torch = _torch()
    n, h = x.shape
    v = w.shape[0]
    dummy = torch.empty(n, dtype=torch.int32, device=x.device)
    _check_inputs(x, w, dummy)
    p = _problem(n, h, v, -100, "mean")
    if ws is None:
        nbytes = int(lib().flce_topk_workspace_bytes(ctypes.byref(p), int(k)))
        if nbytes == 0:
            raise FlceError(1, "flce_topk_workspace_bytes")
        ws = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    idx = torch.empty(n, k, dtype=torch.int32, device=x.device)
    val = torch.empty(n, k, dtype=torch.float32, device=x.device)
    lse = torch.empty(n, dtype=torch.float32, device=x.device)
    _call("flce_topk", lib().flce_topk(ctypes.byref(p), int(k), x.data_ptr(), w.data_ptr(), idx.data_ptr(),
                                       val.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(), _stream_ptr(stream)))
    return idx, val, lse, ws


def soft_fwd_bwd(x, w, tgt_idx, tgt_prob, reduction="mean", ws=None, stream=None, rowchunk=False):
    """KL of sparse soft targets (k ids and probabilities per row) against softmax(x @ w.T),
    forward and backward.  Returns (loss, lse, dX, dW, ws).  Bounded workspace by default;
    ``rowchunk=True``: flce_soft_fwd_bwd_rowchunk."""
    torch = _torch()
    n, h = x.shape
    v = w.shape[0]
    k = int(tgt_idx.shape[1])
    if tgt_idx.shape != (n, k) or tgt_prob.shape != (n, k) or tgt_idx.dtype != torch.int32 or \
            tgt_prob.dtype != torch.float32 or not (tgt_idx.is_contiguous() and tgt_prob.is_contiguous()):
        raise ValueError("targets must be contiguous [N, k] int32 ids and fp32 probabilities")
    _check_inputs(x, w, torch.empty(n, dtype=torch.int32, device=x.device))
    p = _problem(n, h, v, -100, reduction)
    if ws is None:
        ws = _alloc_ws(n, h, v, -100, reduction, x.device, rowchunk=rowchunk)
    loss = torch.empty(n if reduction == "none" else 1, dtype=torch.float32, device=x.device)
    lse = torch.empty(n, dtype=torch.float32, device=x.device)
    dX = torch.empty_like(x)
    dW = torch.empty_like(w)
    name = "flce_soft_fwd_bwd_rowchunk" if rowchunk else "flce_soft_fwd_bwd"
    _call(name, getattr(lib(), name)(ctypes.byref(p), k, x.data_ptr(), w.data_ptr(), tgt_idx.data_ptr(),
                                     tgt_prob.data_ptr(), loss.data_ptr(), lse.data_ptr(), dX.data_ptr(),
                                     dW.data_ptr(), ws.data_ptr(), ws.numel(), _stream_ptr(stream)))
    return loss, lse, dX, dW, ws


def read_device_status(ws, stream=None) -> int:
    """Synchronises the stream and returns (and clears) the workspace's status word."""
    return int(lib().flce_read_device_status(ctypes.c_void_p(ws.data_ptr()), _stream_ptr(stream)))


def profile_enable(on: bool = True, kinds=None) -> None:
    """Time the launches of the given kernel kinds (names from KERNEL_KINDS; all when None)."""
    mask = 0
    if on:
        mask = -1 if kinds is None else sum(1 << KERNEL_KINDS.index(k) for k in kinds)
    _call("flce_profile_enable", lib().flce_profile_enable(mask))


def profile_read() -> dict:
    """{kind: (launches, total_ms, flops)} for the launches recorded since profile_enable."""
    out = {}
    for k, name in enumerate(KERNEL_KINDS):
        n, ms, fl = ctypes.c_int64(), ctypes.c_double(), ctypes.c_double()
        _call("flce_profile_read", lib().flce_profile_read(k, ctypes.byref(n), ctypes.byref(ms), ctypes.byref(fl)))
        out[name] = (int(n.value), float(ms.value), float(fl.value))
    return out


def scale_grads(dX, dW, grad_loss, stream=None):
    """dX *= g, dW *= g in place (g: one-element fp32 CUDA tensor)."""
    n, h = dX.shape
    v = dW.shape[0]
    p = _problem(n, h, v, -100, "mean")
    _call("flce_scale_grads", lib().flce_scale_grads(ctypes.byref(p), grad_loss.data_ptr(), dX.data_ptr(),
                                                     dW.data_ptr(), _stream_ptr(stream)))


def _f32(t, shape, name):
    torch = _torch()
    if t.dtype != torch.float32 or tuple(t.shape) != tuple(shape) or not t.is_contiguous() or not t.is_cuda:
        raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor of shape {tuple(shape)}")


def shard_workspace_bytes(n, h, v_total, v_offset, v_rows, ignore_index=-100, reduction="mean") -> int:
    p = _problem(n, h, v_total, ignore_index, reduction)
    sh = VocabShard(int(v_offset), int(v_rows))
    return int(lib().flce_shard_workspace_bytes(ctypes.byref(p), ctypes.byref(sh)))


def _shard_ws(x, w_shard, v_total, v_offset, ignore_index, reduction, shift, seq_len, ws):
    torch = _torch()
    n, h = x.shape
    if ws is not None:
        return ws
    p = _problem(n, h, v_total, ignore_index, reduction, shift, seq_len)
    sh = VocabShard(int(v_offset), int(w_shard.shape[0]))
    nbytes = int(lib().flce_shard_workspace_bytes(ctypes.byref(p), ctypes.byref(sh)))
    if nbytes == 0:
        raise FlceError(1, "flce_shard_workspace_bytes")
    return torch.empty(nbytes, dtype=torch.uint8, device=x.device)


def shard_forward(x, w_shard, labels, v_offset, v_total, ignore_index=-100, shift=0, seq_len=0, ws=None,
                  stream=None):
    """Vocabulary shard [v_offset, v_offset + w_shard.shape[0]) of a v_total-row LM head:
    (lse_part [N], tgt_part [N], ws) — the shard's per-row lse and the target logit
    where the shard holds the label (else 0)."""
    torch = _torch()
    _check_inputs(x, w_shard, labels)
    n, h = x.shape
    p = _problem(n, h, v_total, ignore_index, "mean", shift, seq_len)
    sh = VocabShard(int(v_offset), int(w_shard.shape[0]))
    ws = _shard_ws(x, w_shard, v_total, v_offset, ignore_index, "mean", shift, seq_len, ws)
    lse_p = torch.empty(n, dtype=torch.float32, device=x.device)
    tgt_p = torch.empty(n, dtype=torch.float32, device=x.device)
    _call("flce_shard_forward", lib().flce_shard_forward(ctypes.byref(p), ctypes.byref(sh), x.data_ptr(),
                                                         w_shard.data_ptr(), labels.data_ptr(), lse_p.data_ptr(),
                                                         tgt_p.data_ptr(), ws.data_ptr(), ws.numel(),
                                                         _stream_ptr(stream)))
    return lse_p, tgt_p, ws


def shard_combine(lse_parts, tgt_parts, labels, v_total, h, ignore_index=-100, reduction="mean", shift=0,
                  seq_len=0, ws=None, stream=None):
    """lse_parts, tgt_parts: [P, N] fp32 (shard r in row r).  Returns (loss, lse [N], ws).
    ``ws``: any workspace of a shard call (or of fwd_bwd) on the same rows serves."""
    torch = _torch()
    P, n = lse_parts.shape
    _f32(lse_parts, (P, n), "lse_parts")
    _f32(tgt_parts, (P, n), "tgt_parts")
    if labels.dtype != torch.int32 or labels.shape != (n,) or not labels.is_contiguous():
        raise ValueError("labels must be contiguous int32 [N]")
    p = _problem(n, h, v_total, ignore_index, reduction, shift, seq_len)
    if ws is None:
        nbytes = int(lib().flce_workspace_bytes(ctypes.byref(p)))
        ws = torch.empty(nbytes, dtype=torch.uint8, device=lse_parts.device)
    loss = torch.empty(n if reduction == "none" else 1, dtype=torch.float32, device=lse_parts.device)
    lse = torch.empty(n, dtype=torch.float32, device=lse_parts.device)
    _call("flce_shard_combine", lib().flce_shard_combine(ctypes.byref(p), int(P), lse_parts.data_ptr(),
                                                         tgt_parts.data_ptr(), labels.data_ptr(), loss.data_ptr(),
                                                         lse.data_ptr(), ws.data_ptr(), ws.numel(),
                                                         _stream_ptr(stream)))
    return loss, lse, ws


def shard_backward(x, w_shard, labels, lse, v_offset, v_total, grad_loss=None, ignore_index=-100,
                   reduction="mean", shift=0, seq_len=0, ws=None, stream=None):
    """Given the global lse: (dX_part [N, H] fp32, dW_shard [rows, H] bf16, ws)."""
    torch = _torch()
    _check_inputs(x, w_shard, labels)
    n, h = x.shape
    _f32(lse, (n,), "lse")
    p = _problem(n, h, v_total, ignore_index, reduction, shift, seq_len)
    sh = VocabShard(int(v_offset), int(w_shard.shape[0]))
    ws = _shard_ws(x, w_shard, v_total, v_offset, ignore_index, reduction, shift, seq_len, ws)
    dXp = torch.empty(n, h, dtype=torch.float32, device=x.device)
    dWs = torch.empty_like(w_shard)
    g = None if grad_loss is None else grad_loss.data_ptr()
    _call("flce_shard_backward", lib().flce_shard_backward(ctypes.byref(p), ctypes.byref(sh), x.data_ptr(),
                                                           w_shard.data_ptr(), labels.data_ptr(), lse.data_ptr(), g,
                                                           dXp.data_ptr(), dWs.data_ptr(), ws.data_ptr(), ws.numel(),
                                                           _stream_ptr(stream)))
    return dXp, dWs, ws


def valid_count(labels, v, h=8, ignore_index=-100, shift=0, seq_len=0, ws=None, stream=None):
    """Rows whose label is not ignore_index, as a one-element int32 CUDA tensor.
    ``ws``: any workspace of another call on the same rows serves."""
    torch = _torch()
    n = labels.shape[0]
    p = _problem(n, h, v, ignore_index, "sum", shift, seq_len)
    if ws is None:
        ws = torch.empty(max(256, int(lib().flce_workspace_bytes(ctypes.byref(p)))), dtype=torch.uint8,
                         device=labels.device)
    out = torch.empty(1, dtype=torch.int32, device=labels.device)
    _call("flce_valid_count", lib().flce_valid_count(ctypes.byref(p), labels.data_ptr(), out.data_ptr(),
                                                     ws.data_ptr(), ws.numel(), _stream_ptr(stream)))
    return out, ws


def f32_to_bf16(src, out=None, stream=None):
    """bf16 copy of a contiguous fp32 CUDA tensor (round to nearest even)."""
    torch = _torch()
    if src.dtype != torch.float32 or not src.is_contiguous() or not src.is_cuda:
        raise ValueError("src must be a contiguous fp32 CUDA tensor")
    if out is None:
        out = torch.empty(src.shape, dtype=torch.bfloat16, device=src.device)
    _call("flce_f32_to_bf16", lib().flce_f32_to_bf16(src.data_ptr(), out.data_ptr(), src.numel(),
                                                     _stream_ptr(stream)))
    return out


class _LinearCrossEntropy:
    """torch.autograd.Function wrapper, built lazily so importing needs no torch.

    When a gradient is needed, the forward runs the fused forward + backward
    (flce_fwd_bwd, upstream gradient 1) and keeps dX and dW; the backward then
    only multiplies them by the upstream gradient.  Otherwise the forward runs
    the forward pass alone."""
    fn = None

    @classmethod
    def get(cls):
        if cls.fn is None:
            torch = _torch()

            class Fn(torch.autograd.Function):
                @staticmethod
                def forward(ctx, x2, w, labels, ignore_index, reduction, shift, seq_len, rowchunk):
                    ctx.reduction = reduction
                    kw = dict(shift=shift, seq_len=seq_len)
                    needs = ctx.needs_input_grad[0] or ctx.needs_input_grad[1]
                    if needs and reduction != "none":
                        loss, _, dX, dW, _ = fwd_bwd(x2, w, labels, ignore_index, reduction, rowchunk=rowchunk, **kw)
                        ctx.save_for_backward(dX, dW)
                        return loss.reshape(())
                    loss, lse, _ = forward(x2, w, labels, ignore_index, reduction, **kw)
                    if needs:  # per-row upstream gradients are only known in backward: recompute there
                        ctx.save_for_backward(x2, w, labels, lse)
                        ctx.args = (ignore_index, kw)
                    return loss if reduction == "none" else loss.reshape(())

                @staticmethod
                def backward(ctx, grad):
                    if ctx.reduction == "none":
                        x2, w, labels, lse = ctx.saved_tensors
                        ignore_index, kw = ctx.args
                        g = grad.detach().to(torch.float32).reshape(-1).contiguous()
                        dX, dW, _ = backward(x2, w, labels, lse, g, ignore_index, "none", **kw)
                        return dX, dW, None, None, None, None, None, None
                    dX, dW = ctx.saved_tensors
                    g = grad.detach().to(torch.float32).reshape(1).contiguous()
                    scale_grads(dX, dW, g)
                    return dX, dW, None, None, None, None, None, None

            cls.fn = Fn
        return cls.fn


def linear_cross_entropy(x, w, labels, ignore_index: int = -100, reduction: str = "mean", shift: int = 0,
                         rowchunk: bool = False):
    """Cross-entropy of ``x @ w.T`` against ``labels`` without materialising the logits.

    x: [..., H] bf16 CUDA, w: [V, H] bf16, labels: [...] integer (same leading
    shape as x).  reduction: 'mean' (over non-ignored rows), 'sum' or 'none'
    (per-row losses, shaped like labels).  shift=1 scores position t of each
    sequence against the label at t + 1 (x and labels [B, S, ...]; the last
    position of each sequence is ignored).  Autograd flows to x and w.
    The extra device memory is bounded and independent of V (logits recomputed
    in the backward pass); ``rowchunk=True`` computes the logits once and keeps a
    row chunk of the vocabulary gradient instead (memory grows with V).
    """
    torch = _torch()
    h = x.shape[-1]
    seq_len = 0
    if shift:
        if x.dim() < 3:
            raise ValueError("shift=1 needs x shaped [B, S, H]")
        seq_len = int(x.shape[-2])
    x2 = x.reshape(-1, h).contiguous()
    lab = labels.reshape(-1).to(torch.int32).contiguous()
    loss = _LinearCrossEntropy.get().apply(x2, w.contiguous(), lab, int(ignore_index), reduction, int(shift),
                                           seq_len, bool(rowchunk))
    return loss.reshape(labels.shape) if reduction == "none" else loss


class _SparseKL:
    """torch.autograd.Function for the soft-target KL: the forward runs the fused
    forward + backward (flce_soft_fwd_bwd, upstream gradient 1) and keeps dX and
    dW; the backward multiplies them by the upstream gradient."""
    fn = None

    @classmethod
    def get(cls):
        if cls.fn is None:
            torch = _torch()

            class Fn(torch.autograd.Function):
                @staticmethod
                def forward(ctx, x2, w, tgt_idx, tgt_prob, reduction, rowchunk):
                    loss, _, dX, dW, _ = soft_fwd_bwd(x2, w, tgt_idx, tgt_prob, reduction, rowchunk=rowchunk)
                    ctx.save_for_backward(dX, dW)
                    return loss.reshape(())

                @staticmethod
                def backward(ctx, grad):
                    dX, dW = ctx.saved_tensors
                    g = grad.detach().to(torch.float32).reshape(1).contiguous()
                    scale_grads(dX, dW, g)
                    return dX, dW, None, None, None, None

            cls.fn = Fn
        return cls.fn


def sparse_kl_divergence(x, w, tgt_idx, tgt_prob, reduction: str = "mean", rowchunk: bool = False):
    """KL(q || softmax(x @ w.T)) against sparse soft targets (a teacher's top-k ids
    and probabilities per row), without materialising the logits.

    x: [..., H] bf16 CUDA, w: [V, H] bf16, tgt_idx / tgt_prob: [..., k] (k <= 16)
    integer ids and fp32 probabilities; a row whose probabilities are all 0 is
    ignored.  reduction: 'mean' (over rows with targets) or 'sum'.  Autograd flows
    to x and w.  Bounded, V-independent extra memory by default; ``rowchunk=True``
    computes the logits once and keeps a row chunk of the vocabulary gradient.
    """
    torch = _torch()
    if reduction not in ("mean", "sum"):
        raise ValueError("sparse_kl_divergence takes reduction 'mean' or 'sum'")
    h = x.shape[-1]
    k = tgt_idx.shape[-1]
    x2 = x.reshape(-1, h).contiguous()
    idx = tgt_idx.reshape(-1, k).to(torch.int32).contiguous()
    q = tgt_prob.reshape(-1, k).to(torch.float32).contiguous()
    return _SparseKL.get().apply(x2, w.contiguous(), idx, q, reduction, bool(rowchunk))
