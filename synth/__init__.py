"""Seeded synthetic inputs for the fused linear + cross-entropy path.

This module only draws numbers.  It holds none of the method's arithmetic and
is the one piece that both the fp64 oracle (``oracle/``) and the CUDA path are
fed from, so that both sides see byte-identical inputs.

Inputs stand in for the long-sequence, large-vocabulary case of
"What-Each-Parallelism-Actually-Shards" §1.4 (hidden states ``[B,S,H]``, an LM
head weight, labels with an ignore sentinel as in §7.4's fused call).  No
dataset exists here; every value is drawn from a seeded PCG64 stream.

Recipe (fixed draw order, so a seed fixes every byte):

1. ``X[N,H]``: fp32 normal samples with the stated std, rounded to bf16
   (round-to-nearest-even).
2. ``W[V,H]``: fp32 normal samples with std ``w_std``; if ``outlier_rows > 0``,
   that many distinct vocab rows, chosen by the same stream, are multiplied by
   ``outlier_scale`` in fp32; then rounded to bf16.
3. ``labels[N]`` int32: ``uniform`` over ``[0, V)``, or ``zipf`` — rank ``r``
   in ``[1, V]`` drawn with probability proportional to ``r**-s`` by inverse CDF,
   mapped to id ``r - 1``.
4. Exactly ``round(ignore_frac * N)`` rows, picked by a seeded permutation,
   get ``ignore_index``.

bf16 tensors are returned as ``uint16`` bit patterns.
"""
from __future__ import annotations

import dataclasses
import numpy as np

IGNORE_INDEX = -100


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round finite fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns.

    Works in uint32 (no overflow for finite inputs) and in slices, so that a
    half-billion-element tensor does not need a 64-bit temporary.
    """
    flat = np.ascontiguousarray(a, dtype=np.float32).reshape(-1).view(np.uint32)
    out = np.empty(flat.shape, dtype=np.uint16)
    step = 1 << 24
    for s in range(0, flat.size, step):
        u = flat[s:s + step]
        r = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
        out[s:s + step] = (r >> np.uint32(16)).astype(np.uint16)
    return out.reshape(np.shape(a))


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Problem:
    """One synthetic problem: bf16 bit patterns plus the settings that go with them."""
    X: np.ndarray            # uint16 [N, H] (bf16 bits)
    W: np.ndarray            # uint16 [V, H] (bf16 bits)
    labels: np.ndarray       # int32 [N]
    ignore_index: int
    reduction: str           # "mean" | "sum"
    name: str = ""
    outlier_ids: np.ndarray | None = None

    @property
    def n(self) -> int:
        return int(self.X.shape[0])

    @property
    def h(self) -> int:
        return int(self.X.shape[1])

    @property
    def v(self) -> int:
        return int(self.W.shape[0])


def _normal_f32(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    out = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out


def _zipf_ids(rng: np.random.Generator, n: int, v: int, s: float) -> np.ndarray:
    ranks = np.arange(1, v + 1, dtype=np.float64)
    w = ranks ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    u = rng.random(n)
    idx = np.searchsorted(cdf, u, side="right")
    return np.minimum(idx, v - 1).astype(np.int32)


def make_problem(n: int, h: int, v: int, *, seed: int, x_std: float = 1.0, w_std: float = 0.02,
                 labels: str = "uniform", zipf_s: float = 1.1, ignore_frac: float = 0.0,
                 ignore_index: int = IGNORE_INDEX, reduction: str = "mean",
                 outlier_rows: int = 0, outlier_scale: float = 10.0, name: str = "") -> Problem:
    rng = np.random.Generator(np.random.PCG64(seed))
    X = f32_to_bf16_bits(_normal_f32(rng, (n, h), x_std))
    Wf = _normal_f32(rng, (v, h), w_std)
    outlier_ids = None
    if outlier_rows > 0:
        outlier_ids = np.sort(rng.choice(v, size=outlier_rows, replace=False)).astype(np.int64)
        Wf[outlier_ids] *= np.float32(outlier_scale)
    W = f32_to_bf16_bits(Wf)
    del Wf
    if labels == "uniform":
        lab = rng.integers(0, v, size=n, dtype=np.int64).astype(np.int32)
    elif labels == "zipf":
        lab = _zipf_ids(rng, n, v, zipf_s)
    else:
        raise ValueError(f"unknown label distribution {labels!r}")
    n_ignore = int(round(ignore_frac * n))
    if n_ignore:
        lab[rng.permutation(n)[:n_ignore]] = ignore_index
    return Problem(X=X, W=W, labels=lab, ignore_index=ignore_index, reduction=reduction,
                   name=name, outlier_ids=outlier_ids)


# The five workloads: long-sequence / large-vocabulary LM-head shapes, keyed by
# their sizes.
WORKLOADS = {
    "n256_h128_v1024": dict(n=256, h=128, v=1024, seed=0, x_std=1.0, w_std=0.02, labels="uniform",
            ignore_frac=0.10, reduction="mean", name="tiny N=256 H=128 V=1024"),
    "n8192_h2048_v32000": dict(n=8192, h=2048, v=32000, seed=1, x_std=1.0, w_std=0.02, labels="zipf",
            ignore_frac=0.05, reduction="mean", name="N=4x2048 H=2048 V=32000"),
    "n8192_h4096_v128256": dict(n=8192, h=4096, v=128256, seed=2, x_std=4.0 / 64.0, w_std=0.02, labels="zipf",
            ignore_frac=0.02, reduction="mean", name="N=8192 H=4096 V=128256"),
    "n32768_h4096_v151936": dict(n=32768, h=4096, v=151936, seed=3, x_std=1.0, w_std=0.02, labels="zipf",
            ignore_frac=0.05, reduction="sum", outlier_rows=64, outlier_scale=10.0,
            name="N=32768 H=4096 V=151936 (64 outlier vocab rows x10, sum)"),
    "n131072_h4096_v131072": dict(n=131072, h=4096, v=131072, seed=4, x_std=1.0, w_std=0.02, labels="uniform",
            ignore_frac=0.03, reduction="mean", name="N=128K H=4096 V=128K"),
    # not one of the five: three fused row chunks (the fp32 dW accumulator stored, added
    # to and read back) in a few GB of device memory, small enough for a full ncu capture
    "n24576_h2048_v65536": dict(n=24576, h=2048, v=65536, seed=5, x_std=1.0, w_std=0.02, labels="zipf",
            ignore_frac=0.05, reduction="mean", name="N=24576 H=2048 V=65536 (3 row chunks)"),
    # not one of the five: the bounded path's kernels at the 128K x 128K workload's hidden size and
    # vocabulary chunk width (4096, as for N > 16384), in about 1.4 GB of device memory
    "n24576_h4096_v16384": dict(n=24576, h=4096, v=16384, seed=6, x_std=1.0, w_std=0.02, labels="uniform",
            ignore_frac=0.03, reduction="mean", name="N=24576 H=4096 V=16384 (4 vocabulary chunks)"),
}


TINY = "n256_h128_v1024"
DEFAULT_WORKLOAD = "n8192_h2048_v32000"


def workload_problem(name: str) -> Problem:
    return make_problem(**WORKLOADS[name])


def workload_shape(name: str):
    c = WORKLOADS[name]
    return c["n"], c["h"], c["v"]
