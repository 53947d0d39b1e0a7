"""Writes the fp64 oracle's forward results for the large synthetic workloads.

    python tests/golden/make_workload_golden.py [workload ...]

For each workload (default: the three whose full oracle forward takes minutes
rather than seconds) this draws the inputs with ``synth``, runs
``oracle.forward`` over every row and stores, in ``<workload>.npz`` beside
this script:

* ``lse``      float64 [N], every row's log-sum-exp
* ``loss``     float64, the reduced loss, and ``n_valid``
* ``fingerprint``  sha256 (hex) of the X, W and label bytes it was computed on
* ``recipe``   the workload's generator settings (``synth.WORKLOADS`` entry)

Only ``oracle`` and ``synth`` are called; no value comes from the CUDA path.
The parity tests check the fingerprint before they use a file, so a change of
the generator makes them fail loudly instead of comparing against stale data.
Every other oracle quantity the tests need (dX rows, dW of sampled ids) follows
from these per-row lse values cheaply and is computed in the tests.
"""
from __future__ import annotations

import hashlib
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

DEFAULT = ("n8192_h4096_v128256", "n32768_h4096_v151936", "n131072_h4096_v131072")


def fingerprint(problem) -> str:
    h = hashlib.sha256()
    for a in (problem.X, problem.W, problem.labels):
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()


def recipe(name: str) -> str:
    return json.dumps(synth.WORKLOADS[name], sort_keys=True)


def path_of(name: str) -> str:
    return os.path.join(HERE, f"{name}.npz")


def write(name: str) -> str:
    t0 = time.time()
    p = synth.workload_problem(name)
    fp = fingerprint(p)
    Xd = oracle.widen_bf16(p.X)
    Wd = oracle.widen_bf16(p.W)
    t1 = time.time()
    f = oracle.forward(Xd, Wd, p.labels, p.ignore_index, p.reduction)
    t2 = time.time()
    out = path_of(name)
    np.savez(out, lse=np.asarray(f["lse"], np.float64), loss=np.float64(f["loss"]),
             n_valid=np.int64(f["n_valid"]), fingerprint=np.array(fp), recipe=np.array(recipe(name)))
    print(f"{name}: inputs {t1 - t0:.0f} s, oracle forward {t2 - t1:.0f} s, loss {f['loss']:.9f}, "
          f"n_valid {f['n_valid']} -> {out}", flush=True)
    return out


def load(name: str, problem=None):
    """The stored results, after checking they belong to ``problem`` (if given) and to
    the current generator settings."""
    with np.load(path_of(name)) as z:
        d = {k: z[k] for k in z.files}
    if str(d["recipe"]) != recipe(name):
        raise RuntimeError(f"{name}: golden file was written for other generator settings; rerun {__file__}")
    if problem is not None and str(d["fingerprint"]) != fingerprint(problem):
        raise RuntimeError(f"{name}: golden file was written for other input bytes; rerun {__file__}")
    return d


if __name__ == "__main__":
    for name in (sys.argv[1:] or DEFAULT):
        write(name)
