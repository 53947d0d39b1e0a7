"""The C-ABI from a plain C99 program: tests/c/abi_device.c allocates device
memory with the CUDA runtime, calls flce_fwd_bwd through include/flce.h, and
writes the results; they must match the fp64 oracle like the Python path's."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import synth
from helpers import assert_grad, assert_loss, assert_lse

pytestmark = pytest.mark.gpu

import lm_head_cross_gb300 as flce  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_fwd_bwd_matches_oracle(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    lib = flce.lib_path()
    exe = tmp_path / "abi_device"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-I", os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "c", "abi_device.c"),
                        "-o", str(exe), lib, "-L", os.path.join(cuda, "lib64"), "-lcudart",
                        "-Wl,-rpath," + os.path.dirname(lib), "-Wl,-rpath," + os.path.join(cuda, "lib64")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    p = synth.make_problem(700, 136, 3001, seed=41, labels="zipf", ignore_frac=0.1, reduction="sum")
    p.X.tofile(tmp_path / "X.bin")
    p.W.tofile(tmp_path / "W.bin")
    p.labels.astype(np.int32).tofile(tmp_path / "labels.bin")
    r = subprocess.run([str(exe), str(tmp_path), str(p.n), str(p.h), str(p.v), str(p.ignore_index), "1"],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.split() == ["ok", "0"], (r.returncode, r.stdout, r.stderr)
    loss = float(np.fromfile(tmp_path / "loss.bin", dtype=np.float32)[0])
    lse = np.fromfile(tmp_path / "lse.bin", dtype=np.float32)
    dx = synth.bf16_bits_to_f32(np.fromfile(tmp_path / "dX.bin", dtype=np.uint16).reshape(p.n, p.h))
    dw = synth.bf16_bits_to_f32(np.fromfile(tmp_path / "dW.bin", dtype=np.uint16).reshape(p.v, p.h))
    ref = oracle.full_bf16(p)
    assert_loss(loss, ref["loss"])
    assert_lse(lse, ref["lse"])
    assert_grad(dx, ref["dX"], name="dX")
    assert_grad(dw, ref["dW"], name="dW")
