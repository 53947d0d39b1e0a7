"""The C-ABI library loads on the CPU, exports every symbol include/flce.h
declares, and rejects bad arguments on the host (no GPU call is made)."""
import ctypes
import os
import re

import pytest

import lm_head_cross_gb300 as flce
from lm_head_cross_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "flce.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(flce_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    L = flce.lib()
    names = _declared()
    assert set(names) == set(binding.EXPORTED)
    for name in names:
        assert hasattr(L, name), name


def test_status_strings():
    for code in range(0, 10):
        assert flce.status_string(code)


def test_workspace_size_rules():
    ws, wmin = flce.workspace_bytes, flce.workspace_bytes_min
    assert wmin(256, 128, 1024) > 0
    # the minimum is independent of V (the logits are never stored)
    assert wmin(8192, 2048, 32000) == wmin(8192, 2048, 128256) == wmin(8192, 2048, 7)
    # grows with N
    assert wmin(16384, 2048, 32000) > wmin(8192, 2048, 32000)
    # the fused path's size is at least the minimum
    for n, h, v in ((256, 128, 1024), (8192, 2048, 32000), (32768, 4096, 151936)):
        assert ws(n, h, v) >= wmin(n, h, v)
    # the fused path keeps one row chunk of bf16 p~ and, with several chunks, an fp32 dW
    # accumulator; one chunk (N <= 4H) is never larger than two chunks' buffer plus it
    n, h, v = 8192, 2048, 32000
    one = ws(n, h, v)
    assert 2 * n * v <= one <= 2 * n * v + 2 * n * h + 4 * n * 125 + (8 << 20)         # no accumulator
    assert one <= n * v + 4 * v * h + 2 * n * h + 4 * n * 125 + (8 << 20)              # <= the two-chunk layout
    two = ws(2 * n, h, v)                                                                 # N > 4H: two chunks
    assert two >= n * v * 2 + 4 * v * h and two <= n * v * 2 + 4 * v * h + 2 * n * h + 4 * n * 125 + (16 << 20)
    assert ws(1024, 4096, 128256) < 300e6    # one chunk: no 2.1 GB fp32 accumulator
    # invalid problems give 0
    for f in (ws, wmin):
        assert f(-1, 128, 10) == 0 and f(10, 12, 10) == 0 and f(10, 4, 10) == 0 and f(10, 128, 0) == 0
        assert f(0, 128, 10) == 256   # an empty batch needs only the status word
    # the largest workload stays under 4 GB of extra device memory on either path
    assert ws(131072, 4096, 131072) < 4e9 and wmin(131072, 4096, 131072) < 4e9


def _call_forward(p, X=0x1000, W=0x2000, lab=0x3000, loss=0x4000, lse=0x5000, ws=0x100000, nbytes=None):
    L = flce.lib()
    if nbytes is None:
        nbytes = L.flce_workspace_bytes(ctypes.byref(p))
    return L.flce_forward(ctypes.byref(p), X, W, lab, loss, lse, ws, nbytes, None)


def test_host_side_validation_without_gpu():
    P = binding.Problem
    ok = P(256, 128, 1024, -100, 0)
    assert _call_forward(ok, X=None) == 1            # null pointer
    assert _call_forward(ok, X=0x1008) == 3          # misaligned X
    assert _call_forward(ok, lab=0x3002) == 3        # misaligned labels
    assert _call_forward(ok, ws=0x100010) == 3       # misaligned workspace
    assert _call_forward(ok, nbytes=16) == 4         # workspace too small
    assert _call_forward(P(256, 12, 1024, -100, 0)) == 2   # h % 8 != 0
    assert _call_forward(P(256, 128, 1024, -100, 7)) == 1  # bad reduction
    assert _call_forward(P(256, 128, 1024, -100, 0, 2, 0)) == 1  # bad shift
    assert _call_forward(P(256, 128, 1024, -100, 0, 1, 100)) == 1  # n not a multiple of seq_len
    assert _call_forward(P(-1, 128, 1024, -100, 0)) == 1   # negative row count
    empty = P(0, 128, 1024, -100, 0)
    assert _call_forward(empty, X=None, lab=None, lse=None, ws=None) == 1   # empty batch still needs a workspace
    assert _call_forward(empty, X=None, lab=None, lse=None, ws=0x100010) == 3
    assert _call_forward(empty, X=None, lab=None, lse=None, nbytes=16) == 4
    assert _call_forward(empty, loss=None) == 1       # the scalar loss is still written
    L = flce.lib()
    assert L.flce_selftest_timeout(None, 256, 1000, None) == 1
    assert L.flce_selftest_timeout(0x100010, 256, 1000, None) == 3
    assert L.flce_read_device_status(None, None) == 1


def test_python_binding_rejects_bad_reduction():
    with pytest.raises(ValueError):
        flce.workspace_bytes(10, 16, 10, reduction="avg")


def test_footprint_golden():
    """Logits footprint of the worked 128K x 128K case, as printed on the page."""
    import os
    from lm_head_cross_gb300 import logits_footprint_bytes
    path = os.path.join(os.path.dirname(__file__), "golden", "footprint_128k.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    assert rows
    for b, s, v, e, want, _ in rows:
        assert logits_footprint_bytes(int(b) * int(s), int(v), int(e)) == int(want)
    assert logits_footprint_bytes(131072, 131072, 2) == 32 << 30


def test_header_is_c_and_host_calls_link_from_c(tmp_path):
    """include/flce.h compiles as C99, and a C program linked against libflce.so
    runs its host-side calls (no GPU needed)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = flce.lib_path()
    exe = tmp_path / "abi_host"
    src = os.path.join(ROOT, "tests", "c", "abi_host.c")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), src, "-o", str(exe),
                        lib, "-Wl,-rpath," + os.path.dirname(lib)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.startswith("ok"), (r.stdout, r.stderr)


def test_workspace_sizes_on_random_shapes():
    """For random valid shapes the fastest-path workspace is never smaller than the
    minimum, and both are positive (the host-side layout arithmetic)."""
    import random
    rng = random.Random(1)
    for _ in range(2000):
        n = rng.choice([0, 1, 7, 255, 256, 257, rng.randint(1, 300000)])
        h = 8 * rng.randint(1, 2048)
        v = rng.randint(1, 300000)
        full, mn = flce.workspace_bytes(n, h, v), flce.workspace_bytes_min(n, h, v)
        assert 0 < mn <= full, (n, h, v, full, mn)
