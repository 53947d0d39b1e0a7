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
    return sorted(set(re.findall(r"\b(flce_[a-z0-9_]+)\s*\(", text)))


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
    ws, wrc = flce.workspace_bytes, flce.workspace_bytes_rowchunk
    assert ws(256, 128, 1024) > 0
    # the workspace of forward / backward / fwd_bwd is independent of V (the logits are never stored)
    assert ws(8192, 2048, 32000) == ws(8192, 2048, 128256) == ws(8192, 2048, 7) == ws(8192, 2048, 1 << 30)
    # grows with N and H: one N x C bf16 chunk of G plus the N x H fp32 dX accumulator, O(N) words
    n, h = 8192, 2048
    assert ws(16384, 2048, 32000) > ws(8192, 2048, 32000)
    assert 2 * n * 8192 + 4 * n * h <= ws(n, h, 32000) <= 2 * n * 8192 + 4 * n * h + 400 * n + (1 << 20)
    n = 131072
    assert 2 * n * 4096 + 4 * n * 4096 <= ws(n, 4096, 131072) <= 2 * n * 4096 + 4 * n * 4096 + 400 * n + (1 << 20)
    # the row-chunk calls keep one row chunk of bf16 p~ and, with several chunks, an fp32 dW
    # accumulator; one chunk (N <= 4H) is never larger than two chunks' buffer plus it
    n, h, v = 8192, 2048, 32000
    one = wrc(n, h, v)
    assert 2 * n * v <= one <= 2 * n * v + 2 * n * h + 4 * n * 125 + (8 << 20)         # no accumulator
    assert one <= n * v + 4 * v * h + 2 * n * h + 4 * n * 125 + (8 << 20)              # <= the two-chunk layout
    two = wrc(2 * n, h, v)                                                                # N > 4H: two chunks
    assert two >= n * v * 2 + 4 * v * h and two <= n * v * 2 + 4 * v * h + 2 * n * h + 4 * n * 125 + (16 << 20)
    assert wrc(1024, 4096, 128256) < 300e6    # one chunk: no 2.1 GB fp32 accumulator
    assert wrc(8192, 2048, 64000) > wrc(8192, 2048, 32000)   # grows with V
    # invalid problems give 0
    for f in (ws, wrc):
        assert f(-1, 128, 10) == 0 and f(10, 12, 10) == 0 and f(10, 4, 10) == 0 and f(10, 128, 0) == 0
        assert f(0, 128, 10) == 256   # an empty batch needs only the status word
    # the largest workload stays under 4 GB of extra device memory on either path
    assert ws(131072, 4096, 131072) < 4e9 and wrc(131072, 4096, 131072) < 4e9


def test_shard_workspace_rules():
    sw = binding.shard_workspace_bytes
    n, h, v = 8192, 2048, 32000
    a = sw(n, h, v, 0, 16000)
    # independent of the shard's size and of V, no dX accumulator, N shard-local labels more
    assert a == sw(n, h, v, 16000, 16000) == sw(n, h, 4 * v, 7, 1000) > 0
    assert a <= flce.workspace_bytes(n, h, v) - 4 * n * h + 4 * n + 256
    # every layout places the header and the block partials first: a shard workspace serves
    # flce_shard_combine and flce_valid_count
    assert sw(n, h, v, 0, v) > 0
    for off, rows in ((-1, 10), (0, 0), (v - 5, 6), (v, 1)):
        assert sw(n, h, v, off, rows) == 0, (off, rows)


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
    """For random valid shapes both workspace sizes are positive, the bounded one does
    not depend on V, and a shard's is below the bounded one (the host-side layout
    arithmetic)."""
    import random
    rng = random.Random(1)
    for _ in range(2000):
        n = rng.choice([0, 1, 7, 255, 256, 257, rng.randint(1, 300000)])
        h = 8 * rng.randint(1, 2048)
        v = rng.randint(1, 300000)
        b, rc = flce.workspace_bytes(n, h, v), flce.workspace_bytes_rowchunk(n, h, v)
        assert b > 0 and rc > 0, (n, h, v, b, rc)
        assert b == flce.workspace_bytes(n, h, rng.randint(1, 300000))
        off = rng.randint(0, v - 1)
        sw = binding.shard_workspace_bytes(n, h, v, off, rng.randint(1, v - off))
        assert 0 < sw <= b + 4 * n + 256, (n, h, v, sw, b)


def test_shard_host_validation_without_gpu():
    L = flce.lib()
    P, S = binding.Problem, binding.VocabShard
    p = P(256, 128, 1000, -100, 0)
    z = 0x1000
    ws = 0x100000
    nb = binding.shard_workspace_bytes(256, 128, 1000, 0, 500)
    ok = S(0, 500)
    assert L.flce_shard_forward(ctypes.byref(p), None, z, z, z, z, z, ws, nb, None) == 1          # no shard
    assert L.flce_shard_forward(ctypes.byref(p), ctypes.byref(S(600, 500)), z, z, z, z, z, ws, nb, None) == 1
    assert L.flce_shard_forward(ctypes.byref(p), ctypes.byref(ok), 0x1008, z, z, z, z, ws, nb, None) == 3
    assert L.flce_shard_forward(ctypes.byref(p), ctypes.byref(ok), z, z, z, z, z, ws, 64, None) == 4
    assert L.flce_shard_backward(ctypes.byref(p), ctypes.byref(ok), z, z, z, z, None, 0x1004, z, ws, nb, None) == 3
    assert L.flce_shard_combine(ctypes.byref(p), 0, z, z, z, z, z, ws, nb, None) == 1             # no parts
    assert L.flce_shard_combine(ctypes.byref(p), 2, z, z, z, z, z, ws, 16, None) == 4
    assert L.flce_valid_count(ctypes.byref(p), z, None, ws, nb, None) == 1
    assert L.flce_f32_to_bf16(0x1004, z, 8, None) == 3
    assert L.flce_f32_to_bf16(None, z, 8, None) == 1
    assert L.flce_f32_to_bf16(None, None, 0, None) == 0
    assert L.flce_fwd_bwd_rowchunk(ctypes.byref(p), z, z, z, z, z, z, z, ws,
                                   flce.workspace_bytes(256, 128, 1000), None) in (4, 7)  # bounded size: too small


def test_debug_build_loads_and_exports_the_same_symbols():
    """libflce_debug.so (FLCE_DEBUG_CHECKS) is built beside the release library,
    exports every declared symbol and reports its checks; the release build does not."""
    lib = os.path.join(os.path.dirname(flce.lib_path()), "libflce_debug.so")
    assert os.path.exists(lib), "build() makes the debug library too"
    D = ctypes.CDLL(lib)
    for name in _declared():
        assert hasattr(D, name), name
    assert D.flce_debug_checks() == 1
    assert flce.lib().flce_debug_checks() == 0
    D.flce_selftest_bounds.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    assert D.flce_selftest_bounds(None, 256, None) == 1
    assert D.flce_selftest_bounds(ctypes.c_void_p(0x100010), 256, None) == 3
