"""The debug build (libflce_debug.so, FLCE_DEBUG_CHECKS): on small problems
through every path — bounded and row-chunk fwd_bwd, top-k, vocabulary-shard
forward and backward — no index or TMA-coordinate check fires and the results
match the fp64 oracle; and its self-test shows a failing check is recorded in
the status word instead of trapping.  Runs in a child process that loads the
debug library instead of the release one."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

import lm_head_cross_gb300 as flce  # noqa: E402


def test_debug_build_runs_clean_on_small_problems():
    here = os.path.dirname(os.path.abspath(__file__))
    lib = os.path.join(os.path.dirname(flce.lib_path()), "libflce_debug.so")
    assert os.path.exists(lib)
    env = dict(os.environ, FLCE_LIB=lib)
    r = subprocess.run([sys.executable, os.path.join(here, "debug_checks_run.py")], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), (r.stdout[-2000:], r.stderr[-4000:])
