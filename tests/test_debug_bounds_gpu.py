"""The library built with device bounds checks (libmoe_ep_debug.so,
MOE_DEBUG_BOUNDS), a stand-in for a memory checker (compute-sanitizer is
closed on this pool): every row index a kernel computes is checked against
its buffer before the access. Run in child processes that load that build
(MOE_EP_DEBUG_BOUNDS=1): small layers in every dispatch mode must match the
oracle with a clean status, and an expert offset overwritten on the host
with a row past the receive buffer must be caught (MOE_STATUS_BOUNDS, the
access skipped) instead of written."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def _run(case):
    import importlib
    build = importlib.import_module("combine_top_histogram_gb300.build")
    build.build(variants=("debug",))
    env = dict(os.environ, MOE_EP_DEBUG_BOUNDS="1")
    out = subprocess.run([sys.executable, os.path.join(HERE, "debug_bounds_case.py"), case],
                         capture_output=True, text=True, timeout=600, env=env)
    assert out.returncode == 0, out.stdout[-3000:] + out.stderr[-3000:]
    return out.stdout


def test_debug_build_clean_layers_every_mode(gpu):
    assert _run("clean").count(" ok") == 6


def test_debug_build_catches_a_row_past_the_buffer(gpu):
    assert "corrupt ok" in _run("corrupt")
