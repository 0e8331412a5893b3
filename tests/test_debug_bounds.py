"""The debug-bounds build (libsdpa_bwd_debug.so, compiled with SDPA_DEBUG_BOUNDS):
its kernels check every raw-pointer global access (bulk copies, reductions,
counters, direct stores) against the region it belongs to and report a
violation through the status word (SDPA_ERR_BOUNDS) instead of making it. A
child process loads that build and runs small shapes on every dQ route (the
reduction route, the ordered relay, the stored-dS route with a band or the full
rectangle, D_qk 192, GQA partial sets, a single row, ragged tails); no
violation may be reported and the gradients must match the oracle."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_bounds_build_reports_no_violation():
    from attention_backward_sdpa_gb300 import _build
    if not os.path.exists(_build.LIB_DEBUG) or _build.is_stale(_build.LIB_DEBUG):
        _build.build(debug=True)
    env = dict(os.environ, SDPA_BWD_LIBRARY=_build.LIB_DEBUG)
    r = subprocess.run([sys.executable, os.path.join(HERE, "_debug_bounds_child.py")], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "DEBUG_BOUNDS_OK" in r.stdout
