"""The bounds-checking build (HLA2_DEBUG) on the GPU.

Builds the debug variant of the library (global-memory indices of the float32, mma.sync,
scan, decode and tcgen05 first-order scan kernels checked against their buffers; a failed
check records a site and skips the access, nothing traps), then runs small odd shapes on it
in a fresh process (d = 16, n equal to the chunk width, ragged tails, every path of the
forward, the backward and the decode steps), each against the float64 oracle, and requires
the debug words to stay clean.  The recording itself is checked with a failing check that
guards no access.
"""
import os
import subprocess
import sys

import pytest

from chunked_scan_mixer_gb300 import build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_small_odd_shapes_leave_the_debug_words_clean():
    lib = build.build(debug=True)
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_build_check.py"), lib], capture_output=True,
                       text=True, timeout=1200)
    assert r.returncode == 0 and "DEBUG_BUILD_OK" in r.stdout, (r.stdout[-3000:], r.stderr[-3000:])
