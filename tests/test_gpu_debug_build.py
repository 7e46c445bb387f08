"""The bounds-checked build (libdprc_debug.so), the memory-safety check used in
place of compute-sanitizer.

Every computed global or distributed-shared-memory index of the streaming
kernels is checked before its access in that build; a failed check records
DPRC_DEVERR_BOUNDS with its source line and skips the access (no trap).  A
child process loads that build (DPRC_LIBRARY=debug) and runs small odd shapes
through every kernel family (tests/debug_build_cases.py): the one-launch
kernel with and without clusters and with many layers, the two-kernel path,
the +-1 projection, Hutch++, narrow layers both ways, the exact norm in both
forms, the fp32 path and the noise at an offset.  Every result must match
the oracle and no check may have failed.
"""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
RTOL = 1e-3


def test_bounds_checked_build_on_odd_shapes():
    from randomized_norm_clipping_gb300 import build
    if not os.path.exists(build.DEBUG_LIB_PATH):
        build.build(variants=("debug",))
    env = dict(os.environ, DPRC_LIBRARY="debug")
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_build_cases.py")], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["device_error"] == 0, res  # no index failed its check, no wait ran out
    for name, err in res["errors"].items():
        tol = 2e-5 if name == "noise_at" else RTOL
        assert err < tol, (name, err)
