"""The MOE_DEBUG library: its device-side bounds checks of the row indices
taken from row maps report nothing on correct inputs, and every path still
matches the CPU oracle on small shapes (the checks of smoke(): BF16 forward
and backward, the fused gate, MXFP8 forward and backward)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_debug_build_passes_smoke_without_bounds_errors():
    code = ("import __graft_entry__ as g, moe_expert_dispatch_gb300 as m; "
            "assert m.LIB_PATH.endswith('libmoe_gb300_debug.so'), m.LIB_PATH; "
            "g.smoke(); print('debug smoke ok')")
    env = dict(os.environ, MOE_GB300_DEBUG="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "debug smoke ok" in r.stdout
