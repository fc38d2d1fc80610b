"""The bounds-checked build (libbeammoe_debug.so, every data-dependent index checked; a failed
check latches MOE_DEV_CHECK) on the small and odd-shape parity tests: it must give the same
results with no check failing. Runs them in a child process with BEAMMOE_LIBRARY=debug."""
import os
import subprocess
import sys

import pytest

from sparse_moe_layer_14_b300.build import build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_debug_build_small_and_odd_shapes():
    build(debug=True)
    env = dict(os.environ, BEAMMOE_LIBRARY="debug")
    sel = "tiny or odd or permute or combine or ffn or single_token or route_parity"
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_gpu_parity.py"), "-m", "gpu",
                        "-q", "-p", "no:cacheprovider", "-k", sel], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=1200)
    tail = "\n".join(r.stdout.strip().splitlines()[-5:])
    assert r.returncode == 0, tail + r.stderr[-2000:]
    assert " passed" in tail and "failed" not in tail
