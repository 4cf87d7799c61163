"""The debug build (libtsa_debug.so, -DTSA_DEBUG): every path's small-shape
parity with the device-side checks on, and a check made to fail on purpose is
reported as TSA_ERR_DEVICE_CHECK (tests/debug_build_cases.py, run in a child
process so that the binding loads the debug library)."""
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_build_parity_and_checks():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fixed_state_recurrence_phi_b300 import build
    build.build(debug=True)
    env = dict(os.environ, TSA_DEBUG="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_build_cases.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    print(r.stdout)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "debug build ok" in r.stdout
