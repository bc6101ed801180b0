"""The bounds-checking debug library (libkvq_debug.so) over parity cases of
every kernel: outputs match the oracle and no device-side bounds check fails."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_library_bounds_checks_stay_clear():
    lib = os.path.join(os.path.dirname(HERE), "sub_byte_quantized_write_gb300", "libkvq_debug.so")
    if not os.path.exists(lib):
        pytest.fail("libkvq_debug.so is not built (build() makes it)")
    env = dict(os.environ, KVQ_BOUNDS_CHECK="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "bounds_debug_cases.py")], env=env, capture_output=True,
                       text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "BOUNDS-DEBUG OK" in r.stdout
