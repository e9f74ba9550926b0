"""GPU: the bounds-checking build (libftmoe_checks.so, FTMOE_CHECKS=1), the stand-in for a
memory checker.  A child process loads it (FTMOE_LIBRARY=checks) and runs
tests/checks_run.py: small layers on every expert-FFN path with status 0 and oracle
parity, then host-made malformed offsets / sorted_pair tables whose bad entries are
reported in the device status word and skipped while every other row stays correct.
No case reads or writes out of bounds: the checks turn each bad index into an in-range one."""
import os
import subprocess
import sys

import pytest

from tests._util import ensure_built

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checks_build_parity_and_malformed_tables(cuda_device):
    ensure_built()
    from quantized_expert_ffn_layer_b300.build import build
    build(checks=True)
    env = dict(os.environ, FTMOE_LIBRARY="checks")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checks_run.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "checks ok" in r.stdout
