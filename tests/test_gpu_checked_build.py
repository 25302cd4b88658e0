"""The bounds-checked build (every permuted row, TMA coordinate, TMEM column
and tile checked on the device, a failure latched as BEAM_ERR_DEVICE_CHECK)
latches nothing on valid calls of every expert format, at the batch sizes
that reach each kernel's edge cases: 16-row blocks, CTA-pair blocks whose
second half holds no valid row, several blocks per expert, the counting-sort
permutation and the tensor-core router."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_checked_build_latches_nothing_on_valid_calls():
    from group_limited_routed_gb300 import build
    build.build(checked=True)          # compiled once; later runs reuse it
    env = dict(os.environ, BEAM_MOE_DEVICE_CHECKS="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "_checked_forward.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    lines = [ln.split() for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 22, r.stdout
    bad = [ln for ln in lines if ln[2] != "0"]
    assert not bad, f"status latched by the checked build: {bad}"
