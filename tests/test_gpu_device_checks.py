"""The device-side index checks: the library built with -DSGEMM_DEVICE_CHECKS
(TMA box coordinates inside their tensors, stream-K workspace slots and
arrival counters inside their buffers, cluster split-K slots inside the
owner's shared memory; a failed check sets a status bit and replaces the
index with one in range -- never a trap, an assert or an out-of-range
access) runs a parity sweep with every check passing, and reports a
provoked failure.  The checked build loads in a child process of its own
(tests/device_checks_sweep.py), so the release build of this process is not
involved."""
import os
import subprocess
import sys

import pytest

from dense_fp32_matrix_09_gb300 import build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_sweep():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    lib = build.build(checked=True)
    env = dict(os.environ, SGEMM_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-m", "tests.device_checks_sweep"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "every check passing" in r.stdout
