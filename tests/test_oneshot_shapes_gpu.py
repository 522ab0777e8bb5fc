"""Every one-shot launch shape (registers / shared memory / persistent blocks /
persistent blocks fed by bulk copies, units per thread, residual_out written
before or after the row barrier) gives oracle-parity results, and no kernel
gives up a bounded wait.  Each shape runs in a child process because the shape
override is read once per process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SHAPES = ["1:0:1", "2:0:0", "4:0:1", "8:0:0", "1:1:0", "2:1:1", "4:1:0", "8:1:1", "2:2:1", "4:2:0", "4:2:1",
          # persistent blocks fed by bulk copies: chunks per row : 3 : early : blocks per SM
          "1:3:0", "2:3:1", "4:3:0", "4:3:1:2", "8:3:0:2", "8:3:1", "2:3:1:1:2", "4:3:1:1:4",
          # one row split across a thread-block cluster: units per thread : 4 : early : cluster size
          "1:4:1:8", "2:4:0:4", "4:4:1:2", "1:4:0:2", "8:4:1:8"]


@pytest.mark.parametrize("shape", SHAPES)
def test_oneshot_shape_parity(shape):
    env = dict(os.environ, AR_ONESHOT_SHAPE=shape)
    res = subprocess.run([sys.executable, "-m", "tests.shape_child"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=600)
    assert res.returncode == 0 and "shape ok" in res.stdout, res.stdout[-3000:] + res.stderr[-3000:]
