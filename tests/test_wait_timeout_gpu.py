"""The bulk-copy-fed fused kernel's bounded waits, made to run out on purpose:
a test-only setting leaves one ring stage of every block unarmed (a stage
no copy will ever complete).  The kernel must give up after about a second,
wind down without hanging, report through ar_device_status, and leave the
CUDA context usable.  Runs in a child process because the setting and the
shape override are read once per process, by the test build of the library
(libar_test.so) only; the product library (libar.so) must ignore both."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bounded_waits_run_out_and_the_context_stays_usable():
    env = dict(os.environ, AR_TEST_STALL_STAGE="1", AR_ONESHOT_SHAPE="2:3:1:1:2")
    res = subprocess.run([sys.executable, "-m", "tests.timeout_child"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0 and "timeout ok" in res.stdout, res.stdout[-3000:] + res.stderr[-3000:]


def test_product_library_ignores_the_test_settings():
    env = dict(os.environ, AR_TEST_STALL_STAGE="1", AR_ONESHOT_SHAPE="2:3:1:1:2")
    res = subprocess.run([sys.executable, "-m", "tests.timeout_child", "product"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0 and "product library ignores" in res.stdout, res.stdout[-3000:] + res.stderr[-3000:]
