import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from tests import tolerance  # noqa: E402


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_cuda = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_cuda = False
    if have_cuda:
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(autouse=True)
def _name_parity_checks(request):
    """Every parity check made during a test is recorded under the test's id."""
    tolerance.CURRENT_TEST = request.node.nodeid
    yield
    tolerance.CURRENT_TEST = ""


def pytest_terminal_summary(terminalreporter):
    """Totals of the parity checks: elements compared and elements beyond a strict 2 ulp, per dtype and
    output.  AR_PARITY_REPORT=<path> also writes every check's record there as JSON."""
    if not tolerance.REPORT:
        return
    tot = tolerance.summary()
    terminalreporter.section("parity checks against the oracle (strict 2-ulp report)")
    for k in sorted(tot):
        t = tot[k]
        terminalreporter.write_line(
            f"{k:>18}: {t['checks']:5d} checks, {t['elements']:13,d} elements, "
            f"{t['strict_violations']:6d} beyond a strict 2 ulp (each explained by the accumulation floor), "
            f"max {t['max_err_ulp']:.2f} ulp, least floor at a violation: {t['min_floor_ulp_at_violations']}")
    path = os.environ.get("AR_PARITY_REPORT")
    if path:
        with open(path, "w") as f:
            json.dump({"totals": tot, "checks": tolerance.REPORT}, f, indent=1)
