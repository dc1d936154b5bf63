import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)

# Parity margins recorded by the GPU tests: name -> {quantity: error / tolerance}.
# Printed in the terminal summary and, when TDT_PARITY_MARGINS names a file,
# written there as JSON.
_MARGINS = {}


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle

    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def record_margin():
    """record_margin(case, quantity, error, tolerance): keep error / tolerance
    (the larger one if the same case and quantity are recorded twice)."""

    def rec(case, quantity, error, tolerance):
        d = _MARGINS.setdefault(case, {})
        ratio = float(error) / float(tolerance)
        d[quantity] = max(ratio, d.get(quantity, 0.0))
        return ratio

    return rec


def pytest_terminal_summary(terminalreporter):
    if not _MARGINS:
        return
    terminalreporter.section("parity margins: largest error / tolerance (1.0 = at the limit)")
    for case in sorted(_MARGINS):
        parts = ", ".join("%s %.3g" % (q, r) for q, r in sorted(_MARGINS[case].items()))
        terminalreporter.write_line("%-34s %s" % (case, parts))
    path = os.environ.get("TDT_PARITY_MARGINS")
    if path:
        with open(path, "w") as f:
            json.dump(_MARGINS, f, indent=1, sort_keys=True)
