import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")


@pytest.fixture(scope="session")
def golden():
    import json
    with open(os.path.join(ROOT, "tests", "golden", "pages_printed_values.json")) as f:
        return json.load(f)


@pytest.fixture(autouse=True)
def _parity_record_current_test(request):
    import parity
    parity.CURRENT[0] = request.node.nodeid
    yield
    parity.CURRENT[0] = "(outside a test)"


def pytest_terminal_summary(terminalreporter):
    """The counts the parity checks kept: rows and tiles compared, how many fell under the
    near-tie rule, and the tail-miss counts of the tail-rate tests."""
    import parity
    if not parity.RECORD:
        return
    terminalreporter.section("parity counts (near-tie rule, tail misses)")
    for test, counts in sorted(parity.RECORD.items()):
        terminalreporter.write_line(f"{test}: " + ", ".join(f"{k}={v}" for k, v in counts.items()))


def pytest_sessionfinish(session):
    import json
    import parity
    path = os.environ.get("LMS_PARITY_RECORD")
    if path and parity.RECORD:
        with open(path, "w") as f:
            json.dump(parity.RECORD, f, indent=1, sort_keys=True)
