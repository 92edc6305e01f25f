import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

_MARGINS = []


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture
def margin(request):
    """margin(label, value, bound): record the error a parity check reached next to its bound.
    The values are listed at the end of the run (and written as JSON lines to the file named by
    ESM_PARITY_MARGINS, if set), so a passing run still shows how close each check came."""
    def record(label, value, bound):
        _MARGINS.append({"test": request.node.nodeid, "check": str(label), "value": float(value),
                         "bound": float(bound), "ok": bool(value < bound)})
        return value
    return record


def pytest_terminal_summary(terminalreporter):
    if not _MARGINS:
        return
    terminalreporter.section("parity margins (error reached / bound)")
    for m in _MARGINS:
        terminalreporter.write_line(f"{m['value']:.3e} / {m['bound']:.0e}  {m['check']}  [{m['test']}]")
    path = os.environ.get("ESM_PARITY_MARGINS")
    if path:
        with open(path, "a") as f:
            for m in _MARGINS:
                f.write(json.dumps(m) + "\n")
