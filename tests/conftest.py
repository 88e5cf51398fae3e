import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload; minutes of oracle time")


def pytest_terminal_summary(terminalreporter):
    """Worst max-normalised and floored elementwise relative errors of each test's comparisons; also
    written as JSON to the file LA_PARITY_REPORT names, when set."""
    from tests.helpers import ERRORS
    if not ERRORS:
        return
    worst = {}
    for test, e, el in ERRORS:
        a, b = worst.get(test, (0.0, 0.0))
        worst[test] = (max(a, e), max(b, el))
    tr = terminalreporter
    tr.section("parity errors (max-normalised | elementwise, floor 1e-6 max|ref|)")
    for test, (e, el) in sorted(worst.items()):
        tr.write_line(f"{e:10.3e} | {el:10.3e}  {test}")
    path = os.environ.get("LA_PARITY_REPORT")
    if path:
        import json
        with open(path, "w") as f:
            json.dump({t: {"max_normalised": e, "elementwise_floored": el} for t, (e, el) in worst.items()}, f,
                      indent=1, sort_keys=True)
