import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))
for p in (ROOT, TESTS):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU oracle checks")


@pytest.fixture(autouse=True)
def _parity_test_id(request):
    """Tags the parity metrics recorded during a test with its id."""
    import parity_util
    parity_util.CURRENT["test"] = request.node.nodeid
    yield
    parity_util.CURRENT["test"] = "?"


def pytest_terminal_summary(terminalreporter):
    """The parity metrics of every test that compared against the oracle: the
    per-slice maximum (the asserted bar), the element-by-element one (floor
    1e-3 of the slice maximum) and the per-row one, worst of each test."""
    import parity_util
    if not parity_util.RECORDS:
        return
    worst: dict[str, list[float]] = {}
    for test, sl, el, ro in parity_util.RECORDS:
        w = worst.setdefault(test, [0.0, 0.0, 0.0, 0])
        w[0] = max(w[0], sl)
        w[1] = max(w[1], el)
        w[2] = max(w[2], ro)
        w[3] += 1
    tr = terminalreporter
    tr.section("parity metrics (per slice | element by element, floor 1e-3 | per row)")
    for test, (sl, el, ro, n) in worst.items():
        tr.write_line(f"{sl:9.2e} | {el:9.2e} | {ro:9.2e}  ({n:3d}) {test}")
    sl_all = max(w[0] for w in worst.values())
    el_all = max(w[1] for w in worst.values())
    ro_all = max(w[2] for w in worst.values())
    tr.write_line(f"parity: {len(parity_util.RECORDS)} comparisons in {len(worst)} tests; "
                  f"worst per slice {sl_all:.2e}, element by element {el_all:.2e}, "
                  f"per row {ro_all:.2e}")
