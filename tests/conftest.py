import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
# The oracle-mutation test runs the pin tests against a planted-mistake copy of
# the oracle package placed in this directory.
if os.environ.get("EP_ORACLE_MUTANT_DIR"):
    sys.path.insert(0, os.environ["EP_ORACLE_MUTANT_DIR"])


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload (seconds of oracle time)")


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library, loaded through the Python binding (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import transformer_epilogue_gb300 as te
    te.load_library()
    return te


@pytest.fixture(autouse=True)
def _parity_record_name(request):
    """Parity comparisons record their errors under the running test's id."""
    from tests import _helpers
    _helpers.CURRENT_TEST[0] = request.node.nodeid
    yield
    _helpers.CURRENT_TEST[0] = "(outside a test)"


def pytest_terminal_summary(terminalreporter):
    """The literal max |gpu - oracle| of every parity comparison that ran,
    grouped by op kind and dtype (worst test named), and the largest ratio of
    an error to its tolerance.  EP_PARITY_REPORT=path also writes every record
    as JSON."""
    from tests import _helpers
    recs = _helpers.RECORDS
    if not recs:
        return
    tr = terminalreporter
    tr.section("parity: literal max |gpu - oracle| per op kind and dtype")
    groups = {}
    for test, kind, dt, n, mx, ratio in recs:
        g = groups.setdefault((kind, dt), dict(n=0, calls=0, max_abs=0.0, worst_abs="", max_ratio=0.0, worst_ratio=""))
        g["n"] += n
        g["calls"] += 1
        if mx >= g["max_abs"]:
            g["max_abs"], g["worst_abs"] = mx, test
        if ratio >= g["max_ratio"]:
            g["max_ratio"], g["worst_ratio"] = ratio, test
    for (kind, dt), g in sorted(groups.items()):
        tr.write_line(f"{kind:11s} {dt:9s} {g['calls']:5d} comparisons {g['n']:13d} elements  "
                      f"max |d| {g['max_abs']:.3e} ({g['worst_abs']})  "
                      f"max |d|/tol {g['max_ratio']:.3f} ({g['worst_ratio']})")
    path = os.environ.get("EP_PARITY_REPORT")
    if path:
        with open(path, "w") as f:
            json.dump([dict(test=t, kind=k, dtype=d, elements=n, max_abs=m, max_ratio=r)
                       for t, k, d, n, m, r in recs], f, indent=0)
