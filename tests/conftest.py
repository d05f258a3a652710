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
