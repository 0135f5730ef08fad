import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    # GPU tests fail loudly (not skip) when CUDA is missing, so a CPU-only run
    # must deselect them with -m "not gpu"; nothing here silently skips them.
    return None


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library through its Python binding (built on first use)."""
    import block_causal_masked_gb300 as bd
    return bd
