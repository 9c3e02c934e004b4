import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running full-size case")


@pytest.fixture(scope="session")
def mhc_lib():
    """The built C-ABI library (built in-tree on first use)."""
    from manifold_constrained_hyper_mhc_gb300 import _build
    _build.build()
    import manifold_constrained_hyper_mhc_gb300 as mhc
    return mhc
