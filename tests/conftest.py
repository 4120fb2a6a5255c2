import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture
def force_split():
    """Force the split-K segment count of this test's prefill calls (through the
    library's testing aid); the planner is restored afterwards."""
    import gated_delta_rule_24_gb300 as gdn
    yield lambda splits: gdn.testing_force_splits(int(splits))
    gdn.testing_force_splits(0)
