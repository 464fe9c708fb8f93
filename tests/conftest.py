import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_sessionstart(session):
    # compile libpsg.so and the oracle (no-ops when up to date; no GPU needed)
    from primitive_sm_graph_gb300 import build as B
    B.build()
    import oracle
    oracle.build()


@pytest.fixture(scope="session")
def O():
    import oracle
    oracle.build()
    return oracle
