import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: large sizes (still bounded to seconds on the GPU)")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle._load()
    return oracle


@pytest.fixture(scope="session")
def mmq_lib():
    """The C-ABI library (built in-tree by __graft_entry__.build() or on demand here)."""
    from quant_int8_mmq_gb300 import build as b
    b.build()
    import quant_int8_mmq_gb300 as m
    m.load()
    return m
