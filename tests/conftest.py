import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libdq.so")
    config.addinivalue_line("markers", "slow: full-size case (minutes on the host oracle)")


@pytest.fixture(scope="session")
def orc():
    import oracle

    mutant = os.environ.get("DQ_ORACLE_MUTANT")
    if mutant:
        # a deliberately broken build of the oracle (tests/test_oracle_mutants.py
        # checks that the pins reject it); loaded instead of the real one
        oracle.build = lambda force=False: mutant
        oracle._lib = None
    else:
        oracle.build()
    return oracle
