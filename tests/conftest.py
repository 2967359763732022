import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def orc():
    from oracle import oracle
    src = os.environ.get("MOE_ORACLE_MUTANT_SRC")
    if src:
        # A mutated copy of the oracle's C source, compiled next to it
        # (tests/test_oracle_mutants.py runs the pins against such copies).
        oracle._SRC = src
        oracle._SO = os.path.join(os.path.dirname(src), "libmoe_oracle.so")
    oracle.build()
    return oracle
