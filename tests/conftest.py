import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    # tests/test_oracle_mutants.py runs the pins in a child process against
    # a build of the oracle with a planted mistake
    mutant = os.environ.get("ORACLE_MUTANT_LIB")
    if mutant:
        oracle.load_library(mutant)
    return oracle
