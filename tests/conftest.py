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


@pytest.fixture
def knob(monkeypatch):
    """Sets LORA_PUNICA_* tuning variables for one test: knob(NAME=value,
    ...) (None removes one).  The library reads its tuning variables once,
    so each call makes it read them again, and so does the end of the test
    after the environment is restored."""
    import expand_gemm_gb300 as eg

    def set_(**kv):
        for k, v in kv.items():
            if v is None:
                monkeypatch.delenv(k, raising=False)
            else:
                monkeypatch.setenv(k, str(v))
        eg.reload_options()
    yield set_
    monkeypatch.undo()
    eg.reload_options()
