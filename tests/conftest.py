import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libfpd.so")
    config.addinivalue_line("markers", "slow: oracle runs that take tens of seconds")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def full_weights():
    """The 4B-shape drafter's synthetic weights (seed 2000), drawn once per session (tens of seconds)."""
    import synth
    return synth.make_weights(synth.FULL, 2000)
