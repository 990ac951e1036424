import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    # GPU tests run only where a GPU is present; on a CPU host `-m gpu` selects them
    # and they fail loudly instead of silently passing.
    pass


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.load()


@pytest.fixture
def launch_options():
    """Force the library's launch choices for one test (specdec_set_launch_options): call it with
    kernel=, ctas_per_request=, schedule=, wait_limit_us= and/or split_requests= (None: the library
    decides). Every
    choice is put back to automatic afterwards."""
    from speculative_decoding_verification_specdec_gb300 import _native

    state = {"kernel": None, "ctas_per_request": None, "schedule": None, "wait_limit_us": None,
             "split_requests": None}

    def set_(**kw):
        state.update(kw)
        _native.set_launch_options(**state)

    set_()
    yield set_
    _native.set_launch_options()
