import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running (large oracle runs)")


@pytest.fixture(scope="session")
def tiny_weights():
    from prefill_only_decision_gb300 import configs, synth
    return synth.make_weights(configs.TINY)


@pytest.fixture(scope="session")
def tiny_requests():
    from prefill_only_decision_gb300 import configs, synth
    return synth.make_requests(configs.TINY)
