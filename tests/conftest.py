import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libdetreduce.so")
    config.addinivalue_line("markers", "slow: full-size workload")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture
def replay(request):
    """The replay harness (tests/replay.py).  With DETR_REPLAY_LOG=<file> set,
    the fingerprint of every replayed call is appended to that file."""
    from replay import Replay
    r = Replay()
    yield r
    r.write_log(os.environ.get("DETR_REPLAY_LOG"), request.node.nodeid)
