import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def pytest_collection_finish(session):
    """Start the oracle's full-size solves (spawned processes, host cores)
    when the full-size oracle comparisons are selected and not all cached,
    so they run while the other GPU tests do."""
    if not any("test_fullsize_matches_oracle" in it.nodeid for it in session.items):
        return
    try:
        import torch
        if not torch.cuda.is_available():
            return
        import fullsize_oracle
        from workloads import build
    except Exception:
        return
    names = []
    for name in fullsize_oracle.NAMES:
        if not any(f"test_fullsize_matches_oracle[{name}]" in it.nodeid for it in session.items):
            continue
        if fullsize_oracle.load(name, fullsize_oracle.key_of(build(name))) is None:
            names.append(name)
    if names:
        pool, pending = fullsize_oracle.start(tuple(names))
        fullsize_oracle.PENDING = pending
        fullsize_oracle.POOL = pool
