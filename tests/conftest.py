import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes)")
    config.addinivalue_line("markers", "fullsize_oracle(*names): full-size oracle requests the "
                            "test reads (computed in the background from the session's start)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def fullsize_oracle():
    """The background pool of full-size oracle runs (tests/fullsize_oracle.py)."""
    from fullsize_oracle import FullSizeOracle
    pool = FullSizeOracle(workers=min(16, os.cpu_count() or 1))
    yield pool
    pool.close()


@pytest.fixture(scope="session", autouse=True)
def _fullsize_oracle_early(request):
    """Queues every full-size oracle request of the selected tests before the
    first test runs, so that the oracle computes while the other tests use
    the GPU."""
    names = []
    for item in request.session.items:
        for m in item.iter_markers("fullsize_oracle"):
            names.extend(n for n in m.args if n not in names)
    if names:
        import torch
        if torch.cuda.is_available():
            pool = request.getfixturevalue("fullsize_oracle")
            from fullsize_oracle import BACKWARD_REQUESTS
            for n in names:
                if n in BACKWARD_REQUESTS:
                    pool.submit_backward(n)
                else:
                    pool.submit(n)
    yield
