import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libflce")
    config.addinivalue_line("markers", "slow: long CPU-side oracle work (still run by -m gpu)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library on a GPU machine; fails loudly if it is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_lm_head_gb300 import _lib
    return _lib.load()


@pytest.fixture
def flce_opts():
    """Sets libflce run-time options for one test and restores them after it."""
    from chunked_lm_head_gb300 import _lib

    class _Opts:
        def __init__(self):
            self.saved = {}

        def set(self, name, value):
            if name not in self.saved:
                self.saved[name] = _lib.flce_get_option(name)
            _lib.flce_set_option(name, int(value))

    o = _Opts()
    yield o
    for name, value in o.saved.items():
        _lib.flce_set_option(name, value)
