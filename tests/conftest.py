import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long CPU-side oracle work")


@pytest.fixture(scope="session")
def attn():
    """The built library's Python binding (builds libattn.so in-tree if needed)."""
    from attention_attn_prefill_gb300 import build as _build
    _build.build()
    import attention_attn_prefill_gb300 as pkg
    pkg.lib()
    return pkg


@pytest.fixture()
def gpu(attn):
    """A CUDA device with the library loaded; checks no kernel recorded a device error."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("this test needs a CUDA GPU")
    attn.device_status(clear=True)
    yield torch.device("cuda:0")
    assert attn.device_status(clear=True) == 0, "a kernel recorded a device-side error"
