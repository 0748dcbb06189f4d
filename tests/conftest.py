import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running oracle comparison")


@pytest.fixture(scope="session")
def lib():
    """The CUDA library, built in-tree; GPU tests need it and a device."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from text_embedding_encoder_gb300 import binding
    return binding.load()
