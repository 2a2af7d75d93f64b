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
def cuda_lib():
    """The product library on cuda:0; the test fails (not skips) when the CUDA
    extension is missing on a GPU host."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_attention_26_gb300 as pd
    pd.load()  # raises if the library is not built
    return pd
