import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, built in-tree if needed; the test fails if it is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu test collected on a host without a GPU")
    import gemm_epilogue_02_gb300 as tg
    tg.load()
    return tg
