import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size cases (still bounded to a few minutes)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, built and loaded; the test fails loudly if it is missing."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("gpu-marked test run without a visible CUDA device")
    import online_softmax_attention_tiled_gb300 as oa

    oa.load()
    return oa
