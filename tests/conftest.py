import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); runs the CUDA path through the C-ABI")
    config.addinivalue_line("markers", "slow: full-size workload (minutes of oracle time)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library, loaded; skips only if no GPU is present."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_deltanet_linear_16_gb300 as gdn
    gdn.load()
    return gdn
