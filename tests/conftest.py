import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads")


@pytest.fixture(scope="session")
def built_lib():
    """Path of the in-tree C-ABI library, building it if it is missing."""
    from diffusion_transformer_qk_gb300 import build as b

    path = b.library_path()
    if not os.path.exists(path) or b.is_stale():
        b.build_library()
    return path


@pytest.fixture(scope="session")
def cuda_device():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")
