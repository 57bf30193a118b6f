import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle

    return oracle.load()


@pytest.fixture(scope="session")
def moe_lib():
    """Build (if needed) and load libnvfp4moe.so; no GPU is touched."""
    from nvfp4_moe_decode_gb300 import _build
    import nvfp4_moe_decode_gb300 as m

    _build.build()
    return m.load()


@pytest.fixture(scope="session")
def cuda_dev(moe_lib):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return torch.device("cuda:0")
