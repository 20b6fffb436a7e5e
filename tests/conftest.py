import os
import sys

import pytest

ROOT = os.path.dirname(os.path.abspath(__file__))
REPO = os.path.dirname(ROOT)
for p in (REPO, ROOT):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running oracle comparison")


@pytest.fixture(scope="session")
def oracle():
    import oracle as orc
    orc.build()
    return orc


@pytest.fixture(scope="session")
def oracle_lib(oracle):
    """Oracle built and the CUDA library built and loaded (GPU tests)."""
    import torch
    from w4_grouped_gemm_gb300 import build
    build.build()
    import w4_grouped_gemm_gb300 as lily
    lily.lib()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return oracle
