import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running full-size case")


@pytest.fixture(scope="session")
def orc():
    import oracle

    oracle.build_oracle()
    return oracle


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library on a CUDA device; fails (never skips) when missing."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("gpu test collected on a machine without CUDA")
    import block_scaled_fp8_quant_gb300 as bfq

    bfq.load_library()
    return bfq
