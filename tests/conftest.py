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
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def built_lib():
    """Build libsinkattn.so (nvcc cross-compiles without a GPU) and return its path."""
    from paged_gqa_attention_head_gb300 import build
    return build.build()


@pytest.fixture(scope="session")
def sa(built_lib):
    from paged_gqa_attention_head_gb300 import sinkattn
    sinkattn.load(built_lib)
    return sinkattn


@pytest.fixture(scope="session")
def cuda_dev():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")
