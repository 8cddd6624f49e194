import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload, tens of seconds")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.default()


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library, built here if missing; skips without a GPU."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_deferred_finalize_gb300 import build
    build.build_library()
    import moe_deferred_finalize_gb300 as mf
    return mf
