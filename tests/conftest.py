import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def abi():
    """The C-ABI binding, building the library first when it is missing or stale."""
    from zero_sharded_optimizer_gb300 import build as b
    if shutil.which("nvcc") is None and not os.path.exists(b.LIB):
        pytest.skip("nvcc not available and library not built")
    b.build()
    from zero_sharded_optimizer_gb300 import abi as a
    return a


@pytest.fixture(scope="session")
def cuda(abi):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


@pytest.fixture(autouse=True)
def _guard_regions():
    """After every test, the sentinels around every buffer made with
    parity_util.guarded_empty are unchanged (no out-of-range device write)."""
    yield
    import parity_util
    try:
        if parity_util.guard_count():
            parity_util.check_guards()
    finally:
        parity_util.forget_guards()
