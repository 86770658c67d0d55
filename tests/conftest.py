import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) and the CUDA library")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")

TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


@pytest.fixture(scope="session")
def lib():
    """The CUDA library, built in-tree; GPU tests need an sm_103 device."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tensor_transformer_mlp_tmem_gb300 import _build
    import tensor_transformer_mlp_tmem_gb300 as tp
    _build.build()
    torch.cuda.init()
    return tp.load_library()
