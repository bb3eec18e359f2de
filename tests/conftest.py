import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def flash():
    """The CUDA library on a GPU machine (built in-tree if needed); skips without a GPU."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_89_gb300 import build
    build.build()
    from exact_attention_89_gb300 import flashattn
    flashattn.lib()
    return flashattn


@pytest.fixture(scope="session")
def built_lib():
    """libflashattn.so built on this machine (nvcc cross-compiles without a GPU)."""
    from exact_attention_89_gb300 import build
    build.build()
    from exact_attention_89_gb300 import flashattn
    return flashattn
