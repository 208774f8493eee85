import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libwql.so")


def has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def wql_lib():
    """The built library (built here if missing: nvcc cross-compiles without a GPU)."""
    from weight_quantized_linear_gb300 import build
    build.build()
    import weight_quantized_linear_gb300 as wql
    return wql
