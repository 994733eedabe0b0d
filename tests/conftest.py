import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (parity against the oracle)")
    config.addinivalue_line("markers", "slow: long CPU test")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def built_lib():
    """Path of libpagedattn.so, compiled in-tree for sm_103a if stale (nvcc works without a GPU)."""
    from paged_kv_cache_257_gb300 import build
    return build.build()


@pytest.fixture(scope="session")
def pa(built_lib):
    import paged_kv_cache_257_gb300 as pa_mod
    return pa_mod


@pytest.fixture(scope="session")
def cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    return torch.device("cuda:0")


@pytest.fixture
def kernel(request, pa):
    """Pin the tensor-core decode kernel ("cta" or "warp", from the test's
    parameter) for one test, then restore the process setting."""
    prev = pa.set_decode_kernel(request.param)
    yield request.param
    pa.set_decode_kernel(prev)
