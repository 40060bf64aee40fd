"""Test configuration: the `gpu` marker and shared fixtures.

`-m "not gpu"` runs the CPU oracle against its pins, the host-side logic and the C-ABI
export/validation checks; `-m gpu` runs the parity tests that call the CUDA library through
the C ABI and compare it with the oracle.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def cuda_lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_moe_router_gb300 import build, capi
    build.build()
    return capi.load_library()
