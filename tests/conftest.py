"""Shared pytest configuration.

``-m gpu`` tests need a CUDA device and the built ``libopam.so``; everything
else runs on the CPU (oracle pins, host-side argument checks, symbol exports,
multi-process host logic over gloo).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload checks")


@pytest.fixture(scope="session")
def oracle_mod():
    from oracle import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def cuda_lib():
    """Build (if stale) and load libopam.so; skip when no CUDA device exists."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from outer_product_associative_chunked_b300 import binding, build
    build.build()
    return binding
