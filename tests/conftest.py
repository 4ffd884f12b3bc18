import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_sessionstart(session):
    # Build the sm_103a library (nvcc cross-compiles without a GPU) and the
    # oracle before any test module imports them.
    from quantized_gemm_decode_02_b300 import build as qbuild
    qbuild.build()
    from oracle import oracle as o
    o.build()


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (runs the sm_103a kernels)")
    config.addinivalue_line("markers", "slow: large oracle work (full-size sampled parity)")


@pytest.fixture(scope="session")
def orc():
    from oracle import oracle as o
    o.build()
    return o


def pytest_collection_modifyitems(config, items):
    # Tests marked gpu are skipped (not failed) when no device is visible, so
    # that a CPU-only run of the whole directory stays green; the GPU machine runs
    # them with -m gpu.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
