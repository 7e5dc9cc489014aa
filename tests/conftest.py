import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def oracle():
    import oracle as _oracle
    _oracle.build()
    return _oracle


# Tolerances: bf16 inputs with fp32 accumulation, fp32 inputs, and exact work
# for integer / byte paths.  The bf16 max bound is read relative to
# max(1, |ref|): a bf16 output of magnitude 4..8 lies up to 2^-6 = 0.0156 away
# from the exact value after rounding alone, so an absolute 1e-2 cannot hold
# there even for an exact computation; below 1 the bound is absolute.
BF16_MAX = 1e-2
BF16_MEAN = 1e-3
BF16_LSE = 1e-3
F32_TOL = 1e-5


@pytest.fixture(scope="session")
def cplib():
    """libcp built in-tree (build() on the machine running the tests)."""
    from context_parallelism_02_gb300 import _lib, build
    build.build()
    return _lib.load()


@pytest.fixture(scope="session")
def cuda_dev(cplib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    return torch.device("cuda:0")
