import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running case")


@pytest.fixture(scope="session")
def orc():
    import oracle

    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def smcsd():
    """The CUDA library, built in-tree if stale, loaded through its binding (GPU tests only)."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from smc_reweight_resample_gb300 import _binding, build

    alt = os.environ.get("SMCSD_TEST_LIB")  # another build of the library (the self-check build)
    if alt:
        _binding.load(alt)
    else:
        build.build()
        _binding.load()
    return _binding
