"""The library built with its opt-in device self-checks (-DSMCSD_CHECKS: every check site tests
an index, a row, a copy size or an address before the access, and records a site code in the
workspace instead of making a bad access) runs the small parity cases and the status tests in a
process of its own, with the same results and statuses as the normal build. A site code showing
up (-101 and below) fails the parity cases' status checks."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CASES = [
    "tests/test_parity_sd.py::test_sd_tiny_fp32_many_seeds",
    "tests/test_parity_sd.py::test_sd_edge_shapes",
    "tests/test_parity_sd.py::test_sd_unaligned_rows_use_scalar_path",
    "tests/test_parity_sd.py::test_sd_masked_tokens",
    "tests/test_parity_sd.py::test_sd_ragged",
    "tests/test_parity_smc.py::test_reweight_small",
    "tests/test_parity_smc.py::test_ess_resample",
    "tests/test_parity_smc.py::test_remap",
    "tests/test_parity_smc.py::test_smc_step_32_steps",
    "tests/test_parity_smc.py::test_fused_step_equals_separate_calls",
    "tests/test_parity_pacer.py",
    "tests/test_parity_draft.py::test_draft_sample_small",
    "tests/test_faults_gpu.py",
]


def test_self_check_build_matches(smcsd):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from smc_reweight_resample_gb300 import build

    lib = build.build_checks()
    env = dict(os.environ, SMCSD_TEST_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p",
                        "no:cacheprovider", *CASES], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=1500)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and " failed" not in r.stdout
