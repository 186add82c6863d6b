"""The GEMM parity tests again, on the single-CTA tensor-core kernel.

The library runs its GEMMs on the CTA-pair kernel by default; VIT_GEMM_PAIR=0 selects
the single-CTA kernel. The choice is read once per process, so the stage tests are
re-run in a child process with the variable set.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_linear_stages_on_single_cta_kernel():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, VIT_GEMM_PAIR="0")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_gpu_stages.py"), "-k", "linear"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
