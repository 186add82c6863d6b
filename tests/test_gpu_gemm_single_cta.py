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


def test_fp32_block_on_cuda_core_gemm():
    """The fp32 block takes the 3xTF32 tensor-core GEMM by default; VIT_FP32_TC=0 keeps
    its products on the CUDA-core kernel."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, VIT_FP32_TC="0")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_gpu_block.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
