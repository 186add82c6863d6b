"""The GEMM parity tests again, on the single-CTA tensor-core kernel.

The library runs its GEMMs on the CTA-pair kernel by default; VIT_GEMM_PAIR=0 selects
the single-CTA kernel. The choice is read once per process, so the stage tests are
re-run in a child process with the variable set; the child must report passed tests
and no skipped ones.
"""
import pytest

from _child import run_child_pytest

pytestmark = pytest.mark.gpu


def test_linear_stages_on_single_cta_kernel():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    run_child_pytest("test_gpu_stages.py", {"VIT_GEMM_PAIR": "0"}, k="linear", timeout=600)


def test_fp32_block_on_cuda_core_gemm():
    """The fp32 block takes the 3xTF32 tensor-core GEMM by default; VIT_FP32_TC=0 keeps
    its products on the CUDA-core kernel."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    run_child_pytest("test_gpu_block.py", {"VIT_FP32_TC": "0"})
