"""The fp32 block parity tests again, on the CUDA-core GEMM.

The fp32 block takes the 3xTF32 tensor-core GEMM by default; VIT_FP32_TC=0 keeps its
products on the CUDA-core kernel. The choice is read once per process, so the block tests
are re-run in a child process with the variable set; the child must report passed tests
and no skipped ones.
"""
import pytest

from _child import run_child_pytest

pytestmark = pytest.mark.gpu


def test_fp32_block_on_cuda_core_gemm():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    run_child_pytest("test_gpu_block.py", {"VIT_FP32_TC": "0"})
