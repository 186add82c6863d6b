"""The attention parity tests again, on the kernels that are not the default.

Head widths 64 and 80 run on tcgen05 kernels by default: for head width 64 and at most
224 tokens the whole-row kernel (all keys in one S tile), otherwise the key-streaming
kernel. VIT_ATTN_TC=0 selects the mma.sync flash kernel and VIT_ATTN_WHOLE=0 the streaming kernel
at every length. For
fp32, head width 64 and T <= 224 run on the 3xTF32 tensor-core kernel by default;
VIT_ATTN_F32_TC=0 keeps them on the CUDA-core kernel.
The switches are read once per process, so the stage tests are re-run in a child
process with them set; the child must report passed tests and no skipped ones.
"""
import pytest

from _child import run_child_pytest

pytestmark = pytest.mark.gpu

VARIANTS = {
    "mma_sync": {"VIT_ATTN_TC": "0"},
    "key_streaming": {"VIT_ATTN_WHOLE": "0"},
    "fp32_cuda_cores": {"VIT_ATTN_F32_TC": "0"},
}


@pytest.mark.parametrize("variant", sorted(VARIANTS))
def test_attention_stages_on_other_kernel(variant):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    run_child_pytest("test_gpu_stages.py", VARIANTS[variant], k="attention", timeout=600)
