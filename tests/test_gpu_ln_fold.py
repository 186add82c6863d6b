"""The block parity tests again, on the LayerNorm-folded path.

VIT_LN_FOLD=1 makes the bf16 block fold both LayerNorms into the GEMMs that follow
them (row statistics plus per-column sums of the weights, applied in the GEMM
epilogue). The switch is read once per process, so the block tests and the
allocation-free entry point are re-run in a child process with it set; the child must
report passed tests and no skipped ones.
"""
import pytest

from _child import run_child_pytest

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("test_file", ["test_gpu_block.py", "test_zz_no_alloc.py"])
def test_block_on_ln_fold_path(test_file):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    run_child_pytest(test_file, {"VIT_LN_FOLD": "1"})
