"""The block parity tests again, on the LayerNorm-folded path.

VIT_LN_FOLD=1 makes the bf16 block fold both LayerNorms into the GEMMs that follow
them (row statistics plus per-column sums of the weights, applied in the GEMM
epilogue). The switch is read once per process, so the block tests and the
allocation-free entry point are re-run in a child process with it set.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("test_file", ["test_gpu_block.py", "test_zz_no_alloc.py"])
def test_block_on_ln_fold_path(test_file):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, VIT_LN_FOLD="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", test_file)],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
