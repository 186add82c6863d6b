"""The attention parity tests again, on the bf16 mma.sync kernel.

Head widths 64 and 80 run on the tcgen05 kernel by default; VIT_ATTN_TC=0 makes the
library use the mma.sync flash kernel for them instead. The choice is read per call
from the environment, so the stage tests are re-run in a child process with it set.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_attention_stages_on_mma_sync_kernel():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, VIT_ATTN_TC="0")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_gpu_stages.py"), "-k", "attention"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


def test_attention_stages_on_cta_pair_kernel():
    """Head width 64 runs on the single-CTA tcgen05 kernel by default; VIT_ATTN_PAIR=1
    selects the CTA-pair kernel."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, VIT_ATTN_PAIR="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_gpu_stages.py"), "-k", "attention"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
