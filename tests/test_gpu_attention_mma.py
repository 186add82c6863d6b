"""The attention parity tests again, on the kernels that are not the default.

Head widths 64 and 80 run on tcgen05 kernels by default: for head width 64 and at most
224 tokens the whole-row kernel (all keys in one S tile), otherwise the key-streaming
kernel. VIT_ATTN_WHOLE_PAIR=1 selects the whole-row kernel on CTA pairs,
VIT_ATTN_TC=0 the mma.sync flash kernel, VIT_ATTN_WHOLE=0 the streaming kernel at every
length, and VIT_ATTN_PAIR=1 (with VIT_ATTN_WHOLE=0) the streaming CTA-pair kernel.
The switches are read once per process, so the stage tests are re-run in a child
process with them set.
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
    env = dict(os.environ, VIT_ATTN_PAIR="1", VIT_ATTN_WHOLE="0")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_gpu_stages.py"), "-k", "attention"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


def test_attention_stages_on_key_streaming_kernel():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, VIT_ATTN_WHOLE="0")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_gpu_stages.py"), "-k", "attention"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


def test_attention_stages_on_cta_pair_whole_row_kernel():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, VIT_ATTN_WHOLE_PAIR="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_gpu_stages.py"), "-k", "attention"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
