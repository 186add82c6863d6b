"""Device-side failure detection without a GPU fault: a bounded wait made to run out.

Every wait in the library's kernels gives up after a limit (or at once when another part
of the kernel has set its abort flag) and records a bit in the device error word, which
the host reads with vit_device_error. vit_selftest_wait runs that same wait on a barrier
that nothing completes; the GPU must stay usable afterwards.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from vision_transformer_encoder_gb300 import api
from vision_transformer_encoder_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

SELFTEST_BIT = 1 << 5


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def test_wait_runs_out_and_is_reported():
    _dev()
    assert api.device_error() == 0
    t0 = time.time()
    api.selftest_wait()
    word = api.device_error()          # synchronises: the kernel has ended by its limit
    elapsed = time.time() - t0
    assert word == SELFTEST_BIT
    assert 0.2 < elapsed < 60, elapsed  # the limit is about two seconds of SM clock
    assert api.device_error() == 0      # reading clears the word


def test_abort_flag_ends_the_wait_at_once():
    _dev()
    t0 = time.time()
    api.selftest_wait(abort_first=True)
    word = api.device_error()
    assert word == SELFTEST_BIT
    assert time.time() - t0 < 0.5


def test_gpu_usable_after_a_wait_ran_out():
    d = _dev()
    api.selftest_wait(abort_first=True)
    assert api.device_error() == SELFTEST_BIT
    inp = make_inputs(2, 5, 8, 16, seed=3, dtype=torch.float32)
    di = inp.to(device=d)
    out = api.vit_block(di.x, *di.weights(), 2, 1e-5)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    ref = oracle.vit_block(inp.x, *inp.weights(), 2, 1e-5)
    assert float(np.abs(out.double().cpu().numpy() - ref).max()) <= 2e-4
