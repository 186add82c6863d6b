"""vit_block_noalloc: the block with its scratch in the library's fixed device array.

Some callers cannot allocate device memory while the block runs (all memory reserved
up front, or allocation not allowed where the call is made). For them the library
offers vit_block_noalloc, which takes the same arguments as vit_block_ex but keeps its
scratch in one fixed 64 MiB array instead of a memory pool. These tests call it
through the C ABI and compare it with vit_block_ex on the same inputs, twice in a row
(the array keeps the previous call's contents), within the tolerances the other block
tests use. This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from vision_transformer_encoder_gb300 import api
from vision_transformer_encoder_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 << 20
TOL = {torch.bfloat16: 3e-2, torch.float32: 2e-4}
DTYPE = {torch.float32: 0, torch.bfloat16: 1}


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(d, H, eps, out, affine):
    lib = api.load_library()
    aff = [d.ln1_g, d.ln1_b, d.ln2_g, d.ln2_b, d.b1, d.b2] if affine else [None] * 6
    N, T, D = d.x.shape
    F = d.w_mlp1.shape[1]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.vit_block_noalloc(_p(d.x), *[_p(w) for w in d.weights()], *[_p(t) for t in aff],
                                 N, T, D, F, H, float(eps), DTYPE[d.x.dtype], _p(out), stream)


@pytest.mark.parametrize("dtype,shape,affine", [
    (torch.bfloat16, (16, 197, 768, 12, 3072), False),   # ViT-B/16 block shape, 16 sequences
    (torch.bfloat16, (16, 197, 768, 12, 3072), True),
    (torch.float32, (8, 197, 192, 3, 768), False),       # ViT-Ti/16 block shape, CUDA cores
])
def test_noalloc_matches_vit_block_twice(dtype, shape, affine):
    dev = _dev()
    N, T, D, H, F = shape
    eps = 1e-6
    inp = make_inputs(N, T, D, F, seed=11, dtype=dtype, affine=affine)
    d = inp.to(device=dev)
    ref = api.vit_block_ex(d.x, *d.weights(), H, eps, **(d.affine() if affine else {}))
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full_like(d.x, float("nan"))
        rc = _noalloc(d, H, eps, out, affine)
        assert rc == 0, api.status_string(rc)
        torch.cuda.synchronize()
        got = out.double().cpu().numpy()
        assert np.isfinite(got).all(), "call %d left elements unwritten" % call
        err = np.abs(got - ref.double().cpu().numpy()).max()
        assert err <= TOL[dtype], "call %d differs from vit_block_ex by %g" % (call, err)
    assert api.device_error() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch():
    dev = _dev()
    # 64 sequences of the ViT-B/16 block need 64*197*15360 bytes (> 64 MiB) of scratch
    N, T, D, H, F = 64, 197, 768, 12, 3072
    assert N * T * (12 * D + 2 * F) > SCRATCH_BYTES
    inp = make_inputs(N, T, D, F, seed=12, dtype=torch.bfloat16)
    d = inp.to(device=dev)
    out = torch.full_like(d.x, float("nan"))
    rc = _noalloc(d, H, 1e-6, out, False)
    assert rc == -6   # VIT_ERR_UNSUPPORTED, and nothing launched
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()
