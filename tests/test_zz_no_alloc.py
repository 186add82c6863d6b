"""vit_block_noalloc: the block with its scratch in the library's fixed device array.

Some callers cannot allocate device memory while the block runs (all memory reserved
up front, or allocation not allowed where the call is made). For them the library
offers vit_block_noalloc, which takes the same arguments as vit_block_ex but keeps its
scratch in one fixed 64 MiB array instead of a memory pool.

The array keeps whatever the previous call left in it. So each test first runs the
entry point on OTHER inputs (another seed, and one more sequence when that still fits,
which shifts every scratch region), and only then on the inputs it checks, twice in a
row. Both entry points run the same deterministic kernels on the same inputs, so the
result must equal vit_block_ex's bit for bit; a stale scratch byte read anywhere would
break that. A small case is also checked against the float64 oracle at the block
tolerances (3e-2 bf16, 2e-4 fp32). This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from vision_transformer_encoder_gb300 import api
from vision_transformer_encoder_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 64 << 20
TOL = {torch.bfloat16: 3e-2, torch.float32: 2e-4}
DTYPE = {torch.float32: 0, torch.bfloat16: 1}
VIT_ERR_UNSUPPORTED = -6


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


def _ex(d, H, eps, affine):
    return api.vit_block_ex(d.x, *d.weights(), H, eps, **(d.affine() if affine else {}))


def _fill_with_other_call(dev, shape, dtype, affine, eps):
    """Runs vit_block_noalloc on other inputs, checked bitwise against vit_block_ex, so
    the scratch array holds that call's values when the checked call starts."""
    N, T, D, H, F = shape
    for n_other in (N + 1, N):
        d = make_inputs(n_other, T, D, F, seed=29, dtype=dtype, affine=affine).to(device=dev)
        out = torch.full_like(d.x, float("nan"))
        rc = _noalloc(d, H, eps, out, affine)
        if rc == VIT_ERR_UNSUPPORTED and n_other > N:
            continue   # one more sequence does not fit the array on this path
        assert rc == 0, api.status_string(rc)
        ref = _ex(d, H, eps, affine)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), "other-input call differs from vit_block_ex"
        return
    raise AssertionError("unreachable")


@pytest.mark.parametrize("dtype,shape,affine", [
    (torch.bfloat16, (16, 197, 768, 12, 3072), False),   # ViT-B/16 block shape, 16 sequences
    (torch.bfloat16, (16, 197, 768, 12, 3072), True),
    (torch.float32, (8, 197, 192, 3, 768), False),       # ViT-Ti/16 block shape, fp32 path
])
def test_noalloc_equals_vit_block_ex_after_other_inputs(dtype, shape, affine):
    dev = _dev()
    N, T, D, H, F = shape
    eps = 1e-6
    _fill_with_other_call(dev, shape, dtype, affine, eps)
    d = make_inputs(N, T, D, F, seed=11, dtype=dtype, affine=affine).to(device=dev)
    ref = _ex(d, H, eps, affine)
    torch.cuda.synchronize()
    for call in range(2):
        out = torch.full_like(d.x, float("nan"))
        rc = _noalloc(d, H, eps, out, affine)
        assert rc == 0, api.status_string(rc)
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all(), "call %d left elements unwritten" % call
        assert torch.equal(out, ref), "call %d differs from vit_block_ex: max |diff| %g" % (
            call, (out.double() - ref.double()).abs().max().item())
    assert api.device_error() == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_matches_oracle(dtype):
    dev = _dev()
    N, T, D, H, F = 2, 197, 192, 3, 768
    eps = 1e-5
    _fill_with_other_call(dev, (N, T, D, H, F), dtype, True, eps)
    inp = make_inputs(N, T, D, F, seed=13, dtype=dtype, affine=True)
    d = inp.to(device=dev)
    for call in range(2):
        out = torch.full_like(d.x, float("nan"))
        rc = _noalloc(d, H, eps, out, True)
        assert rc == 0, api.status_string(rc)
        torch.cuda.synchronize()
        ref = oracle.vit_block(inp.x, *inp.weights(), H, eps, **inp.affine())
        err = np.abs(out.double().cpu().numpy() - ref).max()
        assert err <= TOL[dtype], "call %d differs from the oracle by %g" % (call, err)
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
    assert rc == VIT_ERR_UNSUPPORTED   # and nothing launched
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()
