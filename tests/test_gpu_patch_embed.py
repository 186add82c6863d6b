"""Parity of vit_patch_embed (patchify, projection with bias, CLS row, positions) with the
float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from vision_transformer_encoder_gb300 import api

pytestmark = pytest.mark.gpu

# bf16: inputs exact in the oracle; the projection accumulates in fp32 and the tokens are
# rounded once to bf16: |token| <= ~5 gives 2^-9 * 5 = 1e-2, plus fp32 accumulation error
TOL = {torch.bfloat16: 1.6e-2, torch.float32: 2e-4, torch.float64: 1e-11}


def _inputs(N, C, Hi, Wi, P, D, seed, dtype, with_cls=True):
    g = torch.Generator().manual_seed(seed)
    K, T = C * P * P, (Hi // P) * (Wi // P) + (1 if with_cls else 0)
    im = torch.randn(N, C, Hi, Wi, generator=g)
    w = torch.randn(K, D, generator=g) / K ** 0.5
    b = torch.randn(D, generator=g) * 0.02
    cls = torch.randn(D, generator=g) * 0.02 if with_cls else None
    pos = torch.randn(T, D, generator=g) * 0.02
    cv = lambda t: None if t is None else t.to(dtype)
    return cv(im), cv(w), cv(b), cv(cls), cv(pos)


def _check(shape, order, dtype, with_cls=True, with_pos=True):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    N, C, Hi, Wi, P, D = shape
    im, w, b, cls, pos = _inputs(N, C, Hi, Wi, P, D, seed=sum(shape) + order, dtype=dtype, with_cls=with_cls)
    if not with_pos:
        pos = None
    d = torch.device("cuda:0")
    mv = lambda t: None if t is None else t.to(d)
    out = api.vit_patch_embed(mv(im), P, mv(w), b=mv(b), cls=mv(cls), pos=mv(pos), order=order)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    ref = oracle.patch_embed(im, P, w, b, cls=cls, pos=pos, order=order)
    got = out.double().cpu().numpy()
    assert got.shape == ref.shape
    err = float(np.abs(got - ref).max())
    assert err <= TOL[dtype], err


@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.float64])
def test_vit_b16_front_end(order, dtype):
    _check((2, 3, 224, 224, 16, 768), order, dtype)


@pytest.mark.parametrize("shape", [(3, 3, 32, 48, 16, 64), (2, 1, 28, 28, 14, 40), (1, 3, 56, 28, 14, 96),
                                   (2, 4, 8, 8, 4, 16), (1, 3, 32, 32, 8, 42)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_odd_shapes(shape, dtype):
    _check(shape, 0, dtype)
    _check(shape, 1, dtype, with_cls=False)


def test_without_cls_and_positions():
    _check((2, 3, 64, 64, 16, 128), 0, torch.bfloat16, with_cls=False, with_pos=False)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_many_rows(dtype):
    # 140000 patch rows and 70000 images: more than one 65535-wide grid dimension in both
    # the patch gather and the token assembly
    _check((70000, 1, 16, 8, 8, 16), 0, dtype)
