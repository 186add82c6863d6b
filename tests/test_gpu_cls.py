"""Parity of the CLS-only last block (vit_block_cls) and the stack with a CLS readout
(vit_encoder_cls) with the float64 oracle, on the bf16, fp32 and fp64 paths."""
import numpy as np
import pytest
import torch

import oracle
from vision_transformer_encoder_gb300 import api
from vision_transformer_encoder_gb300.inputs import make_encoder_inputs

pytestmark = pytest.mark.gpu

# bf16: the same stage roundings as the whole block (xn, k/v/q, o, yn, h in bf16, y in
# fp32) and the final rounding of out: the block's bound. fp32 path (3xTF32 products, fp32
# softmax) and fp64 as for the block.
TOL = {torch.bfloat16: 3e-2, torch.float32: 2e-4, torch.float64: 1e-10}


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _to(lay, d):
    return {k: (v.to(d) if v is not None else None) for k, v in lay.items()}


def _block_case(N, T, D, H, F, dtype, seed, affine=True, biases=True):
    x, layers, _, _ = make_encoder_inputs(N, T, D, F, 1, seed=seed, affine=affine, biases=biases, dtype=dtype)
    return x, layers[0]


def _oracle_block(x, lay, H, eps, rows=None):
    xs = x if rows is None else x[rows]
    return oracle.vit_block_cls(xs, *[lay[k] for k in ("w_q", "w_k", "w_v", "w_o", "w_mlp1", "w_mlp2")], H, eps,
                                **{k: lay.get(k) for k in oracle.LAYER_KEYS[6:]})


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32, torch.float64])
@pytest.mark.parametrize("shape", [
    (2, 5, 8, 2, 16),          # tiny: the CUDA-core path for every dtype
    (4, 197, 192, 3, 768),     # ViT-Ti/16
    (3, 33, 96, 3, 192),       # head width 32
    (2, 300, 128, 2, 256),     # more keys than threads
    (5, 1, 64, 1, 128),        # one token
    (2, 50, 320, 4, 640),      # head width 80
])
def test_block_cls_matches_oracle(dtype, shape):
    d = _dev()
    N, T, D, H, F = shape
    x, lay = _block_case(N, T, D, H, F, dtype, seed=sum(shape))
    out = api.vit_block_cls(x.to(d), _to(lay, d), H, 1e-6)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    assert out.shape == (N, D)
    got = out.double().cpu().numpy()
    assert np.isfinite(got).all()
    err = float(np.abs(got - _oracle_block(x, lay, H, 1e-6)).max())
    print("cls block %s %s max err %.3g" % (dtype, shape, err))
    assert err <= TOL[dtype]


def test_block_cls_without_affine_or_biases():
    d = _dev()
    x, lay = _block_case(3, 197, 192, 3, 768, torch.bfloat16, seed=5, affine=False, biases=False)
    lay = {k: v for k, v in lay.items() if v is not None}
    got = api.vit_block_cls(x.to(d), _to(lay, d), 3, 1e-6).double().cpu().numpy()
    assert float(np.abs(got - _oracle_block(x, lay, 3, 1e-6)).max()) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_block_cls_vit_b16_full_size(dtype):
    # the bench's workload: 256 sequences of ViT-B/16; the oracle recomputes four of them
    # (sequences are independent, which the oracle's pins establish)
    d = _dev()
    N, T, D, H, F = 256, 197, 768, 12, 3072
    x, lay = _block_case(N, T, D, H, F, dtype, seed=11)
    got = api.vit_block_cls(x.to(d), _to(lay, d), H, 1e-6).double().cpu().numpy()
    rows = [0, 1, N // 2, N - 1]
    ref = _oracle_block(x, lay, H, 1e-6, rows=rows)
    err = float(np.abs(got[rows] - ref).max())
    print("cls block B/16 %s max err %.3g" % (dtype, err))
    assert np.isfinite(got).all()
    assert err <= TOL[dtype]


@pytest.mark.parametrize("shape", [(64, 577, 1024, 16, 4096), (32, 1025, 1280, 16, 5120)])
def test_block_cls_vit_l_and_h_full_size(shape):
    # ViT-L/16 at 384 px (577 tokens) and ViT-H/14 at 448 px (1025 tokens, head width 80):
    # the full batches, four sequences recomputed by the oracle
    d = _dev()
    N, T, D, H, F = shape
    x, lay = _block_case(N, T, D, H, F, torch.bfloat16, seed=T)
    got = api.vit_block_cls(x.to(d), _to(lay, d), H, 1e-6).double().cpu().numpy()
    rows = [0, 1, N // 2, N - 1]
    err = float(np.abs(got[rows] - _oracle_block(x, lay, H, 1e-6, rows=rows)).max())
    print("cls block %s max err %.3g" % (shape, err))
    assert np.isfinite(got).all()
    assert err <= TOL[torch.bfloat16]


def test_block_cls_is_row0_of_the_block():
    # the readout against the whole block run through the library: same inputs, row 0
    d = _dev()
    x, lay = _block_case(4, 197, 192, 3, 768, torch.float32, seed=21)
    lay_d = _to(lay, d)
    full = api.vit_encoder(x.to(d), [lay_d], 3, 1e-6, final_ln=False)
    cls = api.vit_block_cls(x.to(d), lay_d, 3, 1e-6)
    torch.cuda.synchronize()
    assert float((full[:, 0] - cls).abs().max()) <= 2e-4


def test_block_cls_inputs_unchanged_and_deterministic():
    d = _dev()
    x, lay = _block_case(8, 197, 192, 3, 768, torch.bfloat16, seed=31)
    xd, lay_d = x.to(d), _to(lay, d)
    x0 = xd.clone()
    a = api.vit_block_cls(xd, lay_d, 3, 1e-6)
    b = api.vit_block_cls(xd, lay_d, 3, 1e-6)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert torch.equal(xd, x0)


@pytest.mark.parametrize("dtype,shape,L", [
    (torch.float64, (2, 5, 8, 2, 16), 3),
    (torch.float32, (2, 65, 128, 2, 256), 3),
    (torch.bfloat16, (2, 197, 192, 3, 768), 3),
    (torch.bfloat16, (3, 33, 128, 2, 256), 1),
])
@pytest.mark.parametrize("final_ln", [True, False])
def test_encoder_cls_matches_oracle(dtype, shape, L, final_ln):
    d = _dev()
    N, T, D, H, F = shape
    x, layers, g, b = make_encoder_inputs(N, T, D, F, L, seed=L + T + 1, dtype=dtype)
    out = api.vit_encoder(x.to(d), [_to(l, d) for l in layers], H, 1e-6, lnf_g=g.to(d), lnf_b=b.to(d),
                          final_ln=final_ln, cls_only=True)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    got = out.double().cpu().numpy()
    ref = oracle.vit_encoder(x, layers, H, 1e-6, lnf_g=g, lnf_b=b, final_ln=final_ln, cls_only=True)
    err = float(np.abs(got - ref).max())
    print("cls encoder %s %s L=%d final_ln=%s max err %.3g" % (dtype, shape, L, final_ln, err))
    tol = {torch.float64: 1e-10, torch.float32: 2e-4}.get(dtype, 3e-2 * max(1.0, (L / 2.0) ** 0.5))
    assert err <= tol


def test_too_many_keys_is_unsupported():
    # the T scores of one query live in shared memory; 60,000 fp32 scores do not fit
    d = _dev()
    x, lay = _block_case(1, 60000, 64, 1, 64, torch.float32, seed=1, affine=False, biases=False)
    lay = {k: v for k, v in lay.items() if v is not None}
    with pytest.raises(api.VitError) as e:
        api.vit_block_cls(x.to(d), _to(lay, d), 1, 1e-6)
    assert e.value.status == -6
