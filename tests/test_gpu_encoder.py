"""Parity of vit_encoder (a stack of blocks with projection biases and the final
LayerNorm) with the float64 oracle, on the bf16, fp32 and fp64 paths."""
import numpy as np
import pytest
import torch

import oracle
from vision_transformer_encoder_gb300 import api
from vision_transformer_encoder_gb300.inputs import make_encoder_inputs

pytestmark = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _run(x, layers, H, eps, lnf_g, lnf_b, final_ln):
    d = _dev()
    lay_d = [{k: (v.to(d) if v is not None else None) for k, v in lay.items()} for lay in layers]
    out = api.vit_encoder(x.to(d), lay_d, H, eps, lnf_g=lnf_g.to(d), lnf_b=lnf_b.to(d), final_ln=final_ln)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    return out.double().cpu().numpy()


def _oracle(x, layers, H, eps, lnf_g, lnf_b, final_ln):
    return oracle.vit_encoder(x, layers, H, eps, lnf_g=lnf_g, lnf_b=lnf_b, final_ln=final_ln)


def _err(x, layers, H, eps, lnf_g, lnf_b, final_ln):
    got = _run(x, layers, H, eps, lnf_g, lnf_b, final_ln)
    assert np.isfinite(got).all()
    ref = _oracle(x, layers, H, eps, lnf_g, lnf_b, final_ln)
    return float(np.abs(got - ref).max())


@pytest.mark.parametrize("dtype,shape,L,tol", [
    (torch.float64, (2, 5, 8, 2, 16), 3, 1e-10),
    (torch.float32, (2, 5, 8, 2, 16), 3, 2e-4),
    (torch.float32, (2, 65, 128, 2, 256), 3, 2e-4),
    (torch.bfloat16, (2, 197, 192, 3, 768), 3, None),
    (torch.bfloat16, (3, 33, 128, 2, 256), 4, None),
])
@pytest.mark.parametrize("final_ln", [True, False])
def test_encoder_matches_oracle(dtype, shape, L, tol, final_ln):
    N, T, D, H, F = shape
    x, layers, g, b = make_encoder_inputs(N, T, D, F, L, seed=L + T, dtype=dtype)
    err = _err(x, layers, H, 1e-6, g, b, final_ln)
    print("encoder %s %s L=%d final_ln=%s max err %.3g" % (dtype, shape, L, final_ln, err))
    if tol is None:
        tol = encoder_bf16_tol(L)
    assert err <= tol


def encoder_bf16_tol(L):
    """bf16 stack bound: one block's bf16 stage roundings (xn, qkv, P, o, yn, h) cost up to
    about 1.8e-2 and the final rounding of out 1.6e-2 (the single-block bound 3e-2 covers
    both); between blocks the stream stays fp32, so the blocks' independent errors add
    roughly in quadrature: 3e-2 * max(1, sqrt(L / 2))."""
    return 3e-2 * max(1.0, (L / 2.0) ** 0.5)


def test_single_layer_without_final_ln_is_the_block_bitwise():
    d = _dev()
    x, layers, g, b = make_encoder_inputs(2, 197, 192, 768, 1, seed=3, dtype=torch.bfloat16, biases=False)
    lay = layers[0]
    out_e = api.vit_encoder(x.to(d), [{k: v.to(d) for k, v in lay.items()}], 3, 1e-6, final_ln=False)
    out_b = api.vit_block_ex(x.to(d), *[lay[k].to(d) for k in ("w_q", "w_k", "w_v", "w_o", "w_mlp1", "w_mlp2")],
                             3, 1e-6, ln1_g=lay["ln1_g"].to(d), ln1_b=lay["ln1_b"].to(d),
                             ln2_g=lay["ln2_g"].to(d), ln2_b=lay["ln2_b"].to(d), b1=lay["b1"].to(d),
                             b2=lay["b2"].to(d))
    torch.cuda.synchronize()
    assert torch.equal(out_e, out_b)
