"""Stage-by-stage parity of the CUDA kernels against the float64 oracle (GPU).

Each stage is called alone through its C-ABI entry point on seeded inputs and
compared element by element with the oracle's function for that stage, on shapes
that span several tiles and leave ragged tails (rows not a multiple of 128, columns
narrower than one 256-wide tile, key counts not a multiple of 64).

Tolerances (bf16 outputs, fp32 accumulation): |gpu - ref| <= atol + rtol * |ref|
with rtol = 2^-7 (two bf16 rounding steps: the kernel's output rounding and the
rounding of an fp32 sum that differs from the float64 sum in its last bits).
"""
import numpy as np
import pytest
import torch

import oracle
from vision_transformer_encoder_gb300 import api

pytestmark = pytest.mark.gpu

RTOL = 2.0 ** -7


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _rand(shape, seed, std=1.0, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(dtype)


def _close(gpu, ref, atol, rtol=RTOL):
    g = gpu.double().cpu().numpy()
    assert np.isfinite(g).all(), "non-finite output (unwritten or overflowed element)"
    err = np.abs(g - ref)
    bound = atol + rtol * np.abs(ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), "max excess at %s: gpu %g ref %g" % (worst, g[worst], ref[worst])
    return err.max()


@pytest.mark.parametrize("M,K,N", [(128, 64, 256), (300, 192, 192), (1000, 768, 768),
                                   (517, 1024, 2304), (64, 128, 64)])
def test_linear_store_bf16(M, K, N):
    d = _dev()
    a, w = _rand((M, K), 1), _rand((K, N), 2, std=K ** -0.5)
    out = api.linear(a.to(d), w.to(d))
    torch.cuda.synchronize()
    _close(out, oracle.matmul(a, w), atol=1e-3)


@pytest.mark.parametrize("M,K,N", [(384, 192, 768), (131, 768, 3072)])
def test_linear_gelu_bias_bf16(M, K, N):
    d = _dev()
    a, w, b = _rand((M, K), 3), _rand((K, N), 4, std=K ** -0.5), _rand((N,), 5, std=0.1)
    out = api.linear(a.to(d), w.to(d), bias=b.to(d), epilogue=api.EPI_GELU)
    torch.cuda.synchronize()
    ref = oracle.gelu_tanh(oracle.matmul(a, w, b))
    _close(out, ref, atol=2e-3)


@pytest.mark.parametrize("res_dtype,out_dtype", [(torch.bfloat16, torch.float32),
                                                 (torch.float32, torch.bfloat16)])
@pytest.mark.parametrize("M,K,N", [(256, 768, 768), (200, 3072, 192)])
def test_linear_residual_bf16(M, K, N, res_dtype, out_dtype):
    d = _dev()
    a, w = _rand((M, K), 6), _rand((K, N), 7, std=K ** -0.5)
    r = _rand((M, N), 8, dtype=res_dtype)
    out = api.linear(a.to(d), w.to(d), residual=r.to(d), epilogue=api.EPI_RESIDUAL,
                     out_dtype=out_dtype)
    torch.cuda.synchronize()
    ref = r.double().numpy() + oracle.matmul(a, w)
    _close(out, ref, atol=2e-3 if out_dtype == torch.bfloat16 else 1e-3,
           rtol=RTOL if out_dtype == torch.bfloat16 else 2.0 ** -12)


def test_linear_bias_on_residual():
    d = _dev()
    M, K, N = 130, 256, 512
    a, w, b = _rand((M, K), 9), _rand((K, N), 10, std=K ** -0.5), _rand((N,), 11, std=0.1)
    r = _rand((M, N), 12, dtype=torch.float32)
    out = api.linear(a.to(d), w.to(d), bias=b.to(d), residual=r.to(d), epilogue=api.EPI_RESIDUAL)
    torch.cuda.synchronize()
    _close(out, r.double().numpy() + oracle.matmul(a, w, b), atol=2e-3)


@pytest.mark.parametrize("dtype", [torch.float32, torch.float64])
def test_linear_cuda_core_types(dtype):
    d = _dev()
    M, K, N = 77, 45, 61
    a, w, b = _rand((M, K), 13, dtype=dtype), _rand((K, N), 14, dtype=dtype), _rand((N,), 15, dtype=dtype)
    out = api.linear(a.to(d), w.to(d), bias=b.to(d), epilogue=api.EPI_GELU)
    torch.cuda.synchronize()
    ref = oracle.gelu_tanh(oracle.matmul(a, w, b))
    tol = 1e-5 if dtype == torch.float32 else 1e-12
    _close(out, ref, atol=tol, rtol=tol)


@pytest.mark.parametrize("in_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("D", [192, 768, 1280])
@pytest.mark.parametrize("affine", [False, True])
def test_layernorm_to_bf16(in_dtype, D, affine):
    d = _dev()
    x = _rand((333, D), 16, std=2.0, dtype=in_dtype) + 0.5
    g = (1 + _rand((D,), 17, std=0.1)) if affine else None
    b = _rand((D,), 18, std=0.1) if affine else None
    out = api.layernorm(x.to(d), 1e-6, None if g is None else g.to(d), None if b is None else b.to(d),
                        out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    _close(out, oracle.layernorm(x, 1e-6, g, b), atol=1e-3)


def test_layernorm_constant_row_is_zero():
    d = _dev()
    x = torch.full((9, 768), 3.25).to(torch.bfloat16)
    out = api.layernorm(x.to(d), 1e-6, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert (out.float() == 0).all()


@pytest.mark.parametrize("dtype", [torch.float32, torch.float64])
def test_layernorm_wide_types(dtype):
    d = _dev()
    x = _rand((50, 30), 19, dtype=dtype)
    out = api.layernorm(x.to(d), 1e-5)
    torch.cuda.synchronize()
    tol = 1e-5 if dtype == torch.float32 else 1e-13
    _close(out, oracle.layernorm(x, 1e-5), atol=tol, rtol=tol)


def _close_attention(out, q, k, v, H):
    """Bound from the bf16 arithmetic of the tensor-core attention kernels: each softmax
    weight enters P V as P rounded to bf16 (unit roundoff 2^-8) under a common offset, the
    row sum is taken before that rounding, and out is rounded to bf16 once, so per element
    |out - ref| <= 2^-8 sum_j w_j |v_j| + 2^-8 |ref| (w the exact weights); fp32
    accumulation over at most a few thousand keys adds well under 2^-14 of the same."""
    ref = oracle.attention(q, k, v, H)
    wabs = oracle.attention(q, k, v.abs(), H)
    g = out.double().cpu().numpy()
    assert np.isfinite(g).all(), "non-finite output (unwritten or overflowed element)"
    err = np.abs(g - ref)
    bound = (2.0 ** -8 + 2.0 ** -14) * (wabs + np.abs(ref)) + 1e-6
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert (err <= bound).all(), "max excess at %s: gpu %g ref %g bound %g" % (
        worst, g[worst], ref[worst], bound[worst])
    return float((err / bound).max())


@pytest.mark.parametrize("N,T,D,H", [(2, 197, 128, 2), (1, 65, 64, 1), (3, 77, 160, 2),
                                     (1, 1, 64, 1), (2, 129, 256, 4), (1, 300, 96, 3),
                                     (2, 577, 128, 2), (1, 1025, 160, 2), (3, 256, 64, 1),
                                     (1, 385, 80, 1), (2, 224, 128, 2), (1, 128, 64, 1),
                                     (3, 208, 64, 1), (2, 16, 128, 2), (1, 225, 64, 1),
                                     (5, 100, 192, 3)])
def test_attention_bf16(N, T, D, H):
    d = _dev()
    qkv = _rand((N, T, 3 * D), 20 + T, std=1.5)
    out = api.attention(qkv.to(d), H)
    torch.cuda.synchronize()
    q, k, v = qkv[..., :D], qkv[..., D:2 * D], qkv[..., 2 * D:]
    print("attention %s: max err / bound %.3f" % ((N, T, D, H), _close_attention(out, q, k, v, H)))


@pytest.mark.parametrize("N,T,D,H", [
    (64, 197, 768, 12),     # whole-row kernel, two query tiles per item: ~5 items per CTA
    (100, 100, 768, 12),    # whole-row, one query tile per item: each MMA issuer also
                            # releases the buffers of the other issuer's items
    (33, 128, 768, 12),     # whole-row, one full query tile per item
    (40, 300, 768, 12),     # key-streaming, head width 64: items of two and of one query tile
    (20, 257, 1280, 16),    # key-streaming, head width 80: a last key tile of one key
])
def test_attention_bf16_many_items_per_cta(N, T, D, H):
    # Several work items per persistent CTA: item-to-item hand-offs of the query, key and
    # value buffers, of the score and O slots and of the O staging, over many phases of
    # every barrier.
    d = _dev()
    qkv = _rand((N, T, 3 * D), 90 + T, std=1.5)
    out = api.attention(qkv.to(d), H)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    q, k, v = qkv[..., :D], qkv[..., D:2 * D], qkv[..., 2 * D:]
    print("attention %s: max err / bound %.3f" % ((N, T, D, H), _close_attention(out, q, k, v, H)))


@pytest.mark.parametrize("T", [197, 224, 40, 100])
def test_attention_bf16_dominant_later_keys(T):
    # Keys scaled up so that, for many query rows, a key past the first 32 scores far
    # above every key in [0, 32): in the first half of the keys, in the second half, in
    # the 16-key tail, and by thousands (every earlier term underflows). Softmax is the
    # same under any common offset, so the result must match the oracle exactly as for
    # ordinary scores.
    d = _dev()
    N, D, H = 3, 128, 2
    qkv = _rand((N, T, 3 * D), 70 + T, std=1.5)
    k = qkv[..., D:2 * D].view(N, T, H, 64)
    spikes = [(0, 0, 50, 10.0), (0, 1, 150, 10.0), (1, 0, 200, 10.0), (1, 0, 100, 30.0),
              (1, 1, 60, 1000.0), (1, 1, 170, 1000.0), (2, 0, 33, -1000.0), (2, 1, 120, 6.0)]
    for n, h, t, a in spikes:
        if t < T:
            k[n, t, h] *= a
    out = api.attention(qkv.to(d), H)
    torch.cuda.synchronize()
    assert api.device_error() == 0
    q, k, v = qkv[..., :D], qkv[..., D:2 * D], qkv[..., 2 * D:]
    print("dominant keys T=%d: max err / bound %.3f" % (T, _close_attention(out, q, k, v, H)))


@pytest.mark.parametrize("dtype", [torch.float32, torch.float64])
def test_attention_cuda_core_types(dtype):
    d = _dev()
    N, T, D, H = 2, 37, 12, 3
    qkv = _rand((N, T, 3 * D), 21, dtype=dtype)
    out = api.attention(qkv.to(d), H)
    torch.cuda.synchronize()
    ref = oracle.attention(qkv[..., :D], qkv[..., D:2 * D], qkv[..., 2 * D:], H)
    tol = 1e-5 if dtype == torch.float32 else 1e-12
    _close(out, ref, atol=tol, rtol=tol)


@pytest.mark.parametrize("N,T,D,H", [(2, 197, 128, 2), (1, 65, 160, 2), (3, 33, 96, 1), (1, 129, 256, 2),
                                     (2, 16, 96, 2), (1, 300, 64, 2), (1, 1, 64, 1), (2, 200, 192, 3)])
def test_attention_fp32_tiled(N, T, D, H):
    # head widths 32 .. 128: the tiled fp32 kernel (keys and values staged in shared memory)
    d = _dev()
    qkv = _rand((N, T, 3 * D), 23 + T, std=1.5, dtype=torch.float32)
    out = api.attention(qkv.to(d), H)
    torch.cuda.synchronize()
    ref = oracle.attention(qkv[..., :D], qkv[..., D:2 * D], qkv[..., 2 * D:], H)
    _close(out, ref, atol=1e-5, rtol=1e-5)


@pytest.mark.parametrize("N,T,H", [(3, 1, 2), (2, 17, 3), (2, 128, 2), (2, 129, 1), (4, 197, 12), (2, 224, 4)])
def test_attention_fp32_tensor_cores(N, T, H):
    # head width 64 and T <= 224: the 3xTF32 tensor-core kernel, checked against the bound
    # its arithmetic allows (_close_attention_tf32)
    d = _dev()
    D = 64 * H
    qkv = _rand((N, T, 3 * D), 31 + T, std=1.5, dtype=torch.float32)
    out = torch.full((N, T, D), float("nan"), device=d)
    api.attention(qkv.to(d), H, out=out)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    r = _close_attention_tf32(out, qkv[..., :D], qkv[..., D:2 * D], qkv[..., 2 * D:], H)
    print("T=%d: max err / bound %.3f" % (T, r))
    assert api.device_error() == 0


def test_attention_fp32_tensor_cores_dominant_key():
    # one key far above the others in every row: the softmax is nearly one-hot, P_lo of
    # the large weight carries most of the correction, and the masked tail keys stay 0
    d = _dev()
    N, T, H = 2, 197, 3
    D = 64 * H
    qkv = _rand((N, T, 3 * D), 41, dtype=torch.float32)
    qkv[:, 100, D:2 * D] *= 12.0   # key 100 of every head
    out = api.attention(qkv.to(d), H)
    torch.cuda.synchronize()
    _close_attention_tf32(out, qkv[..., :D], qkv[..., D:2 * D], qkv[..., 2 * D:], H)


def _close_attention_tf32(out, q, k, v, H):
    """Bound from the 3xTF32 arithmetic: each product term q_i k_i (and p_j v_j) is off by
    at most 4 * 2^-20 of its size (the dropped lo x lo term, the TF32 rounding of the lo
    parts and the fp32 sums), so a score moves by e <= 4 * 2^-20 sum_i |q_i k_i| / sqrt(dh),
    each softmax weight by a factor within exp(+-2 e_max) of the row, and per element
    |out - ref| <= (2 e_max + 4 * 2^-20) sum_j w_j |v_j| + 2^-24 |ref|."""
    N, T, D = q.shape
    dh = D // H
    ref = oracle.attention(q, k, v, H)
    wabs = oracle.attention(q, k, v.abs(), H)
    qa = q.double().abs().numpy().reshape(N, T, H, dh).transpose(0, 2, 1, 3)
    ka = k.double().abs().numpy().reshape(N, T, H, dh).transpose(0, 2, 3, 1)
    emax = (4 * 2.0 ** -20) * (qa @ ka).max(axis=-1) / np.sqrt(dh)        # (N, H, T)
    emax = np.repeat(emax.transpose(0, 2, 1), dh, axis=2)                  # (N, T, D)
    bound = (2 * emax + 4 * 2.0 ** -20) * wabs + 2.0 ** -24 * np.abs(ref)
    g = out.double().cpu().numpy()
    assert np.isfinite(g).all()
    err = np.abs(g - ref)
    assert (err <= bound).all(), "max err / bound %.3f" % (err / bound).max()
    return (err / bound).max()


def test_attention_bf16_generic_head_width():
    # head width 24 is not one the tensor-core kernel takes: CUDA-core kernel, bf16 I/O
    d = _dev()
    N, T, D, H = 2, 50, 48, 2
    qkv = _rand((N, T, 3 * D), 22)
    out = api.attention(qkv.to(d), H)
    torch.cuda.synchronize()
    ref = oracle.attention(qkv[..., :D], qkv[..., D:2 * D], qkv[..., 2 * D:], H)
    _close(out, ref, atol=2e-3)


def test_no_device_error_after_stages():
    _dev()
    assert api.device_error() == 0
