"""Prepared weights: vit_weights_create, vit_block_w, vit_block_w_host and
vit_block_w_host_async.

A handle holds one block's weights on the device, copied once, with the concatenated
Q/K/V bias and, for a fold handle, the per-column terms of both folded LayerNorms
("ViT Encoder Block" (ai-engineer-exhaustive), Key Equations, Steps 1 and 4:
LN(x) W = rstd (x W' - mean c) + d with W' = diag(gamma) W, c = column sums of W',
d = beta W + b).

- A plain handle (fold 0) runs the kernels of vit_block_ex / vit_encoder: its results
  must equal theirs bit for bit.
- A fold handle (fold 1) rounds differently (W' in bf16, statistics from x itself). It
  is checked against the float64 oracle at the block tolerance, with and without the
  projection biases, at several block shapes.
- The host-buffer call must equal the device call bit for bit, on both kinds of handle.
"""
import numpy as np
import pytest
import torch

import oracle
from vision_transformer_encoder_gb300 import api
from vision_transformer_encoder_gb300.inputs import make_encoder_inputs, make_inputs

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 3e-2, torch.float32: 2e-4}


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def _layer(d, affine):
    lay = {n: t for n, t in zip(("w_q", "w_k", "w_v", "w_o", "w_mlp1", "w_mlp2"), d.weights())}
    if affine:
        lay.update(d.affine())
    return lay


def _maxerr(gpu, ref):
    g = gpu.double().cpu().numpy()
    assert np.isfinite(g).all()
    return float(np.abs(g - ref).max())


@pytest.mark.parametrize("dtype,shape,affine", [
    (torch.bfloat16, (8, 197, 768, 12, 3072), False),    # ViT-B/16 block shape
    (torch.bfloat16, (8, 197, 768, 12, 3072), True),
    (torch.float32, (4, 197, 192, 3, 768), True),        # ViT-Ti/16 block shape, fp32 path
    (torch.float32, (6, 197, 768, 12, 3072), True),      # ViT-B/16 block shape, fp32: the handle's
                                                         # prepared weight split on multi-tile products
])
def test_plain_handle_equals_vit_block_ex(dtype, shape, affine):
    dev = _dev()
    N, T, D, H, F = shape
    d = make_inputs(N, T, D, F, seed=61, dtype=dtype, affine=affine).to(device=dev)
    w = api.VitWeights(_layer(d, affine), H, fold=0)
    assert not w.fold and (w.D, w.F, w.H) == (D, F, H)
    out = api.vit_block_w(d.x, w, 1e-6)
    ref = api.vit_block_ex(d.x, *d.weights(), H, 1e-6, **(d.affine() if affine else {}))
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    w.close()


def test_plain_handle_with_projection_biases_equals_encoder():
    # b_q, b_k, b_v and b_o: the block of a one-layer vit_encoder without the final LN
    dev = _dev()
    x, layers, _, _ = make_encoder_inputs(4, 197, 192, 768, 1, seed=17, dtype=torch.bfloat16)
    lay = {k: v.to(dev) for k, v in layers[0].items() if v is not None}
    w = api.VitWeights(lay, 3, fold=0)
    out = api.vit_block_w(x.to(dev), w, 1e-6)
    ref = api.vit_encoder(x.to(dev), [lay], 3, 1e-6, final_ln=False)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


@pytest.mark.parametrize("shape,biases", [
    ((2, 197, 768, 12, 3072), False),    # ViT-B/16: three 256-column tiles of D, T ragged
    ((2, 197, 768, 12, 3072), True),
    ((4, 197, 192, 3, 768), True),       # ViT-Ti/16
    ((1, 577, 1024, 16, 4096), True),    # ViT-L/16 at 384 px
    ((3, 33, 128, 2, 192), True),        # several sequences in one 128-row tile
])
def test_fold_handle_matches_oracle(shape, biases):
    dev = _dev()
    N, T, D, H, F = shape
    x, layers, _, _ = make_encoder_inputs(N, T, D, F, 1, seed=T + D, dtype=torch.bfloat16, biases=biases)
    lay = {k: v.to(dev) for k, v in layers[0].items() if v is not None}
    w = api.VitWeights(lay, H, fold=1)
    assert w.fold
    out = api.vit_block_w(x.to(dev), w, 1e-6)
    torch.cuda.synchronize()
    ref = oracle.vit_block_full(x, *[layers[0][k] for k in ("w_q", "w_k", "w_v", "w_o", "w_mlp1", "w_mlp2")],
                                H, 1e-6, **{k: v for k, v in layers[0].items()
                                            if k not in ("w_q", "w_k", "w_v", "w_o", "w_mlp1", "w_mlp2")})
    err = _maxerr(out, ref)
    print("fold handle %s biases=%s max err %.3g" % (shape, biases, err))
    assert err <= TOL[torch.bfloat16], err


def test_fold_handle_is_deterministic_and_reusable():
    dev = _dev()
    d = make_inputs(16, 197, 768, 3072, seed=5, dtype=torch.bfloat16, affine=True).to(device=dev)
    w = api.VitWeights(_layer(d, True), 12, fold=1)
    a = api.vit_block_w(d.x, w, 1e-6)
    b = api.vit_block_w(d.x, w, 1e-6)
    d2 = make_inputs(8, 197, 768, 3072, seed=6, dtype=torch.bfloat16).to(device=dev)
    api.vit_block_w(d2.x, w, 1e-6)     # another batch size in between
    c = api.vit_block_w(d.x, w, 1e-6)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(a, c)


@pytest.mark.parametrize("fold", [0, 1])
def test_host_call_equals_device_call(fold):
    # 128 ViT-B/16 sequences (25,216 tokens): the host call cuts them into two chunks
    dev = _dev()
    d = make_inputs(128, 197, 768, 3072, seed=9, dtype=torch.bfloat16, affine=True)
    w = api.VitWeights(_layer(d.to(device=dev), True), 12, fold=fold)
    ref = api.vit_block_w(d.x.to(dev), w, 1e-6)
    x_host = d.x.pin_memory()
    out_host = torch.full_like(x_host, float("nan")).pin_memory()
    api.vit_block_w_host(x_host, w, 1e-6, out=out_host)
    assert torch.equal(out_host, ref.cpu())


def test_weights_from_host_and_copies_are_independent():
    # a handle made from host arrays equals one made from device arrays; changing the
    # caller's arrays afterwards changes nothing (the handle holds copies)
    dev = _dev()
    d = make_inputs(4, 197, 192, 768, seed=12, dtype=torch.bfloat16, affine=True)
    lay_host = {k: v.contiguous() for k, v in _layer(d, True).items()}
    w_host = api.VitWeights(lay_host, 3, fold=0, device=0)
    dd = d.to(device=dev)
    lay_dev = _layer(dd, True)
    w_dev = api.VitWeights(lay_dev, 3, fold=0)
    a = api.vit_block_w(dd.x, w_host, 1e-6)
    b = api.vit_block_w(dd.x, w_dev, 1e-6)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    for t in lay_dev.values():
        t.zero_()
    c = api.vit_block_w(dd.x, w_dev, 1e-6)
    torch.cuda.synchronize()
    assert torch.equal(a, c)


def test_fold_handle_with_unaligned_x_runs_the_plain_path():
    # x starting 2 bytes past a 16-byte boundary: the folded GEMMs cannot read it, so
    # the fold handle runs the plain path, bit-identical to the plain handle's
    dev = _dev()
    N, T, D, H, F = 2, 33, 128, 2, 256
    d = make_inputs(N, T, D, F, seed=3, dtype=torch.bfloat16, affine=True).to(device=dev)
    buf = torch.empty(N * T * D + 1, dtype=torch.bfloat16, device=dev)
    x = buf[1:].view(N, T, D)
    x.copy_(d.x)
    w_fold = api.VitWeights(_layer(d, True), H, fold=1)
    w_plain = api.VitWeights(_layer(d, True), H, fold=0)
    a = api.vit_block_w(x, w_fold, 1e-5)
    b = api.vit_block_w(x, w_plain, 1e-5)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    ref = oracle.vit_block(d.x.cpu(), *[t.cpu() for t in d.weights()], H, 1e-5,
                           **{k: v.cpu() for k, v in d.affine().items()})
    assert _maxerr(a, ref) <= TOL[torch.bfloat16]


def test_fold_is_refused_where_unavailable_and_closed_handles_refuse_use():
    dev = _dev()
    d = make_inputs(2, 9, 64, 128, seed=1, dtype=torch.float32).to(device=dev)
    with pytest.raises(api.VitError) as e:
        api.VitWeights(_layer(d, False), 2, fold=1)
    assert e.value.status == -6
    w = api.VitWeights(_layer(d, False), 2, fold=-1)
    assert not w.fold               # the library's choice on fp32: the plain path
    w.close()
    with pytest.raises(ValueError):
        api.vit_block_w(d.x, w, 1e-5)
    w.close()                       # closing twice is harmless


def test_async_host_calls_overlap_and_equal_device_calls():
    # six batches issued back to back on a ring of three streams, each into its own pinned
    # output: every output equals vit_block_w on the same batch, bit for bit
    dev = _dev()
    d = make_inputs(32, 197, 768, 3072, seed=21, dtype=torch.bfloat16, affine=True)
    w = api.VitWeights(_layer(d.to(device=dev), True), 12, fold=0)
    xs = [make_inputs(32 + 3 * i, 197, 768, 3072, seed=40 + i, dtype=torch.bfloat16).x.pin_memory()
          for i in range(6)]
    outs = [torch.full_like(x, float("nan")).pin_memory() for x in xs]
    streams = [torch.cuda.Stream(device=dev) for _ in range(3)]
    for i, (x, o) in enumerate(zip(xs, outs)):
        api.vit_block_w_host_async(x, w, 1e-6, o, streams[i % 3])
    for s in streams:
        s.synchronize()
    for x, o in zip(xs, outs):
        ref = api.vit_block_w(x.to(dev), w, 1e-6)
        torch.cuda.synchronize()
        assert torch.equal(o, ref.cpu())
    w.close()


def test_async_host_calls_on_one_stream_run_in_order():
    # two blocks chained through host memory on one stream, with no wait in between: the
    # second call reads the first call's output buffer as its input, so it must start
    # only after the first call's copy out has landed
    dev = _dev()
    d = make_inputs(4, 197, 192, 768, seed=8, dtype=torch.bfloat16, affine=True)
    w = api.VitWeights(_layer(d.to(device=dev), True), 3, fold=1)
    x_host = d.x.pin_memory()
    mid = torch.full_like(x_host, float("nan")).pin_memory()
    out = torch.full_like(x_host, float("nan")).pin_memory()
    s = torch.cuda.Stream(device=dev)
    api.vit_block_w_host_async(x_host, w, 1e-6, mid, s)
    api.vit_block_w_host_async(mid, w, 1e-6, out, s)
    s.synchronize()
    r1 = api.vit_block_w(d.x.to(dev), w, 1e-6)
    r2 = api.vit_block_w(r1, w, 1e-6)
    torch.cuda.synchronize()
    assert torch.equal(mid, r1.cpu()) and torch.equal(out, r2.cpu())
    w.close()
