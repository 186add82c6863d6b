"""Pins of the float64 oracle to facts that do not come from the oracle itself.

Each test checks the oracle against one of: a value the pages print for a worked
example (fixtures under tests/golden/, each with its citation), a closed form, an
invariant the pages state, or a float64 library routine that computes the same
mathematical function. Together they are chosen so that a plausible slip anywhere in
the oracle (wrong eps, sample instead of population variance, a dropped residual,
a transposed weight, a wrong head offset or score scale, a masked key, the erf GELU
instead of the tanh one) fails at least one of them; test_pins_reject_mutants shows
that for each such slip.
"""
import json
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as Fn

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand_block(N, T, D, F, seed, affine=False):
    rng = np.random.default_rng(seed)
    a = dict(
        x=rng.standard_normal((N, T, D)),
        w_q=rng.standard_normal((D, D)) / np.sqrt(D),
        w_k=rng.standard_normal((D, D)) / np.sqrt(D),
        w_v=rng.standard_normal((D, D)) / np.sqrt(D),
        w_o=rng.standard_normal((D, D)) / np.sqrt(D),
        w_mlp1=rng.standard_normal((D, F)) / np.sqrt(D),
        w_mlp2=rng.standard_normal((F, D)) / np.sqrt(F),
    )
    if affine:
        a.update(ln1_g=1 + 0.1 * rng.standard_normal(D), ln1_b=0.1 * rng.standard_normal(D),
                 ln2_g=1 + 0.1 * rng.standard_normal(D), ln2_b=0.1 * rng.standard_normal(D),
                 b1=0.1 * rng.standard_normal(F), b2=0.1 * rng.standard_normal(D))
    return a


def _call_full(a, H, eps, **kw):
    return oracle.vit_block_full(a["x"], a["w_q"], a["w_k"], a["w_v"], a["w_o"], a["w_mlp1"],
                                 a["w_mlp2"], H, eps, **{k: a.get(k) for k in
                                                         ("ln1_g", "ln1_b", "ln2_g", "ln2_b", "b1", "b2",
                                                          "b_q", "b_k", "b_v", "b_o")}, **kw)


def _with_proj_biases(a, seed):
    rng = np.random.default_rng(seed)
    D = a["w_q"].shape[0]
    a = dict(a)
    a.update(b_q=0.2 * rng.standard_normal(D), b_k=0.2 * rng.standard_normal(D),
             b_v=0.2 * rng.standard_normal(D), b_o=0.2 * rng.standard_normal(D))
    return a


def _rand_layers(L, D, F, seed, affine=True, biases=True):
    layers = []
    for l in range(L):
        a = _rand_block(1, 1, D, F, seed=seed + 17 * l, affine=affine)
        a.pop("x")
        if biases:
            a = _with_proj_biases(a, seed + 31 * l)
        layers.append(a)
    return layers


def _torch_encoder(x, layers, H, eps, lnf_g=None, lnf_b=None, final_ln=True):
    """The stack written with the float64 PyTorch block above, then torch's layer_norm."""
    cur = np.asarray(x, dtype=np.float64)
    for lay in layers:
        cur = _torch_block(dict(lay, x=cur), H, eps)
    if not final_ln:
        return cur
    t = lambda v: None if v is None else torch.from_numpy(np.asarray(v, dtype=np.float64))
    return Fn.layer_norm(torch.from_numpy(cur), (cur.shape[-1],), t(lnf_g), t(lnf_b), eps=eps).numpy()


def _call(a, H, eps, **kw):
    return oracle.vit_block(a["x"], a["w_q"], a["w_k"], a["w_v"], a["w_o"], a["w_mlp1"],
                            a["w_mlp2"], H, eps, ln1_g=a.get("ln1_g"), ln1_b=a.get("ln1_b"),
                            ln2_g=a.get("ln2_g"), ln2_b=a.get("ln2_b"), b1=a.get("b1"),
                            b2=a.get("b2"), **kw)


def _p2_args(ex):
    return dict(x=np.array(ex["x"], float), w_q=np.array(ex["Wq"], float),
                w_k=np.array(ex["Wk"], float), w_v=np.array(ex["Wv"], float),
                w_o=np.array(ex["Wo"], float), w_mlp1=np.array(ex["W1"], float),
                w_mlp2=np.array(ex["W2"], float))


# ---------------------------------------------------------------------------------
# Whole block: the three worked examples printed to 6 d.p.
# ---------------------------------------------------------------------------------
@pytest.mark.parametrize("i", [0, 1, 2])
def test_p2_worked_examples(i):
    g = _load("p2_worked_examples.json")
    ex = g["examples"][i]
    out = _call(_p2_args(ex), ex["num_heads"], g["eps"])
    np.testing.assert_allclose(out, np.array(ex["output"]), rtol=0, atol=g["print_tolerance"])


def test_p2_example2_constant_row_is_exact():
    # token [1, 1] has zero variance: LN gives exactly 0, so both stage outputs are 0
    # for that row and it leaves the block unchanged.
    g = _load("p2_worked_examples.json")
    ex = g["examples"][1]
    out = _call(_p2_args(ex), ex["num_heads"], g["eps"])
    assert out[0, 2, 0] == 1.0 and out[0, 2, 1] == 1.0


def test_p2_examples_discriminate_eps_gelu_orientation():
    """The examples only fit eps = 1e-6, x @ W and the tanh GELU: other readings miss."""
    g = _load("p2_worked_examples.json")
    worst_eps = 0.0
    for ex in g["examples"]:
        out = _call(_p2_args(ex), ex["num_heads"], 1e-5)
        worst_eps = max(worst_eps, np.abs(out - np.array(ex["output"])).max())
    assert worst_eps > 1e-4
    ex = g["examples"][2]
    a = _p2_args(ex)
    at = {k: (v.T.copy() if k != "x" else v) for k, v in a.items()}
    out = _call(at, ex["num_heads"], g["eps"])
    assert np.abs(out - np.array(ex["output"])).max() > 0.1


# ---------------------------------------------------------------------------------
# Sub-steps: the partially worked numerical example (4 d.p.)
# ---------------------------------------------------------------------------------
def test_p4_layernorm_rows():
    f = _load("p4_numerical_example.json")["layernorm"]
    x = np.array(f["x"])
    np.testing.assert_allclose(x.mean(axis=1), f["mean"], atol=1e-15)
    np.testing.assert_allclose(((x - x.mean(1, keepdims=True)) ** 2).mean(1), f["variance"],
                               atol=1e-15)
    out = oracle.layernorm(x, f["eps"])
    np.testing.assert_allclose(out, np.array(f["normalized"]), atol=f["tolerance"])


def test_p4_softmax_rows():
    f = _load("p4_numerical_example.json")["softmax"]
    p = oracle.softmax_rows(np.array(f["scaled_scores"]))
    for r in range(2):
        np.testing.assert_allclose(p[r], f["weights"][r], atol=f["tolerance_row"][r])


def test_p4_residual_adds_unnormalised_input():
    """y = x + MSA(LN(x)): choose w_o so that the block's MSA output equals the page's
    'suppose' values, then the block's y must equal the page's x' (printed exactly)."""
    f = _load("p4_numerical_example.json")["residual"]
    rng = np.random.default_rng(3)
    x = np.array(f["x"])[None]
    D = 4
    a = dict(x=x, w_q=rng.standard_normal((D, D)), w_k=rng.standard_normal((D, D)),
             w_v=rng.standard_normal((D, D)), w_o=np.eye(D), w_mlp1=np.eye(D, 8),
             w_mlp2=np.eye(8, D))
    _, st = _call(a, 2, 1e-5, stages=True)
    o = st["o"][0]                                   # (2, 4), rank 2
    a["w_o"] = np.linalg.pinv(o) @ np.array(f["msa_output"])
    _, st = _call(a, 2, 1e-5, stages=True)
    np.testing.assert_allclose(st["y"][0], np.array(f["x_prime"]), atol=1e-12)


def test_p4_gelu_half():
    f = _load("p4_numerical_example.json")["gelu"]
    assert abs(oracle.gelu_tanh(np.array([f["z"]]))[0] - f["value"]) <= f["tolerance"]


# ---------------------------------------------------------------------------------
# Library special cases and closed forms
# ---------------------------------------------------------------------------------
def test_gelu_matches_torch_tanh_gelu():
    z = np.linspace(-8, 8, 2001)
    ref = Fn.gelu(torch.from_numpy(z), approximate="tanh").numpy()
    np.testing.assert_allclose(oracle.gelu_tanh(z), ref, rtol=0, atol=1e-15)
    erf = Fn.gelu(torch.from_numpy(z)).numpy()
    assert np.abs(oracle.gelu_tanh(z) - erf).max() > 1e-4   # not the erf form


def test_gelu_limits():
    g = oracle.gelu_tanh(np.array([0.0, 20.0, -20.0]))
    assert g[0] == 0.0 and g[1] == 20.0 and abs(g[2]) < 1e-300 + 1e-12


def test_layernorm_d2_closed_form():
    """D = 2: LN([a, b]) = (+-1) * |a-b|/2 / sqrt((a-b)^2/4 + eps), signs (sgn(a-b), sgn(b-a))."""
    rng = np.random.default_rng(0)
    x = rng.standard_normal((50, 2)) * 3
    eps = 1e-5
    h = (x[:, 0] - x[:, 1]) / 2
    mag = np.abs(h) / np.sqrt(h * h + eps)
    exp = np.stack([np.sign(h) * mag, -np.sign(h) * mag], axis=1)
    np.testing.assert_allclose(oracle.layernorm(x, eps), exp, atol=1e-14)


def test_layernorm_matches_torch_and_affine():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((37, 24)) * 2 + 0.5
    g, b = rng.standard_normal(24), rng.standard_normal(24)
    for eps in (1e-5, 1e-6):
        ref = Fn.layer_norm(torch.from_numpy(x), (24,), torch.from_numpy(g), torch.from_numpy(b),
                            eps=eps).numpy()
        np.testing.assert_allclose(oracle.layernorm(x, eps, g, b), ref, atol=1e-13)


def test_softmax_rows_sum_to_one_and_are_shift_invariant():
    rng = np.random.default_rng(2)
    s = rng.standard_normal((20, 197)) * 10
    p = oracle.softmax_rows(s)
    np.testing.assert_allclose(p.sum(1), 1.0, atol=1e-14)
    assert (p > 0).all()
    np.testing.assert_allclose(oracle.softmax_rows(s + 1000.0), p, atol=1e-14)
    np.testing.assert_allclose(p, torch.softmax(torch.from_numpy(s), -1).numpy(), atol=1e-15)


def test_matmul_matches_numpy():
    rng = np.random.default_rng(4)
    a, w, b = rng.standard_normal((7, 13)), rng.standard_normal((13, 5)), rng.standard_normal(5)
    np.testing.assert_allclose(oracle.matmul(a, w), a @ w, atol=1e-13)
    np.testing.assert_allclose(oracle.matmul(a, w, b), a @ w + b, atol=1e-13)


def _torch_block(a, H, eps):
    """The block written with float64 PyTorch library routines (layer_norm,
    scaled_dot_product_attention, tanh GELU) -- an independent composition."""
    t = {k: torch.from_numpy(np.asarray(v, dtype=np.float64)) for k, v in a.items()}
    x = t["x"]
    N, T, D = x.shape
    dh = D // H
    xn = Fn.layer_norm(x, (D,), t.get("ln1_g"), t.get("ln1_b"), eps=eps)

    def heads(m):
        return m.reshape(N, T, H, dh).transpose(1, 2)
    def proj(w, b):
        m = xn @ t[w]
        return m + t[b] if b in t else m
    q, k, v = heads(proj("w_q", "b_q")), heads(proj("w_k", "b_k")), heads(proj("w_v", "b_v"))
    o = Fn.scaled_dot_product_attention(q, k, v).transpose(1, 2).reshape(N, T, D)
    a_o = o @ t["w_o"]
    if "b_o" in t:
        a_o = a_o + t["b_o"]
    y = x + a_o
    yn = Fn.layer_norm(y, (D,), t.get("ln2_g"), t.get("ln2_b"), eps=eps)
    z = yn @ t["w_mlp1"]
    if "b1" in t:
        z = z + t["b1"]
    m = Fn.gelu(z, approximate="tanh") @ t["w_mlp2"]
    if "b2" in t:
        m = m + t["b2"]
    return (y + m).numpy()


@pytest.mark.parametrize("shape", [(2, 7, 12, 20, 3), (1, 1, 8, 32, 2), (3, 5, 6, 6, 6),
                                   (2, 33, 16, 64, 1), (1, 13, 20, 40, 4),
                                   (2, 197, 192, 768, 3), (1, 65, 160, 320, 2)])
@pytest.mark.parametrize("affine", [False, True])
def test_block_matches_torch_library_composition(shape, affine):
    N, T, D, F, H = shape
    a = _rand_block(N, T, D, F, seed=hash(shape) % 1000, affine=affine)
    np.testing.assert_allclose(_call(a, H, 1e-5), _torch_block(a, H, 1e-5), rtol=0, atol=1e-11)


def test_stages_match_torch_steps():
    a = _rand_block(2, 9, 12, 24, seed=5)
    out, st = _call(a, 3, 1e-6, stages=True)
    x = torch.from_numpy(a["x"])
    xn = Fn.layer_norm(x, (12,), eps=1e-6).numpy()
    np.testing.assert_allclose(st["xn"], xn, atol=1e-13)
    qkv = np.concatenate([xn @ a["w_q"], xn @ a["w_k"], xn @ a["w_v"]], axis=-1)
    np.testing.assert_allclose(st["qkv"], qkv, atol=1e-13)
    np.testing.assert_allclose(st["y"], a["x"] + st["o"] @ a["w_o"], atol=1e-13)
    np.testing.assert_allclose(out, st["y"] + st["g"] @ a["w_mlp2"], atol=1e-13)


# ---------------------------------------------------------------------------------
# Invariants stated on the pages
# ---------------------------------------------------------------------------------
def test_zero_stage_outputs_return_x_exactly():
    # "If both stage outputs are zero, the residual paths return x unchanged."
    a = _rand_block(2, 6, 8, 16, seed=6, affine=True)
    a["w_o"] = np.zeros_like(a["w_o"])
    a["w_mlp2"] = np.zeros_like(a["w_mlp2"])
    del a["b2"]
    out, st = _call(a, 2, 1e-5, stages=True)
    assert np.array_equal(st["y"], a["x"])
    assert np.array_equal(out, a["x"])


def test_permutation_equivariance():
    # "E2E: Tiny Vision Transformer", "Why position embeddings matter".
    a = _rand_block(1, 11, 12, 24, seed=7)
    perm = np.random.default_rng(8).permutation(11)
    out = _call(a, 3, 1e-5)
    b = dict(a, x=a["x"][:, perm])
    np.testing.assert_allclose(_call(b, 3, 1e-5), out[:, perm], atol=1e-13)


def test_heads_read_only_their_slice():
    a = _rand_block(1, 8, 12, 16, seed=9)
    H, dh, h = 3, 4, 1
    _, st0 = _call(a, H, 1e-5, stages=True)
    # (a constant offset would vanish: LN output rows sum to zero)
    rng = np.random.default_rng(15)
    b = dict(a)
    b["w_q"] = a["w_q"].copy()
    b["w_q"][:, h * dh:(h + 1) * dh] += rng.standard_normal((12, dh))
    b["w_k"] = a["w_k"].copy()
    b["w_k"][:, h * dh:(h + 1) * dh] -= rng.standard_normal((12, dh))
    _, st1 = _call(b, H, 1e-5, stages=True)
    keep = np.ones(12, bool)
    keep[h * dh:(h + 1) * dh] = False
    assert np.array_equal(st0["o"][..., keep], st1["o"][..., keep])
    assert np.abs(st0["o"][..., ~keep] - st1["o"][..., ~keep]).max() > 1e-3


def test_sequences_are_independent():
    a = _rand_block(3, 6, 8, 16, seed=10)
    out = _call(a, 2, 1e-5)
    b = dict(a, x=a["x"].copy())
    b["x"][1] += np.random.default_rng(17).standard_normal((6, 8))
    out2 = _call(b, 2, 1e-5)
    assert np.array_equal(out[0], out2[0]) and np.array_equal(out[2], out2[2])
    single = _call(dict(a, x=a["x"][2:3]), 2, 1e-5)
    assert np.array_equal(single[0], out[2])


def test_no_causal_mask():
    # "ViT Encoder Block" (ai-engineer-exhaustive), "No Causal Mask" and "Pitfalls":
    # the first token must see a change to the last one.
    a = _rand_block(1, 6, 8, 16, seed=11)
    out = _call(a, 2, 1e-5)
    b = dict(a, x=a["x"].copy())
    b["x"][0, -1] += np.random.default_rng(16).standard_normal(8)   # not a constant: LN removes those
    assert np.abs(_call(b, 2, 1e-5)[0, 0] - out[0, 0]).max() > 1e-4


def test_single_token_attention_is_value_row():
    # T = 1: the only softmax weight is exactly 1, so Q and K cannot matter.
    a = _rand_block(2, 1, 8, 16, seed=12)
    out = _call(a, 2, 1e-5)
    b = dict(a, w_q=a["w_q"] * 3 + 1, w_k=-a["w_k"])
    assert np.array_equal(_call(b, 2, 1e-5), out)
    _, st = _call(a, 2, 1e-5, stages=True)
    np.testing.assert_allclose(st["o"], st["qkv"][..., 16:], atol=0)


def test_zero_queries_give_uniform_weights():
    # w_q = 0: every score is 0, weights are 1/T, the head output is the mean of V.
    a = _rand_block(1, 7, 8, 16, seed=13)
    a["w_q"] = np.zeros_like(a["w_q"])
    _, st = _call(a, 2, 1e-5, stages=True)
    v = st["qkv"][..., 16:]
    np.testing.assert_allclose(st["o"][0], np.broadcast_to(v[0].mean(0), (7, 8)), atol=1e-15)
    b = dict(a, w_k=a["w_k"] * 5)
    _, st2 = _call(b, 2, 1e-5, stages=True)
    assert np.array_equal(st["o"], st2["o"])


def test_invalid_sizes_rejected():
    a = _rand_block(1, 3, 6, 8, seed=14)
    with pytest.raises(ValueError):
        _call(a, 4, 1e-5)      # 4 does not divide 6


# ---------------------------------------------------------------------------------
# The pins above catch plausible slips: each mutant is a copy of the oracle source
# with one mistake planted (compiled on the CPU into a temporary library).
# ---------------------------------------------------------------------------------
@pytest.mark.parametrize("shape", [(2, 7, 12, 20, 3), (1, 33, 16, 64, 1), (2, 65, 40, 80, 4)])
def test_projection_biases_match_torch(shape):
    N, T, D, F, H = shape
    a = _with_proj_biases(_rand_block(N, T, D, F, seed=7 + T, affine=True), seed=T)
    np.testing.assert_allclose(_call_full(a, H, 1e-5), _torch_block(a, H, 1e-5), rtol=0, atol=1e-11)


def test_key_bias_changes_nothing():
    # a key bias shifts every score of a query row by q . b_k: the softmax ignores it
    a = _rand_block(2, 9, 12, 24, seed=8, affine=True)
    b = dict(a, b_k=np.random.default_rng(1).standard_normal(12))
    np.testing.assert_allclose(_call_full(b, 3, 1e-6), _call_full(a, 3, 1e-6), rtol=0, atol=1e-12)


def test_value_bias_alone_gives_constant_heads():
    # w_v = 0: every value row is b_v, and attention weights sum to one, so o = b_v
    a = _rand_block(2, 9, 12, 24, seed=9)
    c = np.random.default_rng(2).standard_normal(12)
    a = dict(a, w_v=np.zeros((12, 12)), b_v=c)
    _, st = _call_full(a, 3, 1e-6, stages=True)
    np.testing.assert_allclose(st["o"], np.broadcast_to(c, st["o"].shape), rtol=0, atol=1e-14)


def test_output_bias_with_zero_wo():
    a = _rand_block(2, 9, 12, 24, seed=10)
    c = np.random.default_rng(3).standard_normal(12)
    a = dict(a, w_o=np.zeros((12, 12)), b_o=c)
    _, st = _call_full(a, 3, 1e-6, stages=True)
    np.testing.assert_array_equal(st["y"], a["x"] + c)


def test_encoder_single_layer_is_the_block():
    a = _with_proj_biases(_rand_block(2, 9, 12, 24, seed=11, affine=True), seed=4)
    lay = {k: v for k, v in a.items() if k != "x"}
    np.testing.assert_array_equal(oracle.vit_encoder(a["x"], [lay], 3, 1e-6, final_ln=False),
                                  _call_full(a, 3, 1e-6))


@pytest.mark.parametrize("L,shape", [(3, (2, 9, 12, 24, 3)), (2, (1, 33, 16, 64, 2)), (4, (2, 5, 8, 16, 2))])
def test_encoder_matches_torch_stack(L, shape):
    N, T, D, F, H = shape
    rng = np.random.default_rng(L)
    x = rng.standard_normal((N, T, D))
    layers = _rand_layers(L, D, F, seed=50 + L)
    g, b = 1 + 0.1 * rng.standard_normal(D), 0.1 * rng.standard_normal(D)
    np.testing.assert_allclose(oracle.vit_encoder(x, layers, H, 1e-6, lnf_g=g, lnf_b=b),
                               _torch_encoder(x, layers, H, 1e-6, g, b), rtol=0, atol=1e-11)
    np.testing.assert_allclose(oracle.vit_encoder(x, layers, H, 1e-6, final_ln=False),
                               _torch_encoder(x, layers, H, 1e-6, final_ln=False), rtol=0, atol=1e-11)


def test_encoder_without_updates_is_layernorm_of_x():
    # every block with w_o = 0 and w_mlp2 = 0 (no biases) returns its input exactly, so the
    # stack is the final LayerNorm of x
    rng = np.random.default_rng(12)
    x = rng.standard_normal((2, 7, 12))
    layers = _rand_layers(3, 12, 24, seed=70, affine=True, biases=False)
    for lay in layers:
        lay.update(w_o=np.zeros((12, 12)), w_mlp2=np.zeros((24, 12)), b2=np.zeros(12))
    np.testing.assert_array_equal(oracle.vit_encoder(x, layers, 3, 1e-6, final_ln=False), x)
    np.testing.assert_array_equal(oracle.vit_encoder(x, layers, 3, 1e-6), oracle.layernorm(x, 1e-6))


# --------------------------------------------------------------- CLS-only last block

def _call_cls(a, H, eps, **kw):
    return oracle.vit_block_cls(a["x"], a["w_q"], a["w_k"], a["w_v"], a["w_o"], a["w_mlp1"],
                                a["w_mlp2"], H, eps, **{k: a.get(k) for k in
                                                        ("ln1_g", "ln1_b", "ln2_g", "ln2_b", "b1", "b2",
                                                         "b_q", "b_k", "b_v", "b_o")}, **kw)


@pytest.mark.parametrize("shape", [(2, 7, 12, 20, 3), (3, 5, 6, 6, 6), (2, 33, 16, 64, 1),
                                   (1, 197, 192, 768, 3), (2, 2, 8, 16, 2)])
def test_cls_block_is_row0_of_torch_block(shape):
    # the readout is row 0 of the whole block, whose float64 PyTorch composition is an
    # independent statement of it
    N, T, D, F, H = shape
    a = _with_proj_biases(_rand_block(N, T, D, F, seed=sum(shape), affine=True), seed=6)
    np.testing.assert_allclose(_call_cls(a, H, 1e-6), _torch_block(a, H, 1e-6)[:, 0], rtol=0, atol=1e-11)


def test_cls_block_is_row0_of_the_oracle_block():
    a = _with_proj_biases(_rand_block(3, 11, 12, 24, seed=13, affine=True), seed=8)
    np.testing.assert_array_equal(_call_cls(a, 3, 1e-6), _call_full(a, 3, 1e-6)[:, 0])


def test_cls_block_single_token():
    # T = 1: the one query sees only its own key, so the attention output is its value row
    a = _rand_block(4, 1, 8, 16, seed=14)
    a = dict(a, w_o=np.eye(8), w_mlp2=np.zeros((16, 8)))
    xn = oracle.layernorm(a["x"][:, 0], 1e-6)
    np.testing.assert_allclose(_call_cls(a, 2, 1e-6), a["x"][:, 0] + xn @ a["w_v"], rtol=0, atol=1e-13)


@pytest.mark.parametrize("L", [1, 2, 3])
def test_encoder_cls_matches_torch_stack(L):
    rng = np.random.default_rng(40 + L)
    x = rng.standard_normal((2, 9, 12))
    layers = _rand_layers(L, 12, 24, seed=60 + L)
    g, b = 1 + 0.1 * rng.standard_normal(12), 0.1 * rng.standard_normal(12)
    np.testing.assert_allclose(oracle.vit_encoder(x, layers, 3, 1e-6, lnf_g=g, lnf_b=b, cls_only=True),
                               _torch_encoder(x, layers, 3, 1e-6, g, b)[:, 0], rtol=0, atol=1e-11)
    np.testing.assert_allclose(oracle.vit_encoder(x, layers, 3, 1e-6, final_ln=False, cls_only=True),
                               _torch_encoder(x, layers, 3, 1e-6, final_ln=False)[:, 0], rtol=0, atol=1e-11)


# --------------------------------------------------------------- patch embedding front end

def _rand_images(N, C, H, W, P, D, seed):
    rng = np.random.default_rng(seed)
    T = (H // P) * (W // P) + 1
    return (rng.standard_normal((N, C, H, W)), rng.standard_normal((C * P * P, D)) / np.sqrt(C * P * P),
            rng.standard_normal(D), rng.standard_normal(D), rng.standard_normal((T, D)))


def _torch_patch_rows(im, P, order):
    t = torch.from_numpy(im)
    if order == 0:   # unfold: each patch channel by channel, each channel row by row
        return Fn.unfold(t, P, stride=P).transpose(1, 2)
    N, C, H, W = t.shape   # (p1, p2, c): reshape and permute
    t = t.reshape(N, C, H // P, P, W // P, P).permute(0, 2, 4, 3, 5, 1)
    return t.reshape(N, (H // P) * (W // P), P * P * C)


@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("shape", [(2, 3, 32, 48, 16, 20), (1, 1, 8, 8, 4, 16), (2, 3, 28, 14, 14, 12)])
def test_patch_embed_matches_torch(order, shape):
    N, C, H, W, P, D = shape
    im, w, b, cls, pos = _rand_images(N, C, H, W, P, D, seed=sum(shape) + order)
    rows = _torch_patch_rows(im, P, order) @ torch.from_numpy(w) + torch.from_numpy(b)
    ref = torch.cat([torch.from_numpy(cls).expand(N, 1, D), rows], 1) + torch.from_numpy(pos)
    got = oracle.patch_embed(im, P, w, b, cls=cls, pos=pos, order=order)
    np.testing.assert_allclose(got, ref.numpy(), rtol=0, atol=1e-12)


def test_patch_embed_channel_order_is_the_stride_p_convolution():
    # the lecture's second implementation: the projection weights reshaped into D filters
    # of C x P x P applied by a stride-P convolution give the same rows
    N, C, H, W, P, D = 2, 3, 32, 32, 16, 8
    im, w, b, _, _ = _rand_images(N, C, H, W, P, D, seed=3)
    conv = Fn.conv2d(torch.from_numpy(im), torch.from_numpy(w.T.reshape(D, C, P, P).copy()),
                     torch.from_numpy(b), stride=P)
    ref = conv.flatten(2).transpose(1, 2).numpy()
    np.testing.assert_allclose(oracle.patch_embed(im, P, w, b, order=0), ref, rtol=0, atol=1e-12)


def test_patch_embed_printed_flat_index():
    g = _load("p5_patch_flat_index.json")
    C, P, px = g["channels"], g["patch"], g["pixel"]
    im = np.zeros((1, C, P, P))
    im[0, px["channel"], px["row"], px["col"]] = 1.0
    K = C * P * P
    out = oracle.patch_embed(im, P, np.eye(K), order=0)   # identity projection: the flat patch
    assert out.shape == (1, 1, K)
    assert np.flatnonzero(out[0, 0]).tolist() == [g["flat_index"]]


def test_patchify_printed_example_order_p1_p2_c():
    """The page's printed patchify example pins flatten order 1, (p1, p2, c)."""
    g = _load("p3_patchify_example.json")
    shape = tuple(g["image_shape"])
    im = np.arange(float(np.prod(shape))).reshape(shape)
    N, C, H, W = shape
    P = g["patch"]
    K = C * P * P
    out = oracle.patch_embed(im, P, np.eye(K), order=1)   # identity projection, no CLS row
    assert out.shape == tuple(g["out_shape"])
    np.testing.assert_array_equal(out[0, 0], np.array(g["first_patch"], dtype=float))
    # and order 0 (channel by channel) differs from the printed patch
    assert not np.array_equal(oracle.patch_embed(im, P, np.eye(K), order=0)[0, 0], out[0, 0])


def test_patch_embed_cls_and_positions():
    N, C, H, W, P, D = 2, 3, 16, 16, 8, 6
    im, _, _, cls, pos = _rand_images(N, C, H, W, P, D, seed=4)
    out = oracle.patch_embed(im, P, np.zeros((C * P * P, D)), np.zeros(D), cls=cls, pos=pos)
    np.testing.assert_array_equal(out[:, 0], np.broadcast_to(cls + pos[0], (N, D)))
    np.testing.assert_array_equal(out[:, 1:], np.broadcast_to(pos[1:], (N, pos.shape[0] - 1, D)))


MUTANTS = {
    "eps_fixed_1e-5": ("sqrt(var + eps)", "sqrt(var + 1e-5)"),
    "sample_variance": ("var /= (double)D;", "var /= (double)(D - 1 > 0 ? D - 1 : 1);"),
    "drop_residual_1": ("y[i] = xs[i] + a[i];", "y[i] = a[i];"),
    "residual_1_on_normalised": ("y[i] = xs[i] + a[i];", "y[i] = xn[i] + a[i];"),
    "drop_residual_2": ("os[i] = y[i] + a[i];", "os[i] = a[i];"),
    "residual_2_on_x": ("os[i] = y[i] + a[i];", "os[i] = xs[i] + a[i];"),
    "ln2_of_x": ("oracle_layernorm(y, T, D, eps, ln2_g, ln2_b, yn);",
                 "oracle_layernorm(xs, T, D, eps, ln2_g, ln2_b, yn);"),
    "shared_ln_params": ("oracle_layernorm(y, T, D, eps, ln2_g, ln2_b, yn);",
                         "oracle_layernorm(y, T, D, eps, ln1_g, ln1_b, yn);"),
    "weight_transposed": ("const double* w = W + k * N;\n            for (int64_t n = 0; n < N; ++n) c[n] += a * w[n];",
                          "for (int64_t n = 0; n < N; ++n) c[n] += a * W[n * K + k];"),
    "head_offset_zero": ("const int64_t c0 = h * dh;", "const int64_t c0 = 0 * h;"),
    "score_scale_sqrt_D": ("const double scale = sqrt((double)dh);", "const double scale = sqrt((double)D);"),
    "score_scale_missing": ("s[u] = dot / scale;", "s[u] = dot + 0.0 * scale;"),
    "causal_mask": ("s[u] = dot / scale;", "s[u] = (u > t) ? -INFINITY : dot / scale;"),
    "gelu_erf": ("return 0.5 * z * (1.0 + tanh(sqrt(2.0 / pi) * (z + 0.044715 * z * z * z)));",
                 "return 0.5 * z * (1.0 + erf(z / sqrt(2.0))) + 0.0 * pi;"),
    "gelu_constant": ("0.044715 * z * z * z", "0.04471 * z * z * z"),
    "gelu_square": ("0.044715 * z * z * z", "0.044715 * z * z"),
    "drop_b1": ("oracle_matmul(yn, w_mlp1, b1, T, D, F, z);", "oracle_matmul(yn, w_mlp1, NULL, T, D, F, z);"),
    "wk_for_wv": ("oracle_matmul(xn, w_v, b_v, T, D, D, v);", "oracle_matmul(xn, w_k, b_v, T, D, D, v);"),
    "drop_b_q": ("oracle_matmul(xn, w_q, b_q, T, D, D, q);", "oracle_matmul(xn, w_q, NULL, T, D, D, q);"),
    "drop_b_v": ("oracle_matmul(xn, w_v, b_v, T, D, D, v);", "oracle_matmul(xn, w_v, NULL, T, D, D, v);"),
    "drop_b_o": ("oracle_matmul(o, w_o, b_o, T, D, D, a);", "oracle_matmul(o, w_o, NULL, T, D, D, a);"),
    "encoder_reuses_layer0": ("const double* const* w = layers + (size_t)l * 16;",
                              "const double* const* w = layers + (size_t)l * 0;"),
    "encoder_restarts_from_x": ("        cur = nxt;\n", "        cur = (l + 1 < L) ? x : nxt;\n"),
    "final_ln_without_affine": ("oracle_layernorm(cur, N * T, D, eps, lnf_g, lnf_b, out);",
                                "oracle_layernorm(cur, N * T, D, eps, NULL, NULL, out);"),
    "patch_orders_swapped": ("order == 0 ? (c * P + i) * P + j : (i * P + j) * C + c",
                             "order == 1 ? (c * P + i) * P + j : (i * P + j) * C + c"),
    "patch_rows_transposed": ("for (int64_t i = 0; i < P; ++i)\n                        for (int64_t j = 0; j < P; ++j) {\n                            const double v = images[(((size_t)n * C + c) * Hi + py * P + i) * Wi + px * P + j];",
                              "for (int64_t i = 0; i < P; ++i)\n                        for (int64_t j = 0; j < P; ++j) {\n                            const double v = images[(((size_t)n * C + c) * Hi + py * P + j) * Wi + px * P + i];"),
    "pos_skips_cls_row": ("for (int64_t t = 0; t < T; ++t)\n                for (int64_t d = 0; d < D; ++d) o[(size_t)t * D + d] += pos[(size_t)t * D + d];",
                          "for (int64_t t = 1; t < T; ++t)\n                for (int64_t d = 0; d < D; ++d) o[(size_t)t * D + d] += pos[(size_t)t * D + d];"),
    "cls_query_from_row1": ("oracle_matmul(xn, w_q, b_q, 1, D, D, q0);",
                            "oracle_matmul(xn + D, w_q, b_q, 1, D, D, q0);"),
    "cls_drop_b_q": ("oracle_matmul(xn, w_q, b_q, 1, D, D, q0);", "oracle_matmul(xn, w_q, NULL, 1, D, D, q0);"),
    "cls_keys_without_ln": ("oracle_matmul(xn, w_k, b_k, T, D, D, keys);",
                            "oracle_matmul(xs, w_k, b_k, T, D, D, keys);"),
    "cls_first_key_only": ("oracle_softmax_rows(sc, 1, T, pw);",
                           "oracle_softmax_rows(sc, 1, 1, pw);\n            for (int64_t u = 1; u < T; ++u) pw[u] = 0.0;"),
    "cls_residual_on_normalised": ("y0[j] = xs[j] + a0[j];", "y0[j] = xn[j] + a0[j];"),
    "cls_skips_earlier_blocks": ("rc = oracle_vit_block_cls(L > 1 ? body : x,", "rc = oracle_vit_block_cls(x,"),
    "cls_final_ln_skipped": ("oracle_layernorm(c, N, D, eps, lnf_g, lnf_b, out);",
                             "memcpy(out, c, sizeof(double) * (size_t)(N * D));"),
    "drop_patch_bias": ("                if (b)\n                    for (int64_t d = 0; d < D; ++d) row[d] += b[d];",
                        "                if (b && 0)\n                    for (int64_t d = 0; d < D; ++d) row[d] += b[d];"),
}


def _pins_pass(lib):
    """Run the whole-block pins (worked examples + library composition) on a library."""
    g = _load("p2_worked_examples.json")
    for ex in g["examples"]:
        out = _call(_p2_args(ex), ex["num_heads"], g["eps"], lib=lib)
        if not np.allclose(out, np.array(ex["output"]), rtol=0, atol=g["print_tolerance"]):
            return False
    for shape, affine in (((2, 7, 12, 20, 3), False), ((2, 7, 12, 20, 3), True)):
        N, T, D, F, H = shape
        a = _rand_block(N, T, D, F, seed=21, affine=affine)
        if not np.allclose(_call(a, H, 1e-5, lib=lib), _torch_block(a, H, 1e-5), rtol=0, atol=1e-11):
            return False
    # projection biases and the stack with its final LayerNorm
    a = _with_proj_biases(_rand_block(2, 7, 12, 20, seed=22, affine=True), seed=5)
    if not np.allclose(_call_full(a, 3, 1e-5, lib=lib), _torch_block(a, 3, 1e-5), rtol=0, atol=1e-11):
        return False
    rng = np.random.default_rng(23)
    x = rng.standard_normal((2, 7, 12))
    layers = _rand_layers(3, 12, 20, seed=90)
    g, b = 1 + 0.1 * rng.standard_normal(12), 0.1 * rng.standard_normal(12)
    got = oracle.vit_encoder(x, layers, 3, 1e-5, lnf_g=g, lnf_b=b, lib=lib)
    if not np.allclose(got, _torch_encoder(x, layers, 3, 1e-5, g, b), rtol=0, atol=1e-11):
        return False
    # the CLS-only readout of one block and of a stack
    a = _with_proj_biases(_rand_block(2, 7, 12, 20, seed=25, affine=True), seed=6)
    if not np.allclose(_call_cls(a, 3, 1e-5, lib=lib), _torch_block(a, 3, 1e-5)[:, 0], rtol=0, atol=1e-11):
        return False
    got = oracle.vit_encoder(x, layers, 3, 1e-5, lnf_g=g, lnf_b=b, lib=lib, cls_only=True)
    if not np.allclose(got, _torch_encoder(x, layers, 3, 1e-5, g, b)[:, 0], rtol=0, atol=1e-11):
        return False
    # patch embedding, both orders, with the CLS row and positions
    im, w, bb, cls, pos = _rand_images(2, 3, 16, 24, 8, 10, seed=24)
    for order in (0, 1):
        rows = _torch_patch_rows(im, 8, order) @ torch.from_numpy(w) + torch.from_numpy(bb)
        ref = torch.cat([torch.from_numpy(cls).expand(2, 1, 10), rows], 1) + torch.from_numpy(pos)
        got = oracle.patch_embed(im, 8, w, bb, cls=cls, pos=pos, order=order, lib=lib)
        if not np.allclose(got, ref.numpy(), rtol=0, atol=1e-12):
            return False
    return True


def test_pins_pass_on_unmodified_source(tmp_path):
    src = open(oracle._SRC).read()
    p = tmp_path / "clean.c"
    p.write_text(src)
    lib = oracle.open_library(oracle.build(force=True, src=str(p), out=str(tmp_path / "clean.so")))
    assert _pins_pass(lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutants(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, name
    p = tmp_path / ("m_%s.c" % name)
    p.write_text(src.replace(old, new))
    lib = oracle.open_library(oracle.build(force=True, src=str(p), out=str(tmp_path / ("m_%s.so" % name))))
    assert not _pins_pass(lib), "planted slip %r was not caught" % name
