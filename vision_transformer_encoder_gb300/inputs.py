"""Seeded synthetic inputs for the ViT encoder block.

This module draws random numbers and nothing else: it holds none of the block's
arithmetic, so both the CUDA path's tests/benchmark and the float64 oracle can
consume the same inputs without sharing any of the method.

Recipe (one CPU ``torch.Generator`` seeded with ``seed``, draws in this fixed order):
  x       ~ N(0, 1)                 (N, T, D)
  w_q, w_k, w_v, w_o ~ N(0, 1/D)    (D, D)   stored (in, out)
  w_mlp1  ~ N(0, 1/D)               (D, F)
  w_mlp2  ~ N(0, 1/F)               (F, D)
  then, only for the affine/bias variant:
  ln1_g, ln2_g ~ 1 + N(0, 0.02^2), ln1_b, ln2_b, b1, b2 ~ N(0, 0.02^2)
Everything is drawn in float32 and then cast to the run dtype; callers hand the
oracle the cast values, widened exactly to float64.

The weight scale N(0, 1/fan_in) and the 0.02 scale follow "E2E: Tiny Vision
Transformer" (mlgrind.dev), section "Details" (Initialization); gain 1 / bias 0 at
init follows the same section.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

# Block shapes of the workloads measured and parity-tested.
# ViT-B/L/H sizes: "ViT Encoder Block" (ai-engineer-exhaustive), "Paper Context";
# ViT-Ti sizes (D 192, 3 heads, MLP 768, 197 tokens): "vision1 reference transcript"
# (nipunbatra.github.io), Pages 17, 53 and 74. Token counts 197/577/1025 are
# 14x14, 24x24 and 32x32 patch grids plus one class token.
CONFIGS = {
    "tiny": dict(N=2, T=5, D=8, H=2, F=16, eps=1e-5),
    "vit_ti16": dict(N=64, T=197, D=192, H=3, F=768, eps=1e-5),
    "vit_b16": dict(N=256, T=197, D=768, H=12, F=3072, eps=1e-6),
    "vit_l16_384": dict(N=64, T=577, D=1024, H=16, F=4096, eps=1e-5),
    "vit_h14_448": dict(N=32, T=1025, D=1280, H=16, F=5120, eps=1e-6),
}

WEIGHT_NAMES = ("w_q", "w_k", "w_v", "w_o", "w_mlp1", "w_mlp2")
AFFINE_NAMES = ("ln1_g", "ln1_b", "ln2_g", "ln2_b", "b1", "b2")


@dataclass
class BlockInputs:
    x: torch.Tensor
    w_q: torch.Tensor
    w_k: torch.Tensor
    w_v: torch.Tensor
    w_o: torch.Tensor
    w_mlp1: torch.Tensor
    w_mlp2: torch.Tensor
    ln1_g: torch.Tensor | None = None
    ln1_b: torch.Tensor | None = None
    ln2_g: torch.Tensor | None = None
    ln2_b: torch.Tensor | None = None
    b1: torch.Tensor | None = None
    b2: torch.Tensor | None = None

    def weights(self):
        return [getattr(self, n) for n in WEIGHT_NAMES]

    def affine(self):
        return {n: getattr(self, n) for n in AFFINE_NAMES}

    def to(self, device=None, dtype=None):
        def cv(t):
            if t is None:
                return None
            return t.to(device=device if device is not None else t.device,
                        dtype=dtype if dtype is not None else t.dtype).contiguous()
        return BlockInputs(**{k: cv(v) for k, v in self.__dict__.items()})


def make_inputs(N, T, D, F, seed=0, affine=False, dtype=torch.float32, device="cpu",
                x_scale=1.0) -> BlockInputs:
    """Draw one seeded set of block inputs (see the module docstring for the recipe)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))

    def normal(*shape, std=1.0):
        return torch.randn(*shape, generator=g, dtype=torch.float32) * std

    x = normal(N, T, D) * x_scale
    w = {}
    for name in ("w_q", "w_k", "w_v", "w_o"):
        w[name] = normal(D, D, std=D ** -0.5)
    w["w_mlp1"] = normal(D, F, std=D ** -0.5)
    w["w_mlp2"] = normal(F, D, std=F ** -0.5)
    extra = {}
    if affine:
        extra["ln1_g"] = 1.0 + normal(D, std=0.02)
        extra["ln1_b"] = normal(D, std=0.02)
        extra["ln2_g"] = 1.0 + normal(D, std=0.02)
        extra["ln2_b"] = normal(D, std=0.02)
        extra["b1"] = normal(F, std=0.02)
        extra["b2"] = normal(D, std=0.02)
    inp = BlockInputs(x=x, **w, **extra)
    return inp.to(device=device, dtype=dtype)


def make_config_inputs(name, seed=0, affine=False, dtype=torch.float32, device="cpu", N=None):
    c = CONFIGS[name]
    return make_inputs(N if N is not None else c["N"], c["T"], c["D"], c["F"], seed=seed,
                       affine=affine, dtype=dtype, device=device)


def make_encoder_inputs(N, T, D, F, L, seed=0, affine=True, biases=True, dtype=torch.float32,
                        device="cpu"):
    """Inputs of an L-block stack: x, a list of per-layer dicts (the block's weights and
    affine terms, drawn as make_inputs does with seed + 1000 l, plus, with biases, the Q, K,
    V and output-projection biases ~ N(0, 0.02^2)) and the final LayerNorm's gain and bias
    (1 + N(0, 0.02^2), N(0, 0.02^2)). Everything is drawn in fp32 and cast to dtype."""
    x = make_inputs(N, T, D, F, seed=seed, dtype=dtype, device=device).x
    layers = []
    for l in range(L):
        b = make_inputs(1, 1, D, F, seed=seed + 1000 * (l + 1), affine=affine)
        lay = {n: getattr(b, n) for n in WEIGHT_NAMES}
        if affine:
            lay.update(b.affine())
        if biases:
            g = torch.Generator(device="cpu")
            g.manual_seed(int(seed + 1000 * (l + 1) + 7))
            for n in ("b_q", "b_k", "b_v", "b_o"):
                lay[n] = torch.randn(D, generator=g, dtype=torch.float32) * 0.02
        layers.append({k: (v.to(device=device, dtype=dtype).contiguous() if v is not None else None)
                       for k, v in lay.items()})
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed + 7))
    lnf_g = (1.0 + torch.randn(D, generator=g) * 0.02).to(device=device, dtype=dtype)
    lnf_b = (torch.randn(D, generator=g) * 0.02).to(device=device, dtype=dtype)
    return x, layers, lnf_g, lnf_b
