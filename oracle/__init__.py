"""Plain float64 CPU oracle of one pre-LayerNorm ViT encoder block.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package. The CUDA library never calls it and
shares no code with it.

The arithmetic lives in ``vit_oracle.c`` (straight float64 loops, OpenMP over
sequences). This module compiles it with the host C compiler on first use and
marshals numpy float64 arrays to it. Every input is converted to float64 exactly
(bf16 and fp32 values are representable in float64), so the oracle sees the very
values a lower-precision caller stored.

Passages followed (see the C file for each function):
  "ViT Encoder Block" (crackedaicode): "Normalize before each stage",
  "Multi-head attention", "Feed-forward stage".
  "ViT Encoder Block" (ai-engineer-exhaustive), Key Equations Steps 1-6 for the
  optional LN gain/bias and MLP biases.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vit_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libvit_oracle.so")
_lock = threading.Lock()
_lib = None

_dptr = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle C source into a shared library (gcc, OpenMP, IEEE float64,
    no contraction of a*b+c into fused multiply-adds)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def open_library(path: str):
    """Open a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    lib.oracle_layernorm.argtypes = [_dptr, _i64, _i64, ctypes.c_double, _dptr, _dptr, _dptr]
    lib.oracle_layernorm.restype = None
    lib.oracle_gelu_tanh.argtypes = [ctypes.c_double]
    lib.oracle_gelu_tanh.restype = ctypes.c_double
    lib.oracle_gelu_tanh_array.argtypes = [_dptr, _i64, _dptr]
    lib.oracle_gelu_tanh_array.restype = None
    lib.oracle_matmul.argtypes = [_dptr, _dptr, _dptr, _i64, _i64, _i64, _dptr]
    lib.oracle_matmul.restype = None
    lib.oracle_softmax_rows.argtypes = [_dptr, _i64, _i64, _dptr]
    lib.oracle_softmax_rows.restype = None
    lib.oracle_attention.argtypes = [_dptr, _dptr, _dptr, _i64, _i64, _i64, _i64, _dptr]
    lib.oracle_attention.restype = None
    lib.oracle_vit_block.argtypes = ([_dptr] * 13 + [_i64] * 5 + [ctypes.c_double]
                                     + [_dptr] * 7 + [ctypes.c_int])
    lib.oracle_vit_block.restype = ctypes.c_int
    lib.oracle_vit_block_full.argtypes = ([_dptr] * 17 + [_i64] * 5 + [ctypes.c_double]
                                          + [_dptr] * 7 + [ctypes.c_int])
    lib.oracle_vit_block_full.restype = ctypes.c_int
    lib.oracle_vit_encoder.argtypes = [_dptr, ctypes.POINTER(_dptr), _i64, _dptr, _dptr, ctypes.c_int,
                                       _i64, _i64, _i64, _i64, _i64, ctypes.c_double, _dptr, ctypes.c_int]
    lib.oracle_vit_encoder.restype = ctypes.c_int
    lib.oracle_vit_block_cls.argtypes = [_dptr] * 17 + [_i64] * 5 + [ctypes.c_double, _dptr, ctypes.c_int]
    lib.oracle_vit_block_cls.restype = ctypes.c_int
    lib.oracle_vit_encoder_cls.argtypes = lib.oracle_vit_encoder.argtypes
    lib.oracle_vit_encoder_cls.restype = ctypes.c_int
    lib.oracle_patch_embed.argtypes = [_dptr, _i64, _i64, _i64, _i64, _i64, ctypes.c_int, _dptr, _dptr,
                                       _dptr, _dptr, _i64, _dptr]
    lib.oracle_patch_embed.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = open_library(build())
        return _lib


def _f64(a):
    """Exact float64, C-contiguous numpy copy of a numpy array or torch tensor."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor: widen on the CPU first (exact for bf16/f32)
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a):
    return None if a is None else a.ctypes.data_as(_dptr)


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def layernorm(x, eps, gamma=None, beta=None):
    x = _f64(x)
    g, b = _f64(gamma), _f64(beta)
    D = x.shape[-1]
    out = np.empty_like(x)
    _load().oracle_layernorm(_p(x), x.size // D, D, float(eps), _p(g), _p(b), _p(out))
    return out


def gelu_tanh(z):
    z = _f64(z)
    out = np.empty_like(z)
    _load().oracle_gelu_tanh_array(_p(z), z.size, _p(out))
    return out


def matmul(a, w, bias=None):
    a, w, b = _f64(a), _f64(w), _f64(bias)
    K, N = w.shape
    M = a.size // K
    out = np.empty(a.shape[:-1] + (N,), dtype=np.float64)
    _load().oracle_matmul(_p(a), _p(w), _p(b), M, K, N, _p(out))
    return out


def softmax_rows(s):
    s = _f64(s)
    n = s.shape[-1]
    out = np.empty_like(s)
    _load().oracle_softmax_rows(_p(s), s.size // n, n, _p(out))
    return out


def attention(q, k, v, H):
    """q, k, v: (N, T, D); returns the concatenated head outputs (N, T, D)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    N, T, D = q.shape
    out = np.empty_like(q)
    _load().oracle_attention(_p(q), _p(k), _p(v), N, T, D, H, _p(out))
    return out


def vit_block(x, w_q, w_k, w_v, w_o, w_mlp1, w_mlp2, H, eps, ln1_g=None, ln1_b=None,
              ln2_g=None, ln2_b=None, b1=None, b2=None, stages=False, nthreads=0, lib=None):
    """Block output (N, T, D) in float64; with stages=True also a dict of the
    intermediate values xn, qkv, o, y, yn, g."""
    arrs = [_f64(a) for a in (x, w_q, w_k, w_v, w_o, w_mlp1, w_mlp2)]
    opt = [_f64(a) for a in (ln1_g, ln1_b, ln2_g, ln2_b, b1, b2)]
    x64 = arrs[0]
    if x64.ndim == 2:
        x64 = x64[None]
        arrs[0] = x64
    N, T, D = x64.shape
    F = arrs[5].shape[1]
    out = np.empty_like(x64)
    st = {}
    if stages:
        st = {"xn": np.empty((N, T, D)), "qkv": np.empty((N, T, 3 * D)), "o": np.empty((N, T, D)),
              "y": np.empty((N, T, D)), "yn": np.empty((N, T, D)), "g": np.empty((N, T, F))}
    names = ("xn", "qkv", "o", "y", "yn", "g")
    rc = (lib or _load()).oracle_vit_block(*[_p(a) for a in arrs], *[_p(a) for a in opt],
                                  N, T, D, F, int(H), float(eps), _p(out),
                                  *[_p(st.get(k)) for k in names], int(nthreads))
    if rc != 0:
        raise ValueError("oracle_vit_block failed with status %d" % rc)
    return (out, st) if stages else out


def vit_block_full(x, w_q, w_k, w_v, w_o, w_mlp1, w_mlp2, H, eps, ln1_g=None, ln1_b=None,
                   ln2_g=None, ln2_b=None, b1=None, b2=None, b_q=None, b_k=None, b_v=None,
                   b_o=None, stages=False, nthreads=0, lib=None):
    """vit_block with the optional Q, K, V and output-projection biases."""
    arrs = [_f64(a) for a in (x, w_q, w_k, w_v, w_o, w_mlp1, w_mlp2)]
    opt = [_f64(a) for a in (ln1_g, ln1_b, ln2_g, ln2_b, b1, b2, b_q, b_k, b_v, b_o)]
    x64 = arrs[0]
    if x64.ndim == 2:
        x64 = x64[None]
        arrs[0] = x64
    N, T, D = x64.shape
    F = arrs[5].shape[1]
    out = np.empty_like(x64)
    st = {}
    if stages:
        st = {"xn": np.empty((N, T, D)), "qkv": np.empty((N, T, 3 * D)), "o": np.empty((N, T, D)),
              "y": np.empty((N, T, D)), "yn": np.empty((N, T, D)), "g": np.empty((N, T, F))}
    names = ("xn", "qkv", "o", "y", "yn", "g")
    rc = (lib or _load()).oracle_vit_block_full(*[_p(a) for a in arrs], *[_p(a) for a in opt],
                                       N, T, D, F, int(H), float(eps), _p(out),
                                       *[_p(st.get(k)) for k in names], int(nthreads))
    if rc != 0:
        raise ValueError("oracle_vit_block_full failed with status %d" % rc)
    return (out, st) if stages else out


LAYER_KEYS = ("w_q", "w_k", "w_v", "w_o", "w_mlp1", "w_mlp2", "ln1_g", "ln1_b", "ln2_g",
              "ln2_b", "b1", "b2", "b_q", "b_k", "b_v", "b_o")


def vit_block_cls(x, w_q, w_k, w_v, w_o, w_mlp1, w_mlp2, H, eps, ln1_g=None, ln1_b=None,
                  ln2_g=None, ln2_b=None, b1=None, b2=None, b_q=None, b_k=None, b_v=None,
                  b_o=None, nthreads=0, lib=None):
    """The CLS-only readout of one block: row 0 of each sequence's block output, computed
    from the one CLS query against all T keys and values. Returns (N, D) float64."""
    arrs = [_f64(a) for a in (x, w_q, w_k, w_v, w_o, w_mlp1, w_mlp2)]
    opt = [_f64(a) for a in (ln1_g, ln1_b, ln2_g, ln2_b, b1, b2, b_q, b_k, b_v, b_o)]
    x64 = arrs[0]
    if x64.ndim == 2:
        x64 = x64[None]
        arrs[0] = x64
    N, T, D = x64.shape
    F = arrs[5].shape[1]
    out = np.empty((N, D))
    rc = (lib or _load()).oracle_vit_block_cls(*[_p(a) for a in arrs], *[_p(a) for a in opt],
                                               N, T, D, F, int(H), float(eps), _p(out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_vit_block_cls failed with status %d" % rc)
    return out


def vit_encoder(x, layers, H, eps, lnf_g=None, lnf_b=None, final_ln=True, nthreads=0, lib=None,
                cls_only=False):
    """A stack of blocks (layers: a list of dicts keyed by LAYER_KEYS; the six weights
    required, the rest optional) and, with final_ln, the final LayerNorm. Float64.
    cls_only: the last block is the CLS-only readout and the result is (N, D)."""
    x64 = _f64(x)
    if x64.ndim == 2:
        x64 = x64[None]
    N, T, D = x64.shape
    L = len(layers)
    keep = []
    ptrs = (_dptr * (16 * L))()
    F = None
    for l, lay in enumerate(layers):
        for j, key in enumerate(LAYER_KEYS):
            a = _f64(lay.get(key))
            keep.append(a)
            ptrs[16 * l + j] = _p(a) if a is not None else _dptr()
        F = _f64(lay["w_mlp1"]).shape[1]
    g, b = _f64(lnf_g), _f64(lnf_b)
    lib = lib or _load()
    out = np.empty((N, D)) if cls_only else np.empty_like(x64)
    fn = lib.oracle_vit_encoder_cls if cls_only else lib.oracle_vit_encoder
    rc = fn(_p(x64), ptrs, L, _p(g), _p(b), 1 if final_ln else 0,
            N, T, D, int(F), int(H), float(eps), _p(out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_vit_encoder failed with status %d" % rc)
    return out


def patch_embed(images, P, w, b=None, cls=None, pos=None, order=0, lib=None):
    """Tokens (N, T, D) in float64 from images (N, C, Hi, Wi): patches of P x P flattened in
    `order` (0: channel, row, column; 1: row, column, channel), @ w (+ b), the cls row
    prepended when given, pos (T, D) added when given."""
    im = _f64(images)
    N, C, Hi, Wi = im.shape
    w64, b64, c64, p64 = _f64(w), _f64(b), _f64(cls), _f64(pos)
    D = w64.shape[1]
    T = (Hi // P) * (Wi // P) + (1 if cls is not None else 0)
    out = np.empty((N, T, D), dtype=np.float64)
    rc = (lib or _load()).oracle_patch_embed(_p(im), N, C, Hi, Wi, int(P), int(order), _p(w64), _p(b64),
                                             _p(c64), _p(p64), D, _p(out))
    if rc != 0:
        raise ValueError("oracle_patch_embed failed with status %d" % rc)
    return out
