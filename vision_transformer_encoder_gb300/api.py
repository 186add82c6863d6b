"""Python binding of the C ABI in include/vit_block.h (argument marshalling only).

Every computation runs in the CUDA library ``libvit_block.so``; this module checks
that tensors are contiguous and on the right device, picks the element-type code,
passes raw pointers and the current CUDA stream, and turns a non-zero status into
``VitError``. There is no fallback: if the library is missing, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libvit_block.so")

VIT_F32, VIT_BF16, VIT_F64 = 0, 1, 2
EPI_STORE, EPI_GELU, EPI_RESIDUAL = 0, 1, 2

_DT = {torch.float32: VIT_F32, torch.bfloat16: VIT_BF16, torch.float64: VIT_F64}

LAYER_FIELDS = ("w_q", "w_k", "w_v", "w_o", "w_mlp1", "w_mlp2", "ln1_g", "ln1_b", "ln2_g", "ln2_b",
                "b1", "b2", "b_q", "b_k", "b_v", "b_o")


class VitLayer(ctypes.Structure):
    """vit_layer of include/vit_block.h: sixteen device pointers of one block."""
    _fields_ = [(name, ctypes.c_void_p) for name in LAYER_FIELDS]


# Every exported symbol of the C ABI, with (restype, argtypes).
_vp, _i64, _int, _dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
SIGNATURES = {
    "vit_block": (_int, [_vp] * 7 + [_i64] * 5 + [_dbl, _int, _vp, _vp]),
    "vit_block_ex": (_int, [_vp] * 13 + [_i64] * 5 + [_dbl, _int, _vp, _vp]),
    "vit_block_host": (_int, [_vp] * 13 + [_i64] * 5 + [_dbl, _int, _vp, _vp]),
    "vit_block_noalloc": (_int, [_vp] * 13 + [_i64] * 5 + [_dbl, _int, _vp, _vp]),
    "vit_encoder": (_int, [_vp, ctypes.POINTER(VitLayer), _i64, _vp, _vp, _int] + [_i64] * 5
                    + [_dbl, _int, _vp, _vp]),
    "vit_encoder_cls": (_int, [_vp, ctypes.POINTER(VitLayer), _i64, _vp, _vp, _int] + [_i64] * 5
                        + [_dbl, _int, _vp, _vp]),
    "vit_block_cls": (_int, [_vp, ctypes.POINTER(VitLayer)] + [_i64] * 5 + [_dbl, _int, _vp, _vp]),
    "vit_patch_embed": (_int, [_vp] + [_i64] * 5 + [_int] + [_vp] * 4 + [_i64, _int, _vp, _vp]),
    "vit_layernorm": (_int, [_vp, _i64, _i64, _dbl, _vp, _vp, _int, _vp, _int, _vp]),
    "vit_linear": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _int, _vp, _int, _vp]),
    "vit_attention": (_int, [_vp, _i64, _i64, _i64, _i64, _int, _vp, _vp]),
    "vit_weights_create": (_int, [ctypes.POINTER(VitLayer), _int, _i64, _i64, _i64, _int, _int,
                                  ctypes.POINTER(_vp), _vp]),
    "vit_weights_destroy": (_int, [_vp]),
    "vit_weights_info": (_int, [_vp, ctypes.POINTER(_i64), ctypes.POINTER(_i64), ctypes.POINTER(_i64),
                                ctypes.POINTER(_int), ctypes.POINTER(_int), ctypes.POINTER(_int)]),
    "vit_block_w": (_int, [_vp, _vp, _i64, _i64, _dbl, _vp, _vp]),
    "vit_block_w_host": (_int, [_vp, _vp, _i64, _i64, _dbl, _vp, _vp]),
    "vit_block_w_host_async": (_int, [_vp, _vp, _i64, _i64, _dbl, _vp, _vp]),
    "vit_status_string": (ctypes.c_char_p, [_int]),
    "vit_device_error": (_int, [ctypes.POINTER(ctypes.c_uint32)]),
    "vit_launch_count": (_i64, []),
    "vit_selftest_wait": (_int, [_int, _vp]),
    "vit_timing_enable": (_int, [_int]),
    "vit_timing_collect": (_int, []),
    "vit_timing_kernels": (_int, []),
    "vit_timing_read": (_int, [_int, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64),
                               ctypes.POINTER(ctypes.c_char_p)]),
    "vit_timing_reset": (_int, []),
    "vit_version": (ctypes.c_char_p, []),
}

_lock = threading.Lock()
_lib = None


class VitError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s failed: %s (status %d)" % (what, status_string(status), status))


def load_library(path: str | None = None):
    """Open libvit_block.so (built by ``vision_transformer_encoder_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError("the vit_block CUDA library is not built (%s missing); run "
                               "python -m vision_transformer_encoder_gb300.build" % p)
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        if path is None:
            _lib = lib
        return lib


def status_string(status: int) -> str:
    return load_library().vit_status_string(int(status)).decode()


def _check(rc: int, what: str):
    if rc != 0:
        raise VitError(rc, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t, name, dtype=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s has dtype %s, expected %s" % (name, t.dtype, dtype))
    return t


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(dt):
    if dt not in _DT:
        raise ValueError("unsupported dtype %s" % dt)
    return _DT[dt]


def vit_block_ex(x, w_q, w_k, w_v, w_o, w_mlp1, w_mlp2, H, eps, ln1_g=None, ln1_b=None,
                 ln2_g=None, ln2_b=None, b1=None, b2=None, out=None, stream=None):
    """out (N, T, D) = one pre-LN ViT encoder block of x (N, T, D); optional affine terms."""
    lib = load_library()
    dt = x.dtype
    ts = dict(x=x, w_q=w_q, w_k=w_k, w_v=w_v, w_o=w_o, w_mlp1=w_mlp1, w_mlp2=w_mlp2,
              ln1_g=ln1_g, ln1_b=ln1_b, ln2_g=ln2_g, ln2_b=ln2_b, b1=b1, b2=b2)
    for k, v in ts.items():
        _dev(v, k, dt)
    N, T, D = x.shape
    F = w_mlp1.shape[1]
    if out is None:
        out = torch.empty_like(x)
    _dev(out, "out", dt)
    with torch.cuda.device(x.device):
        rc = lib.vit_block_ex(*[_ptr(ts[k]) for k in ts], N, T, D, F, int(H), float(eps),
                              _dtype_code(dt), _ptr(out), _stream(stream))
    _check(rc, "vit_block_ex")
    return out


def vit_block(x, w_q, w_k, w_v, w_o, w_mlp1, w_mlp2, H, eps, out=None, stream=None):
    """out (N, T, D) = one pre-LN ViT encoder block of x (N, T, D), no affine terms."""
    lib = load_library()
    dt = x.dtype
    ws = [w_q, w_k, w_v, w_o, w_mlp1, w_mlp2]
    _dev(x, "x", dt)
    for i, w in enumerate(ws):
        _dev(w, "weight %d" % i, dt)
    N, T, D = x.shape
    F = w_mlp1.shape[1]
    if out is None:
        out = torch.empty_like(x)
    _dev(out, "out", dt)
    with torch.cuda.device(x.device):
        rc = lib.vit_block(_ptr(x), *[_ptr(w) for w in ws], N, T, D, F, int(H), float(eps),
                           _dtype_code(dt), _ptr(out), _stream(stream))
    _check(rc, "vit_block")
    return out


def _layer_array(layers, dt):
    arr = (VitLayer * max(len(layers), 1))()
    for i, lay in enumerate(layers):
        for name in LAYER_FIELDS:
            t = lay.get(name)
            _dev(t, "layer %d %s" % (i, name), dt)
            setattr(arr[i], name, None if t is None else t.data_ptr())
    return arr


def vit_encoder(x, layers, H, eps, lnf_g=None, lnf_b=None, final_ln=True, out=None, stream=None,
                cls_only=False):
    """out (N, T, D) = the stack of blocks in `layers` (a list of dicts keyed by
    LAYER_FIELDS: the six weights required, the rest optional), then, with final_ln,
    the final LayerNorm with the optional gain lnf_g and bias lnf_b. cls_only: the last
    block computes the CLS row alone (vit_encoder_cls) and out is (N, D)."""
    lib = load_library()
    dt = x.dtype
    _dev(x, "x", dt)
    arr = _layer_array(layers, dt)
    _dev(lnf_g, "lnf_g", dt)
    _dev(lnf_b, "lnf_b", dt)
    N, T, D = x.shape
    F = layers[0]["w_mlp1"].shape[1] if layers else 0
    if out is None:
        out = torch.empty((N, D) if cls_only else (N, T, D), dtype=dt, device=x.device)
    _dev(out, "out", dt)
    fn = lib.vit_encoder_cls if cls_only else lib.vit_encoder
    with torch.cuda.device(x.device):
        rc = fn(_ptr(x), arr, len(layers), _ptr(lnf_g), _ptr(lnf_b), 1 if final_ln else 0,
                N, T, D, F, int(H), float(eps), _dtype_code(dt), _ptr(out), _stream(stream))
    _check(rc, "vit_encoder_cls" if cls_only else "vit_encoder")
    return out


def vit_block_cls(x, layer, H, eps, out=None, stream=None):
    """out (N, D) = row 0 of each sequence's block output, computed for that row alone
    (its query against all T keys and values); layer: a dict keyed by LAYER_FIELDS."""
    lib = load_library()
    dt = x.dtype
    _dev(x, "x", dt)
    arr = _layer_array([layer], dt)
    N, T, D = x.shape
    F = layer["w_mlp1"].shape[1]
    if out is None:
        out = torch.empty((N, D), dtype=dt, device=x.device)
    _dev(out, "out", dt)
    with torch.cuda.device(x.device):
        rc = lib.vit_block_cls(_ptr(x), arr, N, T, D, F, int(H), float(eps), _dtype_code(dt), _ptr(out),
                               _stream(stream))
    _check(rc, "vit_block_cls")
    return out


def vit_patch_embed(images, P, w, b=None, cls=None, pos=None, order=0, out=None, stream=None):
    """tokens (N, T, D) from images (N, C, Hi, Wi): P x P patches flattened in `order`
    (0: channel, row, column; 1: row, column, channel) @ w (+ b), the cls row prepended and
    pos (T, D) added when given."""
    lib = load_library()
    dt = images.dtype
    for name, t in (("images", images), ("w", w), ("b", b), ("cls", cls), ("pos", pos)):
        _dev(t, name, dt)
    N, C, Hi, Wi = images.shape
    D = w.shape[1]
    T = (Hi // P) * (Wi // P) + (1 if cls is not None else 0)
    if out is None:
        out = torch.empty((N, T, D), dtype=dt, device=images.device)
    _dev(out, "out", dt)
    with torch.cuda.device(images.device):
        rc = lib.vit_patch_embed(_ptr(images), N, C, Hi, Wi, int(P), int(order), _ptr(w), _ptr(b), _ptr(cls),
                                 _ptr(pos), D, _dtype_code(dt), _ptr(out), _stream(stream))
    _check(rc, "vit_patch_embed")
    return out


def vit_block_host(x, w_q, w_k, w_v, w_o, w_mlp1, w_mlp2, H, eps, ln1_g=None, ln1_b=None,
                   ln2_g=None, ln2_b=None, b1=None, b2=None, out=None, stream=None, device=0):
    """The block on HOST tensors (pinned for full copy speed): the library copies the
    inputs in, runs, copies `out` back and synchronises the stream."""
    lib = load_library()
    dt = x.dtype
    ts = [x, w_q, w_k, w_v, w_o, w_mlp1, w_mlp2, ln1_g, ln1_b, ln2_g, ln2_b, b1, b2]
    for t in ts:
        if t is not None and (t.is_cuda or not t.is_contiguous() or t.dtype != dt):
            raise ValueError("vit_block_host takes contiguous host tensors of one dtype")
    N, T, D = x.shape
    F = w_mlp1.shape[1]
    if out is None:
        out = torch.empty_like(x)
    with torch.cuda.device(device):
        rc = lib.vit_block_host(*[_ptr(t) for t in ts], N, T, D, F, int(H), float(eps),
                                _dtype_code(dt), _ptr(out), _stream(stream))
    _check(rc, "vit_block_host")
    return out


class VitWeights:
    """One block's weights prepared on a device (vit_weights_create): copied once, with
    the concatenated Q/K/V bias and, when folding, the LayerNorm fold's column terms.

    layer: dict keyed by LAYER_FIELDS (the six weights required), all CUDA tensors on
    one device, or all host tensors (then copied to `device`). fold: 1 / 0 / -1 (the
    library's choice). The handle is freed by close() or when the object is collected."""

    def __init__(self, layer, H, fold=-1, device=None, stream=None):
        lib = load_library()
        w_q = layer["w_q"]
        dt = w_q.dtype
        on_host = not w_q.is_cuda
        arr = (VitLayer * 1)()
        for name in LAYER_FIELDS:
            t = layer.get(name)
            if t is None:
                continue
            if t.is_cuda == on_host or not t.is_contiguous() or t.dtype != dt:
                raise ValueError("layer %s: all tensors contiguous, of one dtype, all on the host "
                                 "or all on one device" % name)
            setattr(arr[0], name, t.data_ptr())
        D, F = layer["w_mlp1"].shape
        if device is None:
            device = 0 if on_host else w_q.device.index
        self._lib = lib
        self._h = _vp()
        self._layer = layer   # keeps the arrays alive until the copies are made
        with torch.cuda.device(device):
            rc = lib.vit_weights_create(arr, 1 if on_host else 0, D, F, int(H), _dtype_code(dt), int(fold),
                                        ctypes.byref(self._h), _stream(stream))
        self._layer = None
        _check(rc, "vit_weights_create")
        d, f, h = _i64(), _i64(), _i64()
        code, fo, dev = _int(), _int(), _int()
        _check(lib.vit_weights_info(self._h, ctypes.byref(d), ctypes.byref(f), ctypes.byref(h),
                                    ctypes.byref(code), ctypes.byref(fo), ctypes.byref(dev)), "vit_weights_info")
        self.D, self.F, self.H, self.fold, self.device = d.value, f.value, h.value, bool(fo.value), dev.value
        self.dtype = dt

    @property
    def handle(self):
        if not self._h:
            raise ValueError("the prepared weights have been freed")
        return self._h

    def close(self):
        if getattr(self, "_h", None):
            h, self._h = self._h, _vp()
            _check(self._lib.vit_weights_destroy(h), "vit_weights_destroy")

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def vit_block_w(x, weights, eps, out=None, stream=None):
    """The block on prepared weights (vit_block_w): x (N, T, D) on the weights' device."""
    lib = load_library()
    _dev(x, "x", weights.dtype)
    N, T, D = x.shape
    if D != weights.D:
        raise ValueError("x has width %d, the weights %d" % (D, weights.D))
    if out is None:
        out = torch.empty_like(x)
    _dev(out, "out", weights.dtype)
    with torch.cuda.device(weights.device):
        rc = lib.vit_block_w(_ptr(x), weights.handle, N, T, float(eps), _ptr(out), _stream(stream))
    _check(rc, "vit_block_w")
    return out


def vit_block_w_host(x, weights, eps, out=None, stream=None):
    """vit_block_w on HOST x and out (pinned for full copy speed); only x and out cross
    the link, and the stream is synchronised before returning."""
    lib = load_library()
    if x.is_cuda or not x.is_contiguous() or x.dtype != weights.dtype:
        raise ValueError("vit_block_w_host takes a contiguous host x of the weights' dtype")
    N, T, D = x.shape
    if D != weights.D:
        raise ValueError("x has width %d, the weights %d" % (D, weights.D))
    if out is None:
        out = torch.empty_like(x)
    with torch.cuda.device(weights.device):
        rc = lib.vit_block_w_host(_ptr(x), weights.handle, N, T, float(eps), _ptr(out), _stream(stream))
    _check(rc, "vit_block_w_host")
    return out


def vit_block_w_host_async(x, weights, eps, out, stream):
    """vit_block_w_host without waiting: enqueues the copy of host x in, the block and the
    copy back into host `out` after the work on `stream`, and returns. `out` holds the
    result once `stream` has reached that point; x, out and the handle must outlive the
    work. Successive calls on different streams overlap their copies with each other's
    blocks (pinned x and out)."""
    lib = load_library()
    if x.is_cuda or not x.is_contiguous() or x.dtype != weights.dtype:
        raise ValueError("vit_block_w_host_async takes a contiguous host x of the weights' dtype")
    if out is None or out.is_cuda or not out.is_contiguous() or out.shape != x.shape or out.dtype != x.dtype:
        raise ValueError("vit_block_w_host_async takes a contiguous host out shaped like x")
    if stream is None:
        raise ValueError("vit_block_w_host_async needs an explicit stream to order its work")
    N, T, D = x.shape
    if D != weights.D:
        raise ValueError("x has width %d, the weights %d" % (D, weights.D))
    with torch.cuda.device(weights.device):
        rc = lib.vit_block_w_host_async(_ptr(x), weights.handle, N, T, float(eps), _ptr(out), _stream(stream))
    _check(rc, "vit_block_w_host_async")
    return out


def layernorm(x, eps, gamma=None, beta=None, out_dtype=None, out=None, stream=None):
    lib = load_library()
    _dev(x, "x")
    od = out_dtype or x.dtype
    D = x.shape[-1]
    rows = x.numel() // D
    if out is None:
        out = torch.empty(x.shape, dtype=od, device=x.device)
    _dev(out, "out", od)
    _dev(gamma, "gamma", od)
    _dev(beta, "beta", od)
    with torch.cuda.device(x.device):
        rc = lib.vit_layernorm(_ptr(x), rows, D, float(eps), _ptr(gamma), _ptr(beta),
                               _dtype_code(x.dtype), _ptr(out), _dtype_code(od), _stream(stream))
    _check(rc, "vit_layernorm")
    return out


def linear(a, w, bias=None, residual=None, epilogue=EPI_STORE, out_dtype=None, out=None,
           stream=None):
    lib = load_library()
    _dev(a, "a")
    _dev(w, "w", a.dtype)
    _dev(bias, "bias", a.dtype)
    _dev(residual, "residual")
    K, N = w.shape
    M = a.numel() // K
    od = out_dtype or a.dtype
    if out is None:
        out = torch.empty(a.shape[:-1] + (N,), dtype=od, device=a.device)
    _dev(out, "out", od)
    rdt = _dtype_code(residual.dtype) if residual is not None else 0
    with torch.cuda.device(a.device):
        rc = lib.vit_linear(_ptr(a), _ptr(w), _ptr(bias), _ptr(residual), M, K, N, int(epilogue),
                            _dtype_code(a.dtype), rdt, _ptr(out), _dtype_code(od), _stream(stream))
    _check(rc, "vit_linear")
    return out


def attention(qkv, H, out=None, stream=None):
    lib = load_library()
    _dev(qkv, "qkv")
    N, T, D3 = qkv.shape
    D = D3 // 3
    if out is None:
        out = torch.empty((N, T, D), dtype=qkv.dtype, device=qkv.device)
    _dev(out, "out", qkv.dtype)
    with torch.cuda.device(qkv.device):
        rc = lib.vit_attention(_ptr(qkv), N, T, D, int(H), _dtype_code(qkv.dtype), _ptr(out),
                               _stream(stream))
    _check(rc, "vit_attention")
    return out


def device_error() -> int:
    """Synchronise, then read and clear the device error word (0 = none)."""
    w = ctypes.c_uint32(0)
    rc = load_library().vit_device_error(ctypes.byref(w))
    if rc not in (0, -4):
        raise VitError(rc, "vit_device_error")
    return int(w.value)


def selftest_wait(abort_first: bool = False, stream=None):
    """Enqueue the bounded-wait self test (a wait that must give up); read the outcome
    with device_error(): bit 1 << 5 is set when the wait ended by its limit or abort."""
    _check(load_library().vit_selftest_wait(1 if abort_first else 0, _stream(stream)),
           "vit_selftest_wait")


def launch_count() -> int:
    return int(load_library().vit_launch_count())


def timing_enable(on: bool):
    load_library().vit_timing_enable(1 if on else 0)


def timing_reset():
    load_library().vit_timing_reset()


def timing_collect() -> dict:
    """Synchronise pending timing records; returns {kernel: (total_ms, launches)}."""
    lib = load_library()
    _check(lib.vit_timing_collect(), "vit_timing_collect")
    out = {}
    for k in range(lib.vit_timing_kernels()):
        ms, n, nm = ctypes.c_double(), ctypes.c_int64(), ctypes.c_char_p()
        lib.vit_timing_read(k, ctypes.byref(ms), ctypes.byref(n), ctypes.byref(nm))
        out[nm.value.decode()] = (ms.value, n.value)
    return out
