"""The C-ABI library without a GPU: it loads, exports every function the header
declares, and the host-side argument checks answer before any CUDA call."""
import ctypes
import os
import re

import pytest

from vision_transformer_encoder_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vit_block.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vit_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_binding_surface():
    assert declared_functions() == sorted(api.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_exports_are_exactly_the_header(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", api.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = sorted(set(re.findall(r" T (vit_[a-z_0-9]+)$", out, flags=re.M)))
    assert exported == declared_functions()


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        s = api.status_string(code)
        assert s and s != "unknown status"
    assert api.status_string(-99) == "unknown status"


def _fake(i):
    # distinct, well-separated fake device addresses; never dereferenced because
    # validation fails first
    return ctypes.c_void_p(0x100000000 * (i + 1))


def _call_block(lib, N=2, T=5, D=8, F=16, H=2, dtype=1, x=None, out=None, null_w=False):
    ws = [None if null_w else _fake(i + 1) for i in range(6)]
    return lib.vit_block(x if x is not None else _fake(0), *ws, N, T, D, F, H, 1e-5, dtype,
                         out if out is not None else _fake(10), None)


def test_invalid_sizes_are_rejected_on_the_host(lib):
    assert _call_block(lib, D=8, H=3) == -1          # H does not divide D
    assert _call_block(lib, N=0) == -1
    assert _call_block(lib, T=-1) == -1
    assert _call_block(lib, F=0) == -1
    assert _call_block(lib, H=0) == -1
    assert _call_block(lib, null_w=True) == -1


def test_unknown_dtype_rejected(lib):
    assert _call_block(lib, dtype=7) == -2


def test_out_aliasing_an_input_is_rejected(lib):
    x = _fake(0)
    assert _call_block(lib, x=x, out=x) == -1
    # out overlapping the tail of x
    assert _call_block(lib, x=x, out=ctypes.c_void_p(x.value + 16)) == -1


def test_step_entry_points_validate(lib):
    assert lib.vit_layernorm(None, 4, 8, 1e-5, None, None, 1, _fake(1), 1, None) == -1
    assert lib.vit_layernorm(_fake(0), 4, 8, 1e-5, None, None, 2, _fake(1), 1, None) == -2
    assert lib.vit_linear(_fake(0), _fake(1), None, None, 4, 8, 8, 2, 1, 1, _fake(2), 1, None) == -1
    assert lib.vit_linear(_fake(0), _fake(1), None, None, 4, 8, 8, 0, 0, 0, _fake(2), 1, None) == -2
    assert lib.vit_attention(_fake(0), 1, 4, 8, 3, 1, _fake(1), None) == -1


def test_timing_interface_without_gpu(lib):
    assert lib.vit_timing_kernels() == 21
    ms, n, nm = ctypes.c_double(), ctypes.c_int64(), ctypes.c_char_p()
    assert lib.vit_timing_read(0, ctypes.byref(ms), ctypes.byref(n), ctypes.byref(nm)) == 0
    assert nm.value == b"ln1"
    assert lib.vit_timing_read(99, None, None, None) == -1


def test_encoder_argument_checks(lib):
    layer = api.VitLayer(*[_fake(i + 1).value for i in range(6)] + [None] * 10)
    arr = (api.VitLayer * 1)(layer)
    assert lib.vit_encoder(_fake(0), arr, 0, None, None, 1, 2, 5, 8, 16, 2, 1e-5, 1, _fake(10), None) == -1
    assert lib.vit_encoder(_fake(0), None, 1, None, None, 1, 2, 5, 8, 16, 2, 1e-5, 1, _fake(10), None) == -1
    assert lib.vit_encoder(_fake(0), arr, 1, None, None, 1, 2, 5, 8, 16, 3, 1e-5, 1, _fake(10), None) == -1
    assert lib.vit_encoder(_fake(0), arr, 1, None, None, 1, 2, 5, 8, 16, 2, 1e-5, 7, _fake(10), None) == -2
    bad = (api.VitLayer * 1)(api.VitLayer(*[_fake(i + 1).value for i in range(5)] + [None] * 11))
    assert lib.vit_encoder(_fake(0), bad, 1, None, None, 1, 2, 5, 8, 16, 2, 1e-5, 1, _fake(10), None) == -1
    # out overlapping a projection bias
    lay2 = api.VitLayer(*[_fake(i + 1).value for i in range(6)] + [None] * 6 + [_fake(10).value + 8] + [None] * 3)
    arr2 = (api.VitLayer * 1)(lay2)
    assert lib.vit_encoder(_fake(0), arr2, 1, None, None, 1, 2, 5, 8, 16, 2, 1e-5, 1, _fake(10), None) == -1


def test_cls_argument_checks(lib):
    layer = api.VitLayer(*[_fake(i + 1).value for i in range(6)] + [None] * 10)
    arr = (api.VitLayer * 1)(layer)
    assert lib.vit_block_cls(_fake(0), None, 2, 5, 8, 16, 2, 1e-5, 1, _fake(10), None) == -1
    assert lib.vit_block_cls(_fake(0), arr, 2, 5, 8, 16, 3, 1e-5, 1, _fake(10), None) == -1   # H does not divide D
    assert lib.vit_block_cls(_fake(0), arr, 2, 5, 8, 16, 2, 1e-5, 9, _fake(10), None) == -2
    assert lib.vit_block_cls(None, arr, 2, 5, 8, 16, 2, 1e-5, 1, _fake(10), None) == -1
    # the (N, D) output overlapping x; (N, D) bf16 is 32 bytes, so an output 64 bytes before
    # x does not overlap it, but one 16 bytes before does
    assert lib.vit_block_cls(_fake(0), arr, 2, 5, 8, 16, 2, 1e-5, 1, ctypes.c_void_p(_fake(0).value - 16),
                             None) == -1
    assert lib.vit_encoder_cls(_fake(0), arr, 0, None, None, 1, 2, 5, 8, 16, 2, 1e-5, 1, _fake(10), None) == -1
    assert lib.vit_encoder_cls(_fake(0), arr, 1, None, None, 1, 0, 5, 8, 16, 2, 1e-5, 1, _fake(10), None) == -1
    # out overlapping the final LayerNorm's gain
    assert lib.vit_encoder_cls(_fake(0), arr, 1, _fake(10), None, 1, 2, 5, 8, 16, 2, 1e-5, 1, _fake(10),
                               None) == -1


def test_patch_embed_argument_checks(lib):
    args = dict(N=2, C=3, Hi=32, Wi=32, P=16, order=0, D=8)
    def call(**kw):
        a = dict(args, **kw)
        return lib.vit_patch_embed(_fake(0), a["N"], a["C"], a["Hi"], a["Wi"], a["P"], a["order"], _fake(1),
                                   None, None, None, a["D"], kw.get("dtype", 1), _fake(10), None)
    assert call(Hi=30) == -1            # not a multiple of P
    assert call(order=2) == -1
    assert call(P=0) == -1
    assert call(dtype=5) == -2
    assert lib.vit_patch_embed(None, 2, 3, 32, 32, 16, 0, _fake(1), None, None, None, 8, 1, _fake(10), None) == -1
    # tokens overlapping the images
    assert lib.vit_patch_embed(_fake(0), 2, 3, 32, 32, 16, 0, _fake(1), None, None, None, 8, 1,
                               ctypes.c_void_p(_fake(0).value + 64), None) == -1


def test_selftest_without_a_device_reports_a_cuda_error(lib):
    # no GPU here: the self test cannot launch and says so with a status, not a crash
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present; tests/test_gpu_failure.py covers it")
    assert lib.vit_selftest_wait(0, None) == -3
    assert lib.vit_selftest_wait(1, None) == -3


def test_prepared_weights_argument_checks(lib):
    layer = api.VitLayer(*[_fake(i + 1).value for i in range(6)] + [None] * 10)
    arr = (api.VitLayer * 1)(layer)
    h = ctypes.c_void_p()
    create = lib.vit_weights_create
    assert create(None, 0, 8, 16, 2, 1, -1, ctypes.byref(h), None) == -1          # no layer
    assert create(arr, 0, 8, 16, 2, 1, -1, None, None) == -1                      # no out
    assert create(arr, 0, 8, 16, 3, 1, -1, ctypes.byref(h), None) == -1          # H does not divide D
    assert create(arr, 0, 0, 16, 2, 1, -1, ctypes.byref(h), None) == -1
    assert create(arr, 0, 8, 16, 2, 7, -1, ctypes.byref(h), None) == -2          # dtype
    assert create(arr, 2, 8, 16, 2, 1, -1, ctypes.byref(h), None) == -1          # from_host
    assert create(arr, 0, 8, 16, 2, 1, 2, ctypes.byref(h), None) == -1           # fold
    bad = (api.VitLayer * 1)(api.VitLayer(*[_fake(i + 1).value for i in range(5)] + [None] * 11))
    assert create(bad, 0, 8, 16, 2, 1, -1, ctypes.byref(h), None) == -1          # null w_mlp2
    assert not h.value                                                            # untouched
    # a null handle: every call that takes one rejects it before touching the GPU
    assert lib.vit_block_w(_fake(0), None, 2, 5, 1e-5, _fake(10), None) == -1
    assert lib.vit_block_w_host(_fake(0), None, 2, 5, 1e-5, _fake(10), None) == -1
    assert lib.vit_block_w_host_async(_fake(0), None, 2, 5, 1e-5, _fake(10), None) == -1
    assert lib.vit_weights_info(None, None, None, None, None, None, None) == -1
    assert lib.vit_weights_destroy(None) == 0


def test_async_host_binding_checks_its_arguments(lib):
    # the binding's own checks run before any call into the library (no GPU needed)
    import torch

    class _Handle:   # stands in for a VitWeights: only the fields the checks read
        dtype, D, device, handle = torch.bfloat16, 8, 0, None

    x = torch.zeros(2, 3, 8, dtype=torch.bfloat16)
    out = torch.empty_like(x)
    with pytest.raises(ValueError):
        api.vit_block_w_host_async(x, _Handle(), 1e-6, None, 0)           # no output array
    with pytest.raises(ValueError):
        api.vit_block_w_host_async(x, _Handle(), 1e-6, out, None)         # no stream to order on
    with pytest.raises(ValueError):
        api.vit_block_w_host_async(x, _Handle(), 1e-6, out[:1], 0)        # out not shaped like x
    with pytest.raises(ValueError):
        api.vit_block_w_host_async(x.float(), _Handle(), 1e-6, out, 0)    # x not of the weights' dtype
    w = _Handle()
    w.D = 16
    with pytest.raises(ValueError):
        api.vit_block_w_host_async(x, w, 1e-6, out, 0)                    # width differs from the weights'
