"""Host-side arithmetic of bench.py (no GPU): the FLOP count the metric divides by, the
per-kernel algorithmic work behind the roofline line, and the derived peaks of the fp32
path."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from vision_transformer_encoder_gb300.inputs import CONFIGS  # noqa: E402


def test_flops_per_step_is_the_block_formula():
    # 2 N T (4 D^2 + 2 D F) for the four products, 4 N T^2 D for Q K^T and P V
    c = CONFIGS["vit_b16"]
    N, T, D, F = c["N"], c["T"], c["D"], c["F"]
    assert bench.flops_per_step(c) == 2 * N * T * (4 * D * D + 2 * D * F) + 4 * N * T * T * D
    assert bench.flops_per_step(c) == pytest.approx(7.444e11, rel=1e-3)


@pytest.mark.parametrize("f32", [False, True])
def test_kernel_work_adds_up_to_the_step(f32):
    c = CONFIGS["vit_b16"]
    N, T, D, F = c["N"], c["T"], c["D"], c["F"]
    M = N * T
    w = bench.kernel_work(c, f32)
    block_gemms = ("qkv_gemm", "wo_gemm_residual", "w1_gemm_gelu", "w2_gemm_residual")
    gemm = sum(w[k][1] for k in block_gemms)
    assert gemm == 2 * M * (4 * D * D + 2 * D * F)
    assert w["attention"][1] == 4 * N * T * T * D
    assert gemm + w["attention"][1] == bench.flops_per_step(c)
    # bf16: read x, write xn; fp32: read x, write xn and its low part (A_lo of the next product)
    assert w["ln1"] == ("hbm", M * D * ((4 + 4 + 4) if f32 else (2 + 2)), "bytes")
    assert w["ln2"][1] == M * D * ((4 + 4 + 4) if f32 else (4 + 2))   # read fp32 y
    assert w["attention"][0] == "tensor"   # head width 64, T <= 224: tensor cores on both paths
    for k in block_gemms:
        assert w[k][0] == "tensor"


def test_fp32_attention_bound_off_the_tensor_core_shapes():
    # the fp32 path's attention runs on the CUDA cores at head width 80 or above 224 tokens
    assert bench.kernel_work(CONFIGS["vit_h14_448"], True)["attention"][0] == "alu"
    assert bench.kernel_work(CONFIGS["vit_l16_384"], True)["attention"][0] == "alu"
    assert bench.kernel_work(CONFIGS["vit_ti16"], True)["attention"][0] == "tensor"


def test_fp32_path_peaks():
    # three TF32 products per fp32 product, at the nominal TF32 / BF16 dense ratio
    assert bench.TF32X3_OF_BF16 == pytest.approx(1.1 / 2.25 / 3)
    # 152 SMs x 128 FP32 lanes x 2 flop (FMA) at 2.07 GHz
    assert bench.FP32_ALU_TFLOPS == pytest.approx(80.55, abs=0.01)


def test_workload_names_carry_the_sizes():
    for name, c in CONFIGS.items():
        s = bench.workload_name(name, c)
        for key in ("N", "T", "D", "H", "F"):
            assert "%s=%d" % (key, c[key]) in s, (name, s)
