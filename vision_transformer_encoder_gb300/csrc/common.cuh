// common.cuh -- small device/host helpers shared by the library's kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "vit_block.h"

namespace vit {

// Device error word bits (see vit_device_error).
enum : uint32_t {
    ERRBIT_TIMEOUT_PRODUCER = 1u << 0,
    ERRBIT_TIMEOUT_MMA = 1u << 1,
    ERRBIT_TIMEOUT_EPILOGUE = 1u << 2,
    ERRBIT_TIMEOUT_TEARDOWN = 1u << 3,
    ERRBIT_TIMEOUT_ATTENTION = 1u << 4,
    ERRBIT_SELFTEST = 1u << 5,   // vit_selftest_wait: the deliberate wait ran out
};

// One bounded device-side wait gives up after this many SM clock cycles (about two
// seconds at 2 GHz; longer at lower clocks).
constexpr long long kWaitTimeoutCycles = 4000000000ll;

// Programmatic dependent launch (PTX griddepcontrol): griddep_wait blocks until the grids
// this one depends on in its stream have completed and their memory writes are visible (a
// no-op for a plain launch); griddep_launch_dependents lets the next launch in the stream,
// if made with programmatic serialisation, schedule its CTAs from now on.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Hardware tanh approximation (MUFU), max relative error about 2^-11.
__device__ __forceinline__ float tanh_approx(float x) {
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// x - x_hi, where x_hi is x with its 13 low mantissa bits cleared (the TF32 value a
// tensor core takes from an fp32 operand): the low part of a 3xTF32 product, exact in fp32.
__device__ __forceinline__ float tf32_low_part(float x) {
    return x - __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

// Hardware base-2 exponential approximation (MUFU).
__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// tanh-approximation GELU, "ViT Encoder Block" (crackedaicode), "Feed-forward stage":
// 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3))). Fast form for bf16 outputs.
// u = z (k0 + k0 k1 z^2) and 0.5 z (1 + t) = fma(0.5 z, t, 0.5 z): five FP32 operations
// and one tanh.
__device__ __forceinline__ float gelu_tanh_fast(float z) {
    const float k0 = 0.7978845608028654f;       // sqrt(2/pi)
    const float k0k1 = 0.7978845608028654f * 0.044715f;
    const float u = z * fmaf(k0k1, z * z, k0);
    const float hz = 0.5f * z;
    return fmaf(hz, tanh_approx(u), hz);
}

// Packed fp32 pairs (f32x2 arithmetic of sm_100 and later): one instruction computes two
// lanes, each rounded exactly as the scalar instruction would, so results are bit for bit
// those of the scalar code while the epilogues issue half the arithmetic instructions.
__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long x, unsigned long long y) {
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(y));
    return r;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long x, unsigned long long y) {
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(y));
    return r;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
// a += c, b += d
__device__ __forceinline__ void f2_add_to(float& a, float& b, float c, float d) {
    f2_unpack(f2_add(f2_pack(a, b), f2_pack(c, d)), a, b);
}
// gelu_tanh_fast of a and b, the same operations lane by lane
__device__ __forceinline__ void gelu_tanh_fast2(float& a, float& b) {
    const unsigned long long k0 = f2_pack(0.7978845608028654f, 0.7978845608028654f);
    const unsigned long long k0k1 = f2_pack(0.7978845608028654f * 0.044715f, 0.7978845608028654f * 0.044715f);
    const unsigned long long half = f2_pack(0.5f, 0.5f);
    const unsigned long long z = f2_pack(a, b);
    const unsigned long long u = f2_mul(z, f2_fma(k0k1, f2_mul(z, z), k0));
    const unsigned long long hz = f2_mul(half, z);
    float u0, u1;
    f2_unpack(u, u0, u1);
    f2_unpack(f2_fma(hz, f2_pack(tanh_approx(u0), tanh_approx(u1)), hz), a, b);
}

// Accurate forms (library tanh) for the fp32 / fp64 paths.
__device__ __forceinline__ float gelu_tanh_acc(float z) {
    const float k0 = 0.7978845608028654f;
    float u = k0 * (z + 0.044715f * z * z * z);
    return 0.5f * z * (1.0f + tanhf(u));
}
__device__ __forceinline__ double gelu_tanh_acc(double z) {
    const double k0 = 0.79788456080286535588;  // sqrt(2/pi)
    double u = k0 * (z + 0.044715 * z * z * z);
    return 0.5 * z * (1.0 + tanh(u));
}

// Element conversions.
template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<double>(double v) { return (float)v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

template <typename A, typename T> __device__ __forceinline__ A to_acc(T v) { return (A)to_f32(v); }
template <> __device__ __forceinline__ double to_acc<double, double>(double v) { return v; }

template <typename T> __device__ __forceinline__ T from_acc(float v);
template <> __device__ __forceinline__ float from_acc<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_acc<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}
template <> __device__ __forceinline__ double from_acc<double>(float v) { return v; }
template <typename T> __device__ __forceinline__ T from_acc(double v) { return from_acc<T>((float)v); }
template <> __device__ __forceinline__ double from_acc<double>(double v) { return v; }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t v) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&v);
    return __bfloat1622float2(h);
}

}  // namespace vit
