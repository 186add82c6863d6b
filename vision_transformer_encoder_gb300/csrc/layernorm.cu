// layernorm.cu -- per-token LayerNorm over the D features.
// "ViT Encoder Block" (crackedaicode), "Normalize before each stage":
//   LN(x) = (x - mean) / sqrt(variance + eps), population variance (divide by D);
// optional gain/bias per feature: "ViT Encoder Block" (ai-engineer-exhaustive),
// Key Equations, Step 1.
//
// Fast kernel (bf16 or fp32 input, bf16 output, D % 8 == 0, D <= 2048): one warp per
// row; the row is read once with 16-byte loads into registers; mean and the centred
// sum of squares (two passes over the registers, never E[x^2] - mean^2, so a constant
// row normalises to exactly 0) are warp-shuffle reductions in fp32. HBM-bound:
// D * (in + out) bytes per row.
// Generic kernel: any supported type pair, one warp per row, strided loops.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace vit {
namespace {

constexpr int LN_THREADS = 256;  // 8 rows per CTA

template <typename TIn> struct VecIO;
template <> struct VecIO<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void load(const __nv_bfloat16* p, float (&v)[N]) {
        uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
        float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y), c = unpack_bf16x2(u.z),
               d = unpack_bf16x2(u.w);
        v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
        v[4] = c.x; v[5] = c.y; v[6] = d.x; v[7] = d.y;
    }
};
template <> struct VecIO<float> {
    static constexpr int N = 4;
    __device__ static void load(const float* p, float (&v)[N]) {
        float4 u = __ldg(reinterpret_cast<const float4*>(p));
        v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
    }
};

template <int N> __device__ __forceinline__ void store_bf16(__nv_bfloat16* p, const float (&v)[N]);
template <> __device__ __forceinline__ void store_bf16<8>(__nv_bfloat16* p, const float (&v)[8]) {
    uint4 u;
    u.x = pack_bf16x2(v[0], v[1]);
    u.y = pack_bf16x2(v[2], v[3]);
    u.z = pack_bf16x2(v[4], v[5]);
    u.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4*>(p) = u;
}
template <> __device__ __forceinline__ void store_bf16<4>(__nv_bfloat16* p, const float (&v)[4]) {
    uint2 u;
    u.x = pack_bf16x2(v[0], v[1]);
    u.y = pack_bf16x2(v[2], v[3]);
    *reinterpret_cast<uint2*>(p) = u;
}

// V consecutive bf16 gains or biases as floats, in one 16-byte (V = 8) or 8-byte (V = 4)
// load; the vectors start at multiples of V elements.
template <int V> __device__ __forceinline__ void load_param_bf16(const __nv_bfloat16* p, float (&o)[V]);
template <> __device__ __forceinline__ void load_param_bf16<8>(const __nv_bfloat16* p, float (&o)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y), c = unpack_bf16x2(u.z), d = unpack_bf16x2(u.w);
    o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
    o[4] = c.x; o[5] = c.y; o[6] = d.x; o[7] = d.y;
}
template <> __device__ __forceinline__ void load_param_bf16<4>(const __nv_bfloat16* p, float (&o)[4]) {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
    const float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y);
    o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
}

template <typename TIn, int MAXV>
__global__ void __launch_bounds__(LN_THREADS)
ln_fast_kernel(const TIn* __restrict__ x, __nv_bfloat16* __restrict__ out,
               const __nv_bfloat16* __restrict__ gamma, const __nv_bfloat16* __restrict__ beta,
               int64_t rows, int D, float inv_d, float eps) {
    constexpr int V = VecIO<TIn>::N;
    griddep_wait();                 // x is the previous kernel's output
    griddep_launch_dependents();
    const int64_t row = (int64_t)blockIdx.x * (LN_THREADS / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int nvec = D / V;
    const TIn* xr = x + row * D;
    float v[MAXV][V];
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
        const int idx = lane + 32 * j;
        if (idx < nvec) {
            VecIO<TIn>::load(xr + idx * V, v[j]);
#pragma unroll
            for (int e = 0; e < V; ++e) sum += v[j][e];
        }
    }
    // the mean by a correctly rounded division, so that a constant row whose sum is
    // exact gets its own value back and normalises to exactly 0; the variance, 0 for such
    // a row either way, by a multiply with 1 / D from the host
    const float mean = warp_sum(sum) / (float)D;
    float sq = 0.f;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
        const int idx = lane + 32 * j;
        if (idx < nvec) {
#pragma unroll
            for (int e = 0; e < V; ++e) {
                v[j][e] -= mean;   // the centred values, kept for the output
                sq = fmaf(v[j][e], v[j][e], sq);
            }
        }
    }
    const float var = warp_sum(sq) * inv_d;
    const float rstd = rsqrtf(var + eps);
    __nv_bfloat16* orow = out + row * D;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
        const int idx = lane + 32 * j;
        if (idx < nvec) {
            float o[V];
#pragma unroll
            for (int e = 0; e < V; ++e) o[e] = v[j][e] * rstd;
            if (gamma) {
                float gv[V];
                load_param_bf16<V>(gamma + idx * V, gv);
#pragma unroll
                for (int e = 0; e < V; ++e) o[e] *= gv[e];
            }
            if (beta) {
                float bv[V];
                load_param_bf16<V>(beta + idx * V, bv);
#pragma unroll
                for (int e = 0; e < V; ++e) o[e] += bv[e];
            }
            store_bf16<V>(orow + idx * V, o);
        }
    }
}

template <typename A>
__device__ __forceinline__ A ld_param(const void* p, int dt, int64_t i) {
    if (dt == DT_F32) return (A) static_cast<const float*>(p)[i];
    if (dt == DT_BF16) return (A)__bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
    return (A) static_cast<const double*>(p)[i];
}

// Accumulation type: double for f64 input, float otherwise. gamma/beta of type gb_dt.
template <typename TIn, typename TOut>
__global__ void __launch_bounds__(LN_THREADS)
ln_generic_kernel(const TIn* __restrict__ x, TOut* __restrict__ out, const void* __restrict__ gamma,
                  const void* __restrict__ beta, int gb_dt, int64_t rows, int64_t D, double eps,
                  float* __restrict__ lo) {
    using A = typename std::conditional<std::is_same<TIn, double>::value, double, float>::type;
    const int64_t row = (int64_t)blockIdx.x * (LN_THREADS / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const TIn* xr = x + row * D;
    A sum = 0;
    for (int64_t j = lane; j < D; j += 32) sum += to_acc<A>(xr[j]);
    const A mean = warp_sum(sum) / (A)D;
    A sq = 0;
    for (int64_t j = lane; j < D; j += 32) {
        const A d = to_acc<A>(xr[j]) - mean;
        sq += d * d;
    }
    const A var = warp_sum(sq) / (A)D;
    const A denom = sqrt(var + (A)eps);
    TOut* orow = out + row * D;
    for (int64_t j = lane; j < D; j += 32) {
        A o = (to_acc<A>(xr[j]) - mean) / denom;
        if (gamma) o = ld_param<A>(gamma, gb_dt, j) * o;
        if (beta) o = o + ld_param<A>(beta, gb_dt, j);
        const TOut v = from_acc<TOut>(o);
        orow[j] = v;
        if constexpr (std::is_same<TOut, float>::value)
            if (lo) lo[row * D + j] = tf32_low_part(v);
    }
}

template <typename TIn, typename TOut>
cudaError_t launch_generic(const void* x, void* out, const void* g, const void* b, int gb_dt,
                           int64_t rows, int64_t D, double eps, cudaStream_t s, float* lo = nullptr) {
    const int64_t blocks = (rows + LN_THREADS / 32 - 1) / (LN_THREADS / 32);
    ln_generic_kernel<TIn, TOut><<<(unsigned)blocks, LN_THREADS, 0, s>>>(
        static_cast<const TIn*>(x), static_cast<TOut*>(out), g, b, gb_dt, rows, D, eps, lo);
    return cudaGetLastError();
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

template <typename TIn, int MAXV>
cudaError_t launch_fast_v(const void* x, void* out, const void* g, const void* b, int64_t rows,
                          int64_t D, double eps, cudaStream_t s) {
    const int64_t blocks = (rows + LN_THREADS / 32 - 1) / (LN_THREADS / 32);
    return launch_dependent(ln_fast_kernel<TIn, MAXV>, dim3((unsigned)blocks), dim3(LN_THREADS), 0, s,
                            static_cast<const TIn*>(x), static_cast<__nv_bfloat16*>(out),
                            static_cast<const __nv_bfloat16*>(g), static_cast<const __nv_bfloat16*>(b), rows,
                            (int)D, (float)(1.0 / (double)D), (float)eps);
}

template <typename TIn>
cudaError_t launch_fast(const void* x, void* out, const void* g, const void* b, int64_t rows,
                        int64_t D, double eps, int per_lane, cudaStream_t s) {
    switch (per_lane) {
        case 1: return launch_fast_v<TIn, 1>(x, out, g, b, rows, D, eps, s);
        case 2: return launch_fast_v<TIn, 2>(x, out, g, b, rows, D, eps, s);
        case 3: return launch_fast_v<TIn, 3>(x, out, g, b, rows, D, eps, s);
        case 4: return launch_fast_v<TIn, 4>(x, out, g, b, rows, D, eps, s);
        case 5: return launch_fast_v<TIn, 5>(x, out, g, b, rows, D, eps, s);
        case 6: return launch_fast_v<TIn, 6>(x, out, g, b, rows, D, eps, s);
        case 7:
        case 8: return launch_fast_v<TIn, 8>(x, out, g, b, rows, D, eps, s);
        case 9:
        case 10: return launch_fast_v<TIn, 10>(x, out, g, b, rows, D, eps, s);
        case 11:
        case 12: return launch_fast_v<TIn, 12>(x, out, g, b, rows, D, eps, s);
        default: return launch_fast_v<TIn, 16>(x, out, g, b, rows, D, eps, s);
    }
}

}  // namespace

cudaError_t launch_layernorm_f32_lo(const float* x, float* out, float* lo, const void* gamma, const void* beta,
                                    int gb_dt, int64_t rows, int64_t D, double eps, cudaStream_t s) {
    if (rows <= 0 || D <= 0) return cudaSuccess;
    if ((rows + LN_THREADS / 32 - 1) / (LN_THREADS / 32) > 0x7fffffff) return cudaErrorInvalidValue;
    return launch_generic<float, float>(x, out, gamma, beta, gb_dt, rows, D, eps, s, lo);
}

cudaError_t launch_layernorm(const void* x, int in_dt, void* out, int out_dt, const void* gamma,
                             const void* beta, int gb_dt, int64_t rows, int64_t D, double eps,
                             cudaStream_t s) {
    if (rows <= 0 || D <= 0) return cudaSuccess;
    const int64_t blocks = (rows + LN_THREADS / 32 - 1) / (LN_THREADS / 32);
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    const bool vec_ok = D % 8 == 0 && D <= 2048 && aligned16(x) && aligned16(out);
    // gains and biases: bf16, read in 16-byte vectors
    const bool gb_bf16 = ((!gamma && !beta) || gb_dt == DT_BF16) && (!gamma || aligned16(gamma)) &&
                         (!beta || aligned16(beta));
    if (out_dt == DT_BF16 && vec_ok && gb_bf16 && (in_dt == DT_BF16 || in_dt == DT_F32)) {
        // registers hold ceil(D / (32 lanes * vector width)) vectors per lane
        const int per_lane = (int)((D / (in_dt == DT_BF16 ? 8 : 4) + 31) / 32);
        return in_dt == DT_BF16 ? launch_fast<__nv_bfloat16>(x, out, gamma, beta, rows, D, eps, per_lane, s)
                                : launch_fast<float>(x, out, gamma, beta, rows, D, eps, per_lane, s);
    }
    if (in_dt == DT_BF16 && out_dt == DT_BF16)
        return launch_generic<__nv_bfloat16, __nv_bfloat16>(x, out, gamma, beta, gb_dt, rows, D, eps, s);
    if (in_dt == DT_F32 && out_dt == DT_BF16)
        return launch_generic<float, __nv_bfloat16>(x, out, gamma, beta, gb_dt, rows, D, eps, s);
    if (in_dt == DT_F32 && out_dt == DT_F32)
        return launch_generic<float, float>(x, out, gamma, beta, gb_dt, rows, D, eps, s);
    if (in_dt == DT_F64 && out_dt == DT_F64)
        return launch_generic<double, double>(x, out, gamma, beta, gb_dt, rows, D, eps, s);
    if (in_dt == DT_BF16 && out_dt == DT_F32)
        return launch_generic<__nv_bfloat16, float>(x, out, gamma, beta, gb_dt, rows, D, eps, s);
    return cudaErrorInvalidValue;
}

}  // namespace vit
