// attention_cls.cu -- attention of one query row per sequence: the CLS readout.
//
// Lecture transcript (nipunbatra.github.io), Page 55: when only the CLS token is read
// after the last block, that block needs the output of row 0 alone. Its query is scored
// against the keys of all T rows and mixes the value rows of all T rows: per sequence n
// and head h (columns [h dh, (h + 1) dh), dh = D / H),
//   s_u = q_h . k_h[u] / sqrt(dh) for u < T,  p = softmax(s),  o_h = sum_u p_u v_h[u].
//
// The work is one pass over the sequence's keys and values (2 T dh elements per (n, h))
// and a handful of flops per element, so the kernel is bound by memory: one CTA of 256
// threads per (sequence, head). The query row goes to shared memory in the accumulation
// type; each thread scores whole key rows (16-byte loads where the layout allows), the T
// scores stay in shared memory; block reductions give the maximum and the sum; then the
// threads split the head's columns (pairs of bf16 columns) and the keys into groups, each
// group summing p_u v_u over its keys with row-contiguous loads, and the groups' partial
// sums are added in shared memory. fp32 accumulation (base-2 exponent with log2(e) folded
// into the score scale) for bf16 and fp32; fp64 with exp for fp64.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace vit {
namespace {

constexpr int CLS_THREADS = 256;
constexpr int CLS_WARPS = CLS_THREADS / 32;

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}
template <>
__device__ __forceinline__ float to_f<float>(float v) {
    return v;
}

template <typename Acc>
__device__ __forceinline__ Acc exp_base(Acc v);
template <>
__device__ __forceinline__ float exp_base<float>(float v) {
    return exp2f(v);
}
template <>
__device__ __forceinline__ double exp_base<double>(double v) {
    return exp(v);
}

template <typename T, typename Acc>
__device__ __forceinline__ Acc ld_acc(const T* p) {
    if constexpr (sizeof(T) == sizeof(Acc))
        return *p;
    else
        return to_f(*p);
}

template <typename T>
__device__ __forceinline__ T from_acc(float v) {
    if constexpr (sizeof(T) == 2)
        return __float2bfloat16_rn(v);
    else
        return v;
}

// Dot product of the shared query (Acc) with one key row of dh elements.
template <typename T, typename Acc, bool VEC>
__device__ __forceinline__ Acc dot_row(const Acc* __restrict__ q, const T* __restrict__ k, int dh) {
    Acc d0 = 0, d1 = 0;
    if constexpr (VEC && sizeof(T) == 2) {
        // 8 bf16 per 16-byte load
        for (int c = 0; c < dh; c += 8) {
            const uint4 u = *reinterpret_cast<const uint4*>(k + c);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
                d0 = fmaf(q[c + 2 * i], f.x, d0);
                d1 = fmaf(q[c + 2 * i + 1], f.y, d1);
            }
        }
    } else if constexpr (VEC && sizeof(T) == 4) {
        for (int c = 0; c < dh; c += 4) {
            const float4 f = *reinterpret_cast<const float4*>(k + c);
            d0 = fmaf(q[c], f.x, d0);
            d1 = fmaf(q[c + 1], f.y, d1);
            d0 = fmaf(q[c + 2], f.z, d0);
            d1 = fmaf(q[c + 3], f.w, d1);
        }
    } else {
        for (int c = 0; c < dh; ++c) {
            if (c & 1)
                d1 += q[c] * ld_acc<T, Acc>(k + c);
            else
                d0 += q[c] * ld_acc<T, Acc>(k + c);
        }
    }
    return d0 + d1;
}

template <typename Acc>
__device__ __forceinline__ Acc warp_max(Acc v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmax(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
template <typename Acc>
__device__ __forceinline__ Acc warp_sum(Acc v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// q: row n at q + n ldq; keys / values: row u of sequence n at k + (n T + u) ldkv (likewise
// v); o: row n at o + n ldo. Head h reads and writes columns [h dh, (h + 1) dh).
// Shared memory (Acc): q (dh) | scores (T) | group partials (red_len) | reduction (2 warps).
template <typename T, typename Acc, bool VEC, bool PAIRS>
__global__ void __launch_bounds__(CLS_THREADS)
attention_cls_kernel(const T* __restrict__ q, int64_t ldq, const T* __restrict__ k, const T* __restrict__ v,
                     int64_t ldkv, int Tn, int H, int dh, int red_len, Acc scale, T* __restrict__ o, int64_t ldo) {
    extern __shared__ __align__(16) unsigned char cls_smem[];
    Acc* sq = reinterpret_cast<Acc*>(cls_smem);
    Acc* sc = sq + dh;
    Acc* red = sc + Tn;
    Acc* wred = red + red_len;   // CLS_WARPS values

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t n = blockIdx.x / H;
    const int h = (int)(blockIdx.x - n * H);
    const int64_t col = (int64_t)h * dh;
    const T* kseq = k + n * Tn * ldkv + col;
    const T* vseq = v + n * Tn * ldkv + col;

    for (int c = tid; c < dh; c += CLS_THREADS) sq[c] = ld_acc<T, Acc>(q + n * ldq + col + c);
    __syncthreads();

    // scores, each thread whole key rows, and the thread's maximum
    Acc mx = -INFINITY;
    for (int u = tid; u < Tn; u += CLS_THREADS) {
        const Acc s = dot_row<T, Acc, VEC>(sq, kseq + (int64_t)u * ldkv, dh) * scale;
        sc[u] = s;
        mx = fmax(mx, s);
    }
    mx = warp_max(mx);
    if (lane == 0) wred[warp] = mx;
    __syncthreads();
    mx = wred[0];
#pragma unroll
    for (int w = 1; w < CLS_WARPS; ++w) mx = fmax(mx, wred[w]);
    __syncthreads();   // every thread has read wred before it is reused

    // weights p_u = exp(s_u - max) (unnormalised) and their sum
    Acc sum = 0;
    for (int u = tid; u < Tn; u += CLS_THREADS) {
        const Acc p = exp_base<Acc>(sc[u] - mx);
        sc[u] = p;
        sum += p;
    }
    sum = warp_sum(sum);
    if (lane == 0) wred[warp] = sum;
    __syncthreads();
    Acc l = 0;
#pragma unroll
    for (int w = 0; w < CLS_WARPS; ++w) l += wred[w];

    // weighted sum of value rows: column units (pairs of bf16 columns, else single
    // columns) x key groups
    const int NU = PAIRS ? dh / 2 : dh;
    const int G = NU >= CLS_THREADS ? 1 : CLS_THREADS / NU;
    const int g = NU >= CLS_THREADS ? 0 : tid / NU;
    if (g < G) {
        const int stride = NU >= CLS_THREADS ? CLS_THREADS : NU;
        for (int unit = NU >= CLS_THREADS ? tid : tid % NU; unit < NU; unit += stride) {
            if constexpr (PAIRS) {
                float a0 = 0.f, a1 = 0.f;
                for (int u = g; u < Tn; u += G) {
                    const float p = sc[u];
                    const float2 f = __bfloat1622float2(
                        *reinterpret_cast<const __nv_bfloat162*>(vseq + (int64_t)u * ldkv + 2 * unit));
                    a0 = fmaf(p, f.x, a0);
                    a1 = fmaf(p, f.y, a1);
                }
                red[g * dh + 2 * unit] = a0;
                red[g * dh + 2 * unit + 1] = a1;
            } else {
                Acc a0 = 0;
                for (int u = g; u < Tn; u += G) a0 += sc[u] * ld_acc<T, Acc>(vseq + (int64_t)u * ldkv + unit);
                red[g * dh + unit] = a0;
            }
        }
    }
    __syncthreads();
    const Acc inv = Acc(1) / l;
    for (int c = tid; c < dh; c += CLS_THREADS) {
        Acc a = 0;
        for (int gg = 0; gg < G; ++gg) a += red[gg * dh + c];
        if constexpr (sizeof(Acc) == 8)
            o[n * ldo + col + c] = a * inv;
        else
            o[n * ldo + col + c] = from_acc<T>(a * inv);
    }
}

int64_t red_len_for(int64_t dh, bool pairs) {
    const int64_t NU = pairs ? dh / 2 : dh;
    const int64_t G = NU >= CLS_THREADS ? 1 : CLS_THREADS / NU;
    return G * dh;
}

size_t smem_bytes(int64_t T, int64_t dh, bool pairs, size_t acc) {
    return (size_t)(dh + T + red_len_for(dh, pairs) + CLS_WARPS) * acc;
}

constexpr size_t kMaxSmem = 200 * 1024;

template <typename E, typename Acc, bool VEC, bool PAIRS>
cudaError_t launch_t(const void* q, int64_t ldq, const void* k, const void* v, int64_t ldkv, int64_t N, int64_t T,
                     int64_t H, int64_t dh, Acc scale, void* o, int64_t ldo, cudaStream_t s) {
    const size_t smem = smem_bytes(T, dh, PAIRS, sizeof(Acc));
    auto kern = attention_cls_kernel<E, Acc, VEC, PAIRS>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    kern<<<(unsigned)(N * H), CLS_THREADS, smem, s>>>(
        static_cast<const E*>(q), ldq, static_cast<const E*>(k), static_cast<const E*>(v), ldkv, (int)T, (int)H,
        (int)dh, (int)red_len_for(dh, PAIRS), scale, static_cast<E*>(o), ldo);
    return cudaGetLastError();
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

bool attention_cls_supported(int64_t N, int64_t T, int64_t D, int64_t H, int dt) {
    if (N <= 0 || T <= 0 || H <= 0 || D % H != 0 || N * H > 0x7fffffff || T > 0x7fffffff) return false;
    const int64_t dh = D / H;
    const bool pairs = dt == DT_BF16 && dh % 2 == 0;
    return smem_bytes(T, dh, pairs, dt == DT_F64 ? 8 : 4) <= kMaxSmem;
}

cudaError_t launch_attention_cls(const void* q, int64_t ldq, const void* k, const void* v, int64_t ldkv, int dt,
                                 int64_t N, int64_t T, int64_t D, int64_t H, void* o, int64_t ldo, cudaStream_t s) {
    if (N <= 0 || T <= 0) return cudaSuccess;
    if (!attention_cls_supported(N, T, D, H, dt)) return cudaErrorInvalidValue;
    const int64_t dh = D / H;
    const size_t es = dt_size(dt);
    // 16-byte key loads need every key row segment 16-byte aligned
    const bool vec = dt != DT_F64 && al16(k) && (ldkv * (int64_t)es) % 16 == 0 && (dh * (int64_t)es) % 16 == 0;
    if (dt == DT_BF16) {
        const float scale = (float)(1.4426950408889634 / sqrt((double)dh));
        const bool pairs = dh % 2 == 0 && (reinterpret_cast<uintptr_t>(v) & 3) == 0 && ldkv % 2 == 0;
        if (vec && pairs)
            return launch_t<__nv_bfloat16, float, true, true>(q, ldq, k, v, ldkv, N, T, H, dh, scale, o, ldo, s);
        if (pairs)
            return launch_t<__nv_bfloat16, float, false, true>(q, ldq, k, v, ldkv, N, T, H, dh, scale, o, ldo, s);
        return launch_t<__nv_bfloat16, float, false, false>(q, ldq, k, v, ldkv, N, T, H, dh, scale, o, ldo, s);
    }
    if (dt == DT_F32) {
        const float scale = (float)(1.4426950408889634 / sqrt((double)dh));
        if (vec) return launch_t<float, float, true, false>(q, ldq, k, v, ldkv, N, T, H, dh, scale, o, ldo, s);
        return launch_t<float, float, false, false>(q, ldq, k, v, ldkv, N, T, H, dh, scale, o, ldo, s);
    }
    if (dt == DT_F64)
        return launch_t<double, double, false, false>(q, ldq, k, v, ldkv, N, T, H, dh, 1.0 / sqrt((double)dh), o, ldo,
                                                      s);
    return cudaErrorInvalidValue;
}

}  // namespace vit
