// generic.cu -- CUDA-core kernels that cover every shape and element type (fp64,
// fp32, bf16): the path for VIT_F64 and VIT_F32, and for bf16 shapes the
// tensor-core kernels do not take. Deterministic: each output is one thread's
// ascending-k sum, no atomics.
//
// GEMM: out (M, N) = epilogue(a (M, K) @ w (K, N) [+ bias]); 64 x 64 output tile per
// CTA, 16-deep k slabs staged in shared memory, 4 x 4 outputs per thread.
// Attention ("ViT Encoder Block" (crackedaicode), "Multi-head attention"): one thread
// per (sequence, head, query); pass 1 finds the row maximum of the scaled scores,
// pass 2 the softmax denominator, pass 3 accumulates the weighted value rows 16
// output columns at a time.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace vit {
namespace {

template <typename Acc>
__device__ __forceinline__ Acc ld_elem(const void* p, int dt, int64_t i) {
    if (dt == DT_F32) return (Acc) static_cast<const float*>(p)[i];
    if (dt == DT_BF16) return (Acc)__bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
    return (Acc) static_cast<const double*>(p)[i];
}

template <typename Acc>
__device__ __forceinline__ void st_elem(void* p, int dt, int64_t i, Acc v) {
    if (dt == DT_F32)
        static_cast<float*>(p)[i] = (float)v;
    else if (dt == DT_BF16)
        static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn((float)v);
    else
        static_cast<double*>(p)[i] = (double)v;
}

__device__ __forceinline__ float gelu_acc(float z) { return gelu_tanh_acc(z); }
__device__ __forceinline__ double gelu_acc(double z) { return gelu_tanh_acc(z); }
__device__ __forceinline__ float exp_acc(float z) { return expf(z); }
__device__ __forceinline__ double exp_acc(double z) { return exp(z); }

constexpr int GT = 64, GK = 16;

template <typename Acc>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const SimtGemmDesc d) {
    __shared__ Acc As[GK][GT + 1];
    __shared__ Acc Ws[GK][GT];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int64_t m0 = (int64_t)blockIdx.y * GT, n0 = (int64_t)blockIdx.x * GT;
    Acc acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0;
    for (int64_t k0 = 0; k0 < d.K; k0 += GK) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = threadIdx.x + 256 * i;
            const int m = e / GK, k = e % GK;
            const int64_t gm = m0 + m, gk = k0 + k;
            As[k][m] = (gm < d.M && gk < d.K) ? ld_elem<Acc>(d.a, d.a_dt, gm * d.lda + gk) : (Acc)0;
            const int kk = e / GT, n = e % GT;
            const int64_t gk2 = k0 + kk, gn = n0 + n;
            Ws[kk][n] = (gk2 < d.K && gn < d.N) ? ld_elem<Acc>(d.w, d.w_dt, gk2 * d.ldw + gn) : (Acc)0;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < GK; ++k) {
            Acc am[4], wn[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) am[i] = As[k][ty * 4 + i];
#pragma unroll
            for (int j = 0; j < 4; ++j) wn[j] = Ws[k][tx * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fma(am[i], wn[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t m = m0 + ty * 4 + i;
        if (m >= d.M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t n = n0 + tx * 4 + j;
            if (n >= d.N) continue;
            Acc v = acc[i][j];
            if (d.bias) v = v + ld_elem<Acc>(d.bias, d.bias_dt, n);
            if (d.epi == TC_EPI_GELU) v = gelu_acc(v);
            if (d.epi == TC_EPI_RESID) v = ld_elem<Acc>(d.residual, d.res_dt, m * d.ldr + n) + v;
            st_elem<Acc>(d.out, d.out_dt, m * d.ldo + n, v);
        }
    }
}

template <typename Acc>
__global__ void __launch_bounds__(128)
attention_simt_kernel(const void* qkv, int dt, void* o, int64_t N, int64_t T, int64_t D, int64_t H) {
    const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t rows = N * H * T;
    if (gid >= rows) return;
    const int64_t t = gid % T;
    const int64_t h = (gid / T) % H;
    const int64_t n = gid / (T * H);
    const int64_t dh = D / H;
    const int64_t ld = 3 * D;
    const int64_t qrow = (n * T + t) * ld + h * dh;
    const int64_t kbase = n * T * ld + D + h * dh;
    const int64_t vbase = n * T * ld + 2 * D + h * dh;
    const Acc scale = (Acc)1 / sqrt((Acc)dh);
    auto score = [&](int64_t u) {
        Acc s = 0;
        for (int64_t c = 0; c < dh; ++c)
            s = fma(ld_elem<Acc>(qkv, dt, qrow + c), ld_elem<Acc>(qkv, dt, kbase + u * ld + c), s);
        return s * scale;
    };
    Acc m = score(0);
    for (int64_t u = 1; u < T; ++u) {
        const Acc s = score(u);
        m = s > m ? s : m;
    }
    Acc l = 0;
    for (int64_t u = 0; u < T; ++u) l += exp_acc(score(u) - m);
    const int64_t orow = (n * T + t) * D + h * dh;
    for (int64_t c0 = 0; c0 < dh; c0 += 16) {
        Acc acc[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) acc[c] = 0;
        for (int64_t u = 0; u < T; ++u) {
            const Acc p = exp_acc(score(u) - m) / l;
#pragma unroll
            for (int c = 0; c < 16; ++c)
                if (c0 + c < dh) acc[c] = fma(p, ld_elem<Acc>(qkv, dt, vbase + u * ld + c0 + c), acc[c]);
        }
#pragma unroll
        for (int c = 0; c < 16; ++c)
            if (c0 + c < dh) st_elem<Acc>(o, dt, orow + c0 + c, acc[c]);
    }
}

}  // namespace

cudaError_t launch_gemm_simt(const SimtGemmDesc& d, cudaStream_t s) {
    if (d.M <= 0 || d.N <= 0) return cudaSuccess;
    const int64_t gx = (d.N + GT - 1) / GT, gy = (d.M + GT - 1) / GT;
    if (gx > 0x7fffffff || gy > 65535) return cudaErrorInvalidValue;
    dim3 grid((unsigned)gx, (unsigned)gy);
    if (d.a_dt == DT_F64)
        gemm_simt_kernel<double><<<grid, 256, 0, s>>>(d);
    else
        gemm_simt_kernel<float><<<grid, 256, 0, s>>>(d);
    return cudaGetLastError();
}

cudaError_t launch_attention_simt(const void* qkv, int dt, void* o, int64_t N, int64_t T, int64_t D,
                                  int64_t H, cudaStream_t s) {
    const int64_t rows = N * H * T;
    if (rows <= 0) return cudaSuccess;
    const int64_t blocks = (rows + 127) / 128;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    if (dt == DT_F64)
        attention_simt_kernel<double><<<(unsigned)blocks, 128, 0, s>>>(qkv, dt, o, N, T, D, H);
    else
        attention_simt_kernel<float><<<(unsigned)blocks, 128, 0, s>>>(qkv, dt, o, N, T, D, H);
    return cudaGetLastError();
}

}  // namespace vit
