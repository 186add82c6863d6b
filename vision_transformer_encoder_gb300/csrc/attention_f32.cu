// attention_f32.cu -- fp32 multi-head attention on the CUDA cores (the fp32 path), for the
// shapes the 3xTF32 tensor-core kernel (attention_tf32.cu) does not take.
//
// "ViT Encoder Block" (crackedaicode), "Multi-head attention": per sequence n and head
// h, out_h = softmax(Q_h K_h^T / sqrt(D/H)) V_h with every key visible; heads written
// side by side in order, Q, K and V read in place from the fused (N, T, 3D) buffer.
//
// One CTA of 128 threads per (sequence, head, block of query rows). TPR threads share a
// query row (1 for head widths up to 64, 2 up to 128), each holding DH / TPR columns of
// the row's q and of its output accumulator in registers. Keys and values pass through
// shared memory 32 at a time; every thread of the CTA reads the same key row, so the
// reads are broadcasts. Online softmax in base 2 in fp32: per 32-key tile the scores,
// the new running maximum, one rescale of the accumulator and of the row sum, then
// P V. Keys past T score -inf.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace vit {
namespace {

constexpr int AF_THREADS = 128;
constexpr int AF_KT = 32;   // keys per shared-memory tile

template <int DH, int TPR>
__global__ void __launch_bounds__(AF_THREADS)
attention_f32_kernel(const float* __restrict__ qkv, float* __restrict__ o, int T, int D, float sl2) {
    constexpr int ROWS = AF_THREADS / TPR;   // query rows per CTA
    constexpr int DW = DH / TPR;             // columns per thread
    static_assert(DH % (4 * TPR) == 0, "columns per thread in whole float4s");
    __shared__ __align__(16) float sK[AF_KT][DH];
    __shared__ __align__(16) float sV[AF_KT][DH];

    const int h = blockIdx.y, n = blockIdx.z;
    const int sub = threadIdx.x % TPR;                       // which columns of the row
    const int t = blockIdx.x * ROWS + threadIdx.x / TPR;     // query row
    const int64_t ld = 3 * (int64_t)D;
    const float* seq = qkv + (int64_t)n * T * ld;
    const int c0 = sub * DW;

    float q[DW], acc[DW];
    const bool valid = t < T;
#pragma unroll
    for (int c = 0; c < DW; c += 4) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (valid) v = *reinterpret_cast<const float4*>(seq + (int64_t)t * ld + h * DH + c0 + c);
        q[c] = v.x; q[c + 1] = v.y; q[c + 2] = v.z; q[c + 3] = v.w;
        acc[c] = acc[c + 1] = acc[c + 2] = acc[c + 3] = 0.f;
    }
    float m = -INFINITY, l = 0.f;

    for (int k0 = 0; k0 < T; k0 += AF_KT) {
        __syncthreads();   // the previous tile is consumed
        for (int i = threadIdx.x; i < AF_KT * DH / 4; i += AF_THREADS) {
            const int r = i / (DH / 4), c4 = i % (DH / 4);
            const int u = k0 + r;
            float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
            if (u < T) {
                const float* row = seq + (int64_t)u * ld + h * DH;
                kv = reinterpret_cast<const float4*>(row + D)[c4];
                vv = reinterpret_cast<const float4*>(row + 2 * D)[c4];
            }
            reinterpret_cast<float4*>(&sK[r][0])[c4] = kv;
            reinterpret_cast<float4*>(&sV[r][0])[c4] = vv;
        }
        __syncthreads();
        const int nk = T - k0 < AF_KT ? T - k0 : AF_KT;
        float s[AF_KT];
        float mt = -INFINITY;
#pragma unroll
        for (int j = 0; j < AF_KT; ++j) {
            float d0 = 0.f, d1 = 0.f;
#pragma unroll
            for (int c = 0; c < DW; c += 2) {
                d0 = fmaf(q[c], sK[j][c0 + c], d0);
                d1 = fmaf(q[c + 1], sK[j][c0 + c + 1], d1);
            }
            float d = d0 + d1;
            if (TPR == 2) d += __shfl_xor_sync(0xffffffffu, d, 1);
            s[j] = j < nk ? d * sl2 : -INFINITY;
            mt = fmaxf(mt, s[j]);
        }
        const float mn = fmaxf(m, mt);
        const float alpha = exp2f(m - mn);   // 0 on the first tile (m = -inf)
        l *= alpha;
#pragma unroll
        for (int c = 0; c < DW; ++c) acc[c] *= alpha;
#pragma unroll
        for (int j = 0; j < AF_KT; ++j) {
            const float pj = exp2f(s[j] - mn);
            l += pj;
#pragma unroll
            for (int c = 0; c < DW; ++c) acc[c] = fmaf(pj, sV[j][c0 + c], acc[c]);
        }
        m = mn;
    }
    if (valid) {
        const float inv = 1.f / l;
        float* orow = o + ((int64_t)n * T + t) * D + h * DH + c0;
#pragma unroll
        for (int c = 0; c < DW; c += 4)
            *reinterpret_cast<float4*>(orow + c) =
                make_float4(acc[c] * inv, acc[c + 1] * inv, acc[c + 2] * inv, acc[c + 3] * inv);
    }
}

template <int DH, int TPR>
cudaError_t launch_dh(const void* qkv, void* o, int64_t N, int64_t T, int64_t D, cudaStream_t s) {
    constexpr int ROWS = AF_THREADS / TPR;
    const int64_t H = D / DH;
    const dim3 grid((unsigned)((T + ROWS - 1) / ROWS), (unsigned)H, (unsigned)N);
    const float sl2 = (float)(1.4426950408889634 / sqrt((double)DH));
    attention_f32_kernel<DH, TPR><<<grid, AF_THREADS, 0, s>>>(static_cast<const float*>(qkv),
                                                             static_cast<float*>(o), (int)T, (int)D, sl2);
    return cudaGetLastError();
}

}  // namespace

bool attention_f32_supported(int64_t N, int64_t T, int64_t D, int64_t H, const void* qkv, const void* o) {
    if (H <= 0 || D % H != 0 || N > 65535 || H > 65535 || T > (int64_t)0x7fffffff / 3 / (D > 0 ? D : 1)) return false;
    const int64_t dh = D / H;
    if (dh != 32 && dh != 48 && dh != 64 && dh != 80 && dh != 96 && dh != 128) return false;
    return (reinterpret_cast<uintptr_t>(qkv) & 15) == 0 && (reinterpret_cast<uintptr_t>(o) & 15) == 0;
}

cudaError_t launch_attention_f32(const void* qkv, void* o, int64_t N, int64_t T, int64_t D, int64_t H,
                                 const DeviceInfo& dev, cudaStream_t s, float* o_lo) {
    if (N <= 0 || T <= 0) return cudaSuccess;
    // head width 64 and at most 224 tokens: the 3xTF32 tensor-core kernel (writes o_lo itself)
    if (attention_tf32_supported(N, T, D, H, qkv, o)) return launch_attention_tf32(qkv, o, N, T, D, H, dev, s, o_lo);
    cudaError_t e = cudaErrorInvalidValue;
    switch (D / H) {
        case 32: e = launch_dh<32, 1>(qkv, o, N, T, D, s); break;
        case 48: e = launch_dh<48, 1>(qkv, o, N, T, D, s); break;
        case 64: e = launch_dh<64, 1>(qkv, o, N, T, D, s); break;
        case 80: e = launch_dh<80, 2>(qkv, o, N, T, D, s); break;
        case 96: e = launch_dh<96, 2>(qkv, o, N, T, D, s); break;
        case 128: e = launch_dh<128, 2>(qkv, o, N, T, D, s); break;
    }
    if (e == cudaSuccess && o_lo) e = launch_split_lo(static_cast<const float*>(o), N * T, D, D, o_lo, s);
    return e;
}

}  // namespace vit
