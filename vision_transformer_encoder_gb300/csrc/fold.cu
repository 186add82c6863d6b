// fold.cu -- LayerNorm folded into the following GEMM.
//
// "ViT Encoder Block" (crackedaicode), "Normalize before each stage", with the optional
// gain/bias of "ViT Encoder Block" (ai-engineer-exhaustive), Key Equations, Step 1:
//   LN(x) @ W = rstd * (x @ W' - mean * c) + d,   W' = diag(gamma) W,
//   c_j = sum_i W'_ij,  d_j = sum_i beta_i W_ij (+ a bias b_j of the next layer),
// with mean and rstd = 1/sqrt(var + eps) of each row of x. The GEMM then reads x itself
// (no normalised copy is written and read back) and applies the per-row and
// per-column terms in its epilogue.
//
// Row statistics travel as partials (mean, M2) over fixed column ranges, M2 the sum of
// squared deviations from the partial's own mean; a consumer merges them with Chan's
// formula, which has no cancellation (a constant row gives M2 = 0 exactly).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace vit {
namespace {

constexpr int ST_THREADS = 256;  // 8 rows per CTA

template <int MAXV>
__global__ void __launch_bounds__(ST_THREADS)
row_parts_kernel(const __nv_bfloat16* __restrict__ x, float2* __restrict__ parts, int64_t rows, int D) {
    griddep_wait();                 // x may be the previous kernel's output
    griddep_launch_dependents();
    const int64_t row = (int64_t)blockIdx.x * (ST_THREADS / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int nvec = D / 8;
    const __nv_bfloat16* xr = x + row * D;
    float v[MAXV][8];
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
        const int idx = lane + 32 * j;
        if (idx < nvec) {
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(xr) + idx);
            const float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y), c = unpack_bf16x2(u.z),
                         d = unpack_bf16x2(u.w);
            v[j][0] = a.x; v[j][1] = a.y; v[j][2] = b.x; v[j][3] = b.y;
            v[j][4] = c.x; v[j][5] = c.y; v[j][6] = d.x; v[j][7] = d.y;
#pragma unroll
            for (int e = 0; e < 8; ++e) sum += v[j][e];
        }
    }
    const float mean = warp_sum(sum) / (float)D;
    float sq = 0.f;
#pragma unroll
    for (int j = 0; j < MAXV; ++j) {
        const int idx = lane + 32 * j;
        if (idx < nvec) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float d = v[j][e] - mean;
                sq += d * d;
            }
        }
    }
    const float m2 = warp_sum(sq);
    if (lane == 0) parts[row] = make_float2(mean, m2);
}

// Column terms in two passes, both deterministic. Pass 1: CTA (column group of 64,
// row chunk of 64): each thread owns two adjacent columns (one bf16 pair per row) and
// 8 rows; the 8 row groups are summed in a fixed order in shared memory and written as
// one partial per (row chunk, column). Pass 2 adds the partials of each column in row-
// chunk order and the layer bias.
constexpr int FP_COLS = 64, FP_ROWS = 64;

__global__ void __launch_bounds__(256)
fold_partial_kernel(const FoldPrep d, float* __restrict__ part_c, float* __restrict__ part_d) {
    __shared__ float sc[8][FP_COLS], sd[8][FP_COLS];
    const int tid = threadIdx.x;
    const int pair = tid & 31, rg = tid >> 5;
    const int64_t col = (int64_t)blockIdx.x * FP_COLS + 2 * pair;   // even; N % 64 == 0
    const int wi = (int)(col / d.n_per_w);
    const int64_t lc = col - (int64_t)wi * d.n_per_w;
    const __nv_bfloat16* w = static_cast<const __nv_bfloat16*>(d.w[wi]);
    __nv_bfloat16* ws = d.gamma ? static_cast<__nv_bfloat16*>(d.w_scaled[wi]) : nullptr;
    const __nv_bfloat16* g = static_cast<const __nv_bfloat16*>(d.gamma);
    const __nv_bfloat16* b = static_cast<const __nv_bfloat16*>(d.beta);
    const int64_t k0 = (int64_t)blockIdx.y * FP_ROWS + rg * (FP_ROWS / 8);
    float c0 = 0.f, c1 = 0.f, d0 = 0.f, d1 = 0.f;
#pragma unroll
    for (int i = 0; i < FP_ROWS / 8; ++i) {
        const int64_t k = k0 + i;
        if (k < d.K) {
            const uint32_t raw = __ldg(reinterpret_cast<const uint32_t*>(w + k * d.n_per_w + lc));
            float2 wf = unpack_bf16x2(raw);
            if (b) {
                const float bk = __bfloat162float(b[k]);
                d0 = fmaf(bk, wf.x, d0);
                d1 = fmaf(bk, wf.y, d1);
            }
            if (g) {
                const float gk = __bfloat162float(g[k]);
                const uint32_t sv = pack_bf16x2(gk * wf.x, gk * wf.y);
                *reinterpret_cast<uint32_t*>(ws + k * d.n_per_w + lc) = sv;
                wf = unpack_bf16x2(sv);   // the MMA reads the rounded scaled weight
            }
            c0 += wf.x;
            c1 += wf.y;
        }
    }
    sc[rg][2 * pair] = c0; sc[rg][2 * pair + 1] = c1;
    sd[rg][2 * pair] = d0; sd[rg][2 * pair + 1] = d1;
    __syncthreads();
    if (tid < FP_COLS) {
        float tc = 0.f, td = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            tc += sc[i][tid];
            td += sd[i][tid];
        }
        const int64_t c = (int64_t)blockIdx.x * FP_COLS + tid;
        part_c[(int64_t)blockIdx.y * d.N + c] = tc;
        part_d[(int64_t)blockIdx.y * d.N + c] = td;
    }
}

__global__ void __launch_bounds__(256)
fold_finish_kernel(const FoldPrep d, const float* __restrict__ part_c, const float* __restrict__ part_d,
                   int chunks) {
    const int64_t col = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (col >= d.N) return;
    float tc = 0.f, td = 0.f;
    for (int i = 0; i < chunks; ++i) {
        tc += part_c[(int64_t)i * d.N + col];
        td += part_d[(int64_t)i * d.N + col];
    }
    if (d.bias) td += __bfloat162float(static_cast<const __nv_bfloat16*>(d.bias)[col]);
    d.colsum[col] = tc;
    d.colbias[col] = td;
}

template <int MAXV>
cudaError_t launch_parts(const void* x, float2* parts, int64_t rows, int64_t D, cudaStream_t s) {
    const int64_t blocks = (rows + ST_THREADS / 32 - 1) / (ST_THREADS / 32);
    return launch_dependent(row_parts_kernel<MAXV>, dim3((unsigned)blocks), dim3(ST_THREADS), 0, s,
                            static_cast<const __nv_bfloat16*>(x), parts, rows, (int)D);
}

}  // namespace

bool row_parts_supported(int64_t D, const void* x) {
    return D % 8 == 0 && D <= 2048 && (reinterpret_cast<uintptr_t>(x) & 15) == 0;
}

cudaError_t launch_row_parts(const void* x, float2* parts, int64_t rows, int64_t D, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    const int per_lane = (int)((D / 8 + 31) / 32);
    switch (per_lane) {
        case 1: return launch_parts<1>(x, parts, rows, D, s);
        case 2: return launch_parts<2>(x, parts, rows, D, s);
        case 3: return launch_parts<3>(x, parts, rows, D, s);
        case 4: return launch_parts<4>(x, parts, rows, D, s);
        case 5: return launch_parts<5>(x, parts, rows, D, s);
        case 6: return launch_parts<6>(x, parts, rows, D, s);
        default: return launch_parts<8>(x, parts, rows, D, s);
    }
}

size_t fold_prep_scratch_bytes(int64_t N, int64_t K) {
    return (size_t)((K + FP_ROWS - 1) / FP_ROWS) * (size_t)N * 2 * sizeof(float);
}

cudaError_t launch_fold_prep(const FoldPrep& d, float* scratch, cudaStream_t s) {
    if (d.N <= 0) return cudaSuccess;
    if (d.N % FP_COLS != 0 || d.n_per_w % FP_COLS != 0) return cudaErrorInvalidValue;
    const int chunks = (int)((d.K + FP_ROWS - 1) / FP_ROWS);
    float* part_c = scratch;
    float* part_d = scratch + (size_t)chunks * d.N;
    fold_partial_kernel<<<dim3((unsigned)(d.N / FP_COLS), (unsigned)chunks), 256, 0, s>>>(d, part_c, part_d);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    fold_finish_kernel<<<(unsigned)((d.N + 255) / 256), 256, 0, s>>>(d, part_c, part_d, chunks);
    return cudaGetLastError();
}

}  // namespace vit
