// attention.cu -- bidirectional multi-head attention, flash style, bf16 in/out.
// "ViT Encoder Block" (crackedaicode), "Multi-head attention":
//   per sequence n and head h: softmax(Q_h K_h^T / sqrt(D/H)) V_h over ALL T keys
//   (no mask), heads written back side by side in their original order.
// Q, K and V are read in place from the fused (N, T, 3D) buffer [Q | K | V], head h at
// columns h*dh of each block ("vision1 reference transcript" (nipunbatra.github.io),
// Page 106); the (T, T) score matrix is never stored.
//
// Kernel: one CTA of 4 warps per (64-query tile, head, sequence); each warp owns 16
// query rows. K/V tiles of 64 keys are double-buffered in shared memory with
// cp.async (keys past T are zero-filled and their scores set to -inf, so a tail tile
// of 197 = 3*64 + 5 keys contributes nothing extra). Scores and P.V run on the
// tensor cores (bf16 inputs, fp32 accumulators); the online softmax keeps a running
// row maximum and sum in fp32, working in base 2 with log2(e)/sqrt(dh) folded into
// one scale. P is rounded to bf16 for the P.V product.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"

namespace vit {
namespace {

constexpr int BQ = 64, BKV = 64, ATT_THREADS = 128;

__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
}

// D (16x8 f32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int DH>
__global__ void __launch_bounds__(ATT_THREADS)
attention_mma_kernel(const __nv_bfloat16* __restrict__ qkv, __nv_bfloat16* __restrict__ o, int T,
                     int D, float scale_log2) {
    constexpr int LDS = DH + 8;       // padded row: ldmatrix rows land on distinct banks
    constexpr int CPR = DH / 8;       // 16-byte chunks per head row
    constexpr int KC = DH / 16;       // k-chunks of the score product
    constexpr int DB = DH / 8;        // 8-column blocks of the output
    extern __shared__ __align__(16) uint8_t att_smem[];
    __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(att_smem);
    __nv_bfloat16* sK = sQ + BQ * LDS;          // [2][BKV][LDS]
    __nv_bfloat16* sV = sK + 2 * BKV * LDS;     // [2][BKV][LDS]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q0 = blockIdx.x * BQ;
    const int h = blockIdx.y;
    const int64_t n = blockIdx.z;
    const int64_t ld = 3 * (int64_t)D;
    const __nv_bfloat16* base = qkv + n * T * ld;
    const int qcol = h * DH, kcol = D + h * DH, vcol = 2 * D + h * DH;

    for (int c = tid; c < BQ * CPR; c += ATT_THREADS) {
        const int r = c / CPR, ch = c % CPR;
        const int t = q0 + r;
        const __nv_bfloat16* src = base + (int64_t)(t < T ? t : 0) * ld + qcol + ch * 8;
        cp_async16(sQ + r * LDS + ch * 8, src, t < T ? 16 : 0);
    }
    auto load_kv = [&](int kt, int stage) {
        __nv_bfloat16* dk = sK + stage * BKV * LDS;
        __nv_bfloat16* dv = sV + stage * BKV * LDS;
        for (int c = tid; c < BKV * CPR; c += ATT_THREADS) {
            const int r = c / CPR, ch = c % CPR;
            const int t = kt * BKV + r;
            const int64_t off = (int64_t)(t < T ? t : 0) * ld + ch * 8;
            cp_async16(dk + r * LDS + ch * 8, base + off + kcol, t < T ? 16 : 0);
            cp_async16(dv + r * LDS + ch * 8, base + off + vcol, t < T ? 16 : 0);
        }
    };
    const int nkt = (T + BKV - 1) / BKV;
    load_kv(0, 0);
    cp_async_commit();

    uint32_t qf[KC][4];
    float oacc[DB][4];
#pragma unroll
    for (int i = 0; i < DB; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    const int g = lane >> 2, cq = lane & 3;

    for (int kt = 0; kt < nkt; ++kt) {
        if (kt + 1 < nkt) load_kv(kt + 1, (kt + 1) & 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        if (kt == 0) {
#pragma unroll
            for (int kc = 0; kc < KC; ++kc) {
                const int r = warp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
                const int c = kc * 16 + 8 * (lane >> 4);
                ldsm_x4(qf[kc], sQ + r * LDS + c);
            }
        }
        const __nv_bfloat16* cK = sK + (kt & 1) * BKV * LDS;
        const __nv_bfloat16* cV = sV + (kt & 1) * BKV * LDS;

        // S = Q K^T for this warp's 16 rows x 64 keys
        float s[BKV / 8][4];
#pragma unroll
        for (int nb = 0; nb < BKV / 8; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
#pragma unroll
        for (int kc = 0; kc < KC; ++kc) {
#pragma unroll
            for (int nb = 0; nb < BKV / 8; nb += 2) {
                uint32_t b[4];
                const int mi = lane >> 3;
                const int key = nb * 8 + 8 * (mi >> 1) + (lane & 7);
                const int c = kc * 16 + 8 * (mi & 1);
                ldsm_x4(b, cK + key * LDS + c);
                mma16816(s[nb], qf[kc], b[0], b[1]);
                mma16816(s[nb + 1], qf[kc], b[2], b[3]);
            }
        }
        // mask keys past T
        const int kbase = kt * BKV;
        if (kbase + BKV > T) {
#pragma unroll
            for (int nb = 0; nb < BKV / 8; ++nb) {
                const int k0 = kbase + nb * 8 + 2 * cq;
                if (k0 >= T) s[nb][0] = s[nb][2] = -INFINITY;
                if (k0 + 1 >= T) s[nb][1] = s[nb][3] = -INFINITY;
            }
        }
        // online softmax, rows g (regs 0,1) and g+8 (regs 2,3)
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nb = 0; nb < BKV / 8; ++nb) {
            mx[0] = fmaxf(mx[0], fmaxf(s[nb][0], s[nb][1]));
            mx[1] = fmaxf(mx[1], fmaxf(s[nb][2], s[nb][3]));
        }
        float alpha[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
            const float m_new = fmaxf(m_run[r], mx[r] * scale_log2);
            alpha[r] = exp2_approx(m_run[r] - m_new);
            m_run[r] = m_new;
            l_run[r] *= alpha[r];
        }
#pragma unroll
        for (int db = 0; db < DB; ++db) {
            oacc[db][0] *= alpha[0];
            oacc[db][1] *= alpha[0];
            oacc[db][2] *= alpha[1];
            oacc[db][3] *= alpha[1];
        }
        uint32_t pf[BKV / 16][4];
#pragma unroll
        for (int nb = 0; nb < BKV / 8; ++nb) {
            const float p0 = exp2_approx(fmaf(s[nb][0], scale_log2, -m_run[0]));
            const float p1 = exp2_approx(fmaf(s[nb][1], scale_log2, -m_run[0]));
            const float p2 = exp2_approx(fmaf(s[nb][2], scale_log2, -m_run[1]));
            const float p3 = exp2_approx(fmaf(s[nb][3], scale_log2, -m_run[1]));
            l_run[0] += p0 + p1;
            l_run[1] += p2 + p3;
            const int kk = nb >> 1, hi = nb & 1;
            pf[kk][0 + 2 * hi] = pack_bf16x2(p0, p1);
            pf[kk][1 + 2 * hi] = pack_bf16x2(p2, p3);
        }
        // O += P V
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk) {
#pragma unroll
            for (int db = 0; db < DB; db += 2) {
                uint32_t b[4];
                const int mi = lane >> 3;
                const int key = kk * 16 + 8 * (mi & 1) + (lane & 7);
                const int c = 8 * (db + (mi >> 1));
                ldsm_x4_t(b, cV + key * LDS + c);
                mma16816(oacc[db], pf[kk], b[0], b[1]);
                mma16816(oacc[db + 1], pf[kk], b[2], b[3]);
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

#pragma unroll
    for (int r = 0; r < 2; ++r) {
        l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
        l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
    }
    const float inv0 = 1.f / l_run[0], inv1 = 1.f / l_run[1];
    const int t0 = q0 + warp * 16 + g, t1 = t0 + 8;
    __nv_bfloat16* orow0 = o + (n * T + t0) * (int64_t)D + h * DH;
    __nv_bfloat16* orow1 = o + (n * T + t1) * (int64_t)D + h * DH;
#pragma unroll
    for (int db = 0; db < DB; ++db) {
        const int c = db * 8 + 2 * cq;
        if (t0 < T)
            *reinterpret_cast<uint32_t*>(orow0 + c) = pack_bf16x2(oacc[db][0] * inv0, oacc[db][1] * inv0);
        if (t1 < T)
            *reinterpret_cast<uint32_t*>(orow1 + c) = pack_bf16x2(oacc[db][2] * inv1, oacc[db][3] * inv1);
    }
}

template <int DH>
cudaError_t launch_dh(const void* qkv, void* o, int64_t N, int64_t T, int64_t D, cudaStream_t s) {
    constexpr int LDS = DH + 8;
    constexpr int smem = (BQ + 4 * BKV) * LDS * 2;
    static std::atomic<uint64_t> attr{0};
    cudaError_t e = set_smem_limit_once(attention_mma_kernel<DH>, smem, attr);
    if (e != cudaSuccess) return e;
    const int64_t H = D / DH;
    dim3 grid((unsigned)((T + BQ - 1) / BQ), (unsigned)H, (unsigned)N);
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)DH);
    attention_mma_kernel<DH><<<grid, ATT_THREADS, smem, s>>>(
        static_cast<const __nv_bfloat16*>(qkv), static_cast<__nv_bfloat16*>(o), (int)T, (int)D,
        scale_log2);
    return cudaGetLastError();
}

}  // namespace

bool attention_fast_supported(int64_t D, int64_t H, const void* qkv, const void* o) {
    if (H <= 0 || D % H != 0) return false;
    const int64_t dh = D / H;
    if (dh != 32 && dh != 64 && dh != 80 && dh != 96 && dh != 128) return false;
    if ((reinterpret_cast<uintptr_t>(qkv) & 15) || (reinterpret_cast<uintptr_t>(o) & 3)) return false;
    return true;
}

cudaError_t launch_attention_fast(const void* qkv, void* o, int64_t N, int64_t T, int64_t D,
                                  int64_t H, cudaStream_t s) {
    if (N <= 0 || T <= 0) return cudaSuccess;
    if (N > 65535 || H > 65535 || T > 0x7fffffff / 4) return cudaErrorInvalidValue;
    switch (D / H) {
        case 32: return launch_dh<32>(qkv, o, N, T, D, s);
        case 64: return launch_dh<64>(qkv, o, N, T, D, s);
        case 80: return launch_dh<80>(qkv, o, N, T, D, s);
        case 96: return launch_dh<96>(qkv, o, N, T, D, s);
        case 128: return launch_dh<128>(qkv, o, N, T, D, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace vit
