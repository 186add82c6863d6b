// attention_tf32.cu -- fp32 multi-head attention on the sm_103a tensor cores, for head
// width 64 and at most 224 tokens, with every product as three TF32 products ("3xTF32").
//
// "ViT Encoder Block" (crackedaicode), "Multi-head attention": per sequence n and head
// h, out_h = softmax(Q_h K_h^T / sqrt(D/H)) V_h with every key visible; heads written
// side by side in order, Q, K and V read in place from the fused (N, T, 3D) buffer.
//
// Precision: a product A B is taken as A_hi B_hi + A_hi B_lo + A_lo B_hi, where x_hi is
// the TF32 value the tensor core takes from an fp32 operand (the 13 low mantissa bits
// cleared) and x_lo = x - x_hi, exact in fp32; the dropped A_lo B_lo is 2^-20 of the
// product. A single TF32 product would leave errors near 1e-3.
//
// With at most 224 keys, S = Q K^T of a 128-row query tile is one M 128 x N ns MMA chain
// (ns = T rounded up to 16), so the row maximum is known before any exponent and the
// softmax is one exact pass. A unit is (sequence, head, 128-row query tile). One CTA per
// SM, 16 warps, the unit's steps in order:
//   1. Q and K arrive by TMA (128-byte swizzled rows of 32 fp32; rows past T read as 0);
//      all warps write their lo parts beside them in shared memory (same layout).
//   2. One thread issues the 24 S MMAs (8 K steps x 3 products) into TMEM.
//   3. Warps 0-7 (two per TMEM lane quarter, splitting the keys) take the row maximum,
//      then write P = exp2((S - max) log2(e) / sqrt(dh)) over S in TMEM and P_lo to a
//      second TMEM region, and keep the row sums. Meanwhile V arrives by TMA in the
//      space Q used, and warps 8-15 write V^T and V^T_lo (head columns as rows, keys
//      contiguous, the K-major layout the MMA reads for B) where K was.
//   4. One thread issues the P.V MMAs (3 per 8-key step) with P and P_lo read from TMEM;
//      the next unit's Q is loaded meanwhile.
//   5. Warps 8-11 read O, divide by the row sum and store fp32 rows; the next unit's K is
//      loaded meanwhile.
// TMEM, 512 columns: S / P at [0, 224), P_lo at [224, 448), O at [448, 512).
// Every mbarrier wait is bounded; on expiry the kernel records an error bit and every
// thread still passes each __syncthreads of the unit, then all leave together.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "ptx.cuh"

namespace vit {
namespace {

constexpr int A3_DH = 64;
constexpr int A3_ROWS = 128;                   // query rows per unit (TMEM lanes)
constexpr int A3_MAX_KEYS = 224;
constexpr int A3_THREADS = 512;                // 16 warps
constexpr int A3_HELP_WARP = 8;                // warps 8-15: lo parts of V, V^T; 8-11 epilogue
constexpr int A3_MMA_WARP = 12, A3_LOAD_WARP = 13;
constexpr int A3_QBOX = A3_ROWS * 128;         // 128 rows x 32 fp32: 16 KB
constexpr int A3_KBOX = A3_MAX_KEYS * 128;     // up to 224 rows x 32 fp32: 28 KB
constexpr int A3_VTBLK = A3_DH * 128;          // V^T block: 64 rows x 32 keys: 8 KB
constexpr int A3_OFF_Q = 0;                    // Q (2 blocks of 32 columns), then raw V
constexpr int A3_OFF_QL = 2 * A3_QBOX;         // Q_lo
constexpr int A3_OFF_K = 4 * A3_QBOX;          // K (2 blocks), then V^T (7 blocks of 32 keys)
constexpr int A3_OFF_KL = A3_OFF_K + 2 * A3_KBOX;
constexpr int A3_OFF_VT = A3_OFF_K;
constexpr int A3_OFF_VTL = A3_OFF_K + 7 * A3_VTBLK;
constexpr int A3_OFF_MX = A3_OFF_K + 4 * A3_KBOX;       // row maxima [half][row]
constexpr int A3_OFF_L = A3_OFF_MX + 2 * A3_ROWS * 4;   // row sums [half][row]
constexpr int A3_OFF_BAR = A3_OFF_L + 2 * A3_ROWS * 4;
constexpr int A3_STG = 32 * 128;                        // one 32 x 32 fp32 staging tile (128B swizzle)
constexpr int A3_OFF_STG = (A3_OFF_BAR + 128 + 1023) / 1024 * 1024;   // [epilogue warp][2 tiles]
constexpr int A3_SMEM = A3_OFF_STG + 4 * 2 * A3_STG + 1024;          // + alignment slack
constexpr uint32_t A3_TMEM_PL = 224, A3_TMEM_O = 448;
static_assert(2 * A3_KBOX <= A3_OFF_K, "raw V fits where Q and Q_lo were");
static_assert(2 * 7 * A3_VTBLK <= 4 * A3_KBOX, "V^T and V^T_lo fit where K and K_lo were");
static_assert(A3_SMEM <= 227 * 1024, "shared memory");

struct A3Params {
    int T, D, H;
    int ns;          // S columns: T rounded up to 16
    int nq;          // query tiles per (sequence, head)
    int units;       // N * H * nq
    float sl2;       // log2(e) / sqrt(64)
    float* o;
    bool lo;         // also write the low part of o (tmOlo)
    uint32_t* err;
};

struct A3Bars {
    uint64_t q_full, k_full, v_full, s_done, o_done, fin;
    uint32_t tmem_slot;
    int abort_flag;
};
static_assert(sizeof(A3Bars) <= 128, "barrier block");

__device__ __forceinline__ void a3_error(uint32_t* err, uint32_t bit) {
    if (err) atomicOr(err, bit);
}

__device__ __forceinline__ float tf32_lo(float x) {
    return x - __uint_as_float(__float_as_uint(x) & 0xFFFFE000u);
}

__device__ __forceinline__ float4 tf32_lo4(float4 v) {
    return make_float4(tf32_lo(v.x), tf32_lo(v.y), tf32_lo(v.z), tf32_lo(v.w));
}

// Instruction descriptor, kind::tf32: D fp32, A and B TF32, both K-major.
__host__ __device__ constexpr uint32_t a3_idesc(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(id), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_tf32_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a_tmem), "l"(b), "r"(id), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void a3_unit(const A3Params& p, int u, int& n, int& h, int& qt) {
    const int item = u / p.nq;
    qt = u - item * p.nq;
    n = item / p.H;
    h = item - n * p.H;
}

__global__ void __launch_bounds__(A3_THREADS, 1)
attention_tf32_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmKV,
                      const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmOlo,
                      const A3Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    float* sMx = reinterpret_cast<float*>(smem + A3_OFF_MX);
    float* sL = reinterpret_cast<float*>(smem + A3_OFF_L);
    A3Bars* bars = reinterpret_cast<A3Bars*>(smem + A3_OFF_BAR);
    volatile int* abort_flag = &bars->abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ns = p.ns;
    const bool loader = warp == A3_LOAD_WARP && lane == 0;
    const bool issuer = warp == A3_MMA_WARP && lane == 0;

    if (threadIdx.x == 0) {
        ptx::mbar_init(&bars->q_full, 1);
        ptx::mbar_init(&bars->k_full, 1);
        ptx::mbar_init(&bars->v_full, 1);
        ptx::mbar_init(&bars->s_done, 1);
        ptx::mbar_init(&bars->o_done, 1);
        ptx::mbar_init(&bars->fin, 1);
        bars->abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (loader) {
        ptx::prefetch_tensormap(&tmQ);
        ptx::prefetch_tensormap(&tmKV);
    }
    if (warp == A3_MMA_WARP) {
        ptx::tmem_alloc(&bars->tmem_slot, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;
    griddep_wait();   // qkv is the previous kernel's output
    griddep_launch_dependents();

    const uint32_t kv_bytes = 2u * (uint32_t)ns * 128u;
    auto load_q = [&](int u) {
        int n, h, qt;
        a3_unit(p, u, n, h, qt);
        ptx::mbar_arrive_expect_tx(&bars->q_full, 2 * A3_QBOX);
        for (int b = 0; b < 2; ++b)
            ptx::tma_load_3d(smem + A3_OFF_Q + b * A3_QBOX, &tmQ, &bars->q_full, h * A3_DH + 32 * b, qt * A3_ROWS, n);
    };
    auto load_k = [&](int u) {
        int n, h, qt;
        a3_unit(p, u, n, h, qt);
        ptx::mbar_arrive_expect_tx(&bars->k_full, kv_bytes);
        for (int b = 0; b < 2; ++b)
            ptx::tma_load_3d(smem + A3_OFF_K + b * A3_KBOX, &tmKV, &bars->k_full, p.D + h * A3_DH + 32 * b, 0, n);
    };
    auto load_v = [&](int u) {
        int n, h, qt;
        a3_unit(p, u, n, h, qt);
        ptx::mbar_arrive_expect_tx(&bars->v_full, kv_bytes);
        for (int b = 0; b < 2; ++b)
            ptx::tma_load_3d(smem + A3_OFF_Q + b * A3_KBOX, &tmKV, &bars->v_full, 2 * p.D + h * A3_DH + 32 * b, 0, n);
    };
    uint32_t ph_q = 0, ph_k = 0, ph_v = 0, ph_s = 0, ph_o = 0;
    // the loader's copies not yet known to have landed, with the phase each completes
    // (for the teardown, which must not leave a copy in flight)
    int pend_q = 0, pend_k = 0, pend_v = 0;
    uint32_t pph_q = 0, pph_k = 0, pph_v = 0;

    const int u0 = (int)blockIdx.x, ustep = (int)gridDim.x;
    if (loader && u0 < p.units) {
        load_q(u0);
        load_k(u0);
        pend_q = pend_k = 1;
    }
    auto fail = [&](uint32_t bit) {
        if (lane == 0) a3_error(p.err, bit);
        *abort_flag = 1;
    };

    for (int u = u0; u < p.units; u += ustep) {
        int n, h, qt;
        a3_unit(p, u, n, h, qt);
        const int unext = u + ustep < p.units ? u + ustep : -1;

        // ---- 1. Q and K in; their lo parts -----------------------------------------
        if (!ptx::mbar_wait_bounded(&bars->q_full, ph_q, abort_flag) ||
            !ptx::mbar_wait_bounded(&bars->k_full, ph_k, abort_flag))
            fail(ERRBIT_TIMEOUT_ATTENTION);
        else if (loader)
            pend_q = pend_k = 0;
        ph_q ^= 1;
        ph_k ^= 1;
        if (!*abort_flag) {
            const float4* q = reinterpret_cast<const float4*>(smem + A3_OFF_Q);
            float4* ql = reinterpret_cast<float4*>(smem + A3_OFF_QL);
            for (int i = threadIdx.x; i < 2 * A3_QBOX / 16; i += A3_THREADS) ql[i] = tf32_lo4(q[i]);
            const int kq = ns * 8;   // 16-byte units of one K block
            for (int i = threadIdx.x; i < 2 * kq; i += A3_THREADS) {
                const int b = i / kq, r = i - b * kq;
                const float4* k = reinterpret_cast<const float4*>(smem + A3_OFF_K + b * A3_KBOX);
                float4* kl = reinterpret_cast<float4*>(smem + A3_OFF_KL + b * A3_KBOX);
                kl[r] = tf32_lo4(k[r]);
            }
            ptx::fence_proxy_async_smem();   // generic-proxy writes before the MMAs read them
        }
        __syncthreads();

        // ---- 2. S = Q K^T ------------------------------------------------------------
        if (issuer && !*abort_flag) {
            ptx::tc_fence_after();
            const uint32_t idS = a3_idesc(A3_ROWS, ns);
            const uint64_t dq = ptx::smem_desc(ptx::smem_addr(smem + A3_OFF_Q), 16, 1024, ptx::kLayoutSw128);
            const uint64_t dql = ptx::smem_desc(ptx::smem_addr(smem + A3_OFF_QL), 16, 1024, ptx::kLayoutSw128);
            const uint64_t dk = ptx::smem_desc(ptx::smem_addr(smem + A3_OFF_K), 16, 1024, ptx::kLayoutSw128);
            const uint64_t dkl = ptx::smem_desc(ptx::smem_addr(smem + A3_OFF_KL), 16, 1024, ptx::kLayoutSw128);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                // 8 fp32 columns (32 bytes, 2 address units) per K step; blocks of 32 columns
                const uint64_t qo = (uint64_t)((ks >> 2) * (A3_QBOX >> 4) + (ks & 3) * 2);
                const uint64_t ko = (uint64_t)((ks >> 2) * (A3_KBOX >> 4) + (ks & 3) * 2);
                mma_tf32_ss(tmem, dq + qo, dk + ko, idS, ks > 0 ? 1u : 0u);
                mma_tf32_ss(tmem, dq + qo, dkl + ko, idS, 1u);
                mma_tf32_ss(tmem, dql + qo, dk + ko, idS, 1u);
            }
            ptx::mma_commit(&bars->s_done);
        }

        // ---- 3. softmax (warps 0-7); V in, V^T (warps 8-15) -------------------------
        if (!ptx::mbar_wait_bounded(&bars->s_done, ph_s, abort_flag)) fail(ERRBIT_TIMEOUT_ATTENTION);
        ph_s ^= 1;
        ptx::tc_fence_after();
        __syncthreads();   // one decision for all threads on whether the unit goes on
        const bool go = !*abort_flag;
        if (go && loader) {
            load_v(u);   // into the space of Q and Q_lo: the S MMAs have read them
            pend_v = 1;
            pph_v = ph_v;
        }
        if (go && warp < A3_HELP_WARP) {
            const int quarter = warp & 3, half = warp >> 2;
            const int row = quarter * 32 + lane;
            const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
            const int nch = ns >> 4, csplit = (nch + 1) >> 1;
            const int c0 = half ? csplit : 0, c1 = half ? nch : csplit;
            const int T = p.T;
            float m = -INFINITY;
            for (int c = c0; c < c1; ++c) {
                uint32_t v[16];
                ptx::tmem_ld_32x32b_x16(tl + c * 16, v);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    if (c * 16 + e < T) m = fmaxf(m, __uint_as_float(v[e]));
            }
            sMx[half * A3_ROWS + row] = m;
            ptx::named_bar_sync(1 + quarter, 64);   // both halves of this lane quarter
            m = fmaxf(m, sMx[(half ^ 1) * A3_ROWS + row]);
            const float ms = m * p.sl2;
            float l = 0.f;
            for (int c = c0; c < c1; ++c) {
                uint32_t v[16], pl[16];
                ptx::tmem_ld_32x32b_x16(tl + c * 16, v);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float pe = c * 16 + e < T ? exp2_approx(fmaf(__uint_as_float(v[e]), p.sl2, -ms)) : 0.f;
                    l += pe;
                    v[e] = __float_as_uint(pe);
                    pl[e] = __float_as_uint(tf32_lo(pe));
                }
                ptx::tmem_st_32x32b_x16(tl + c * 16, v);
                ptx::tmem_st_32x32b_x16(tl + A3_TMEM_PL + c * 16, pl);
            }
            sL[half * A3_ROWS + row] = l;
            ptx::tmem_st_wait();
        } else if (go) {
            // V^T and V^T_lo: a warp task is 32 keys x 16 head columns; lane = (key
            // group of 4, column group of 4); 4 x 4 blocks transposed in registers
            if (!ptx::mbar_wait_bounded(&bars->v_full, ph_v, abort_flag)) {
                fail(ERRBIT_TIMEOUT_ATTENTION);
            } else {
                const int kg = lane & 7, dg = lane >> 3;
                const int nkb = (ns + 31) >> 5, ntask = nkb * 4;
                for (int task = warp - A3_HELP_WARP; task < ntask; task += A3_THREADS / 32 - A3_HELP_WARP) {
                    const int kb = task >> 2, d0 = (task & 3) * 16 + dg * 4;
                    const uint8_t* vbox = smem + A3_OFF_Q + (d0 >> 5) * A3_KBOX;
                    const int cc = (d0 & 31) >> 2;   // 16-byte unit of these 4 columns in a raw row
                    float4 x[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = kb * 32 + kg * 4 + i;
                        x[i] = r < ns ? *reinterpret_cast<const float4*>(vbox + r * 128 + ((cc ^ (r & 7)) << 4))
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                    const float col[4][4] = {{x[0].x, x[1].x, x[2].x, x[3].x}, {x[0].y, x[1].y, x[2].y, x[3].y},
                                             {x[0].z, x[1].z, x[2].z, x[3].z}, {x[0].w, x[1].w, x[2].w, x[3].w}};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int d = d0 + j;
                        const int off = kb * A3_VTBLK + d * 128 + ((kg ^ (d & 7)) << 4);
                        const float4 w = make_float4(col[j][0], col[j][1], col[j][2], col[j][3]);
                        *reinterpret_cast<float4*>(smem + A3_OFF_VT + off) = w;
                        *reinterpret_cast<float4*>(smem + A3_OFF_VTL + off) = tf32_lo4(w);
                    }
                }
                ptx::fence_proxy_async_smem();
            }
        }
        ph_v ^= 1;
        ptx::tc_fence_before();
        __syncthreads();
        if (loader && !*abort_flag) pend_v = 0;   // the helper warps saw it land

        // ---- 4. O = P V; the next Q in -------------------------------------------------
        const bool go2 = !*abort_flag;
        if (go2 && loader && unext >= 0) {
            load_q(unext);   // raw V has been read
            pend_q = 1;
            pph_q = ph_q;
        }
        if (go2 && issuer) {
            ptx::tc_fence_after();
            constexpr uint32_t idO = a3_idesc(A3_ROWS, A3_DH);
            const uint64_t dv = ptx::smem_desc(ptx::smem_addr(smem + A3_OFF_VT), 16, 1024, ptx::kLayoutSw128);
            const uint64_t dvl = ptx::smem_desc(ptx::smem_addr(smem + A3_OFF_VTL), 16, 1024, ptx::kLayoutSw128);
            const int ksteps = ns >> 3;
            for (int ks = 0; ks < ksteps; ++ks) {
                const uint64_t vo = (uint64_t)((ks >> 2) * (A3_VTBLK >> 4) + (ks & 3) * 2);
                const uint32_t pa = tmem + (uint32_t)(ks * 8);
                mma_tf32_ts(tmem + A3_TMEM_O, pa, dv + vo, idO, ks > 0 ? 1u : 0u);
                mma_tf32_ts(tmem + A3_TMEM_O, pa, dvl + vo, idO, 1u);
                mma_tf32_ts(tmem + A3_TMEM_O, pa + A3_TMEM_PL, dv + vo, idO, 1u);
            }
            ptx::mma_commit(&bars->o_done);
        }

        // ---- 5. O out (warps 8-11); the next K in ------------------------------------
        if (go2) {
            if (!ptx::mbar_wait_bounded(&bars->o_done, ph_o, abort_flag)) fail(ERRBIT_TIMEOUT_ATTENTION);
            ph_o ^= 1;
        }
        ptx::tc_fence_after();
        if (go2 && !*abort_flag && loader && unext >= 0) {
            load_k(unext);   // the P.V MMAs have read V^T
            pend_k = 1;
            pph_k = ph_k;
        }
        if (go2 && warp >= A3_HELP_WARP && warp < A3_HELP_WARP + 4) {
            const int quarter = warp & 3;
            const int row = quarter * 32 + lane;
            const int t = qt * A3_ROWS + row;
            if (qt * A3_ROWS + quarter * 32 < p.T && !*abort_flag) {
                uint32_t ov[64];
                const uint32_t to = tmem + A3_TMEM_O + ((uint32_t)(quarter * 32) << 16);
                ptx::tmem_ld_32x32b_x32(to, *reinterpret_cast<uint32_t(*)[32]>(&ov[0]));
                ptx::tmem_ld_32x32b_x32(to + 32, *reinterpret_cast<uint32_t(*)[32]>(&ov[32]));
                ptx::tmem_ld_wait();
                // O / l through two 32 x 32 staging tiles (128-byte rows, 16-byte unit u of
                // row r at u ^ (r % 8)) to TMA stores over (column, token, sequence): rows
                // past T lie outside the tensor and are not written. With p.lo the same tiles
                // then carry the low parts to a second pair of stores.
                const float inv = t < p.T ? 1.f / (sL[row] + sL[A3_ROWS + row]) : 0.f;
                uint8_t* stg = smem + A3_OFF_STG + (warp - A3_HELP_WARP) * 2 * A3_STG;
                const int col0 = h * A3_DH, t0 = qt * A3_ROWS + quarter * 32;
                if (lane == 0) ptx::bulk_wait_group_read<0>();   // the previous unit's stores have read the tiles
                __syncwarp();
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    uint8_t* srow = stg + b * A3_STG + lane * 128;
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        const int c = 8 * b + u;
                        *reinterpret_cast<float4*>(srow + ((u ^ (lane & 7)) << 4)) =
                            make_float4(__uint_as_float(ov[4 * c]) * inv, __uint_as_float(ov[4 * c + 1]) * inv,
                                        __uint_as_float(ov[4 * c + 2]) * inv, __uint_as_float(ov[4 * c + 3]) * inv);
                    }
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ptx::tma_store_3d(&tmO, stg, col0, t0, n);
                    ptx::tma_store_3d(&tmO, stg + A3_STG, col0 + 32, t0, n);
                    ptx::bulk_commit_group();
                }
                if (p.lo) {
                    if (lane == 0) ptx::bulk_wait_group_read<0>();
                    __syncwarp();
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        uint8_t* srow = stg + b * A3_STG + lane * 128;
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int c = 8 * b + u;
                            *reinterpret_cast<float4*>(srow + ((u ^ (lane & 7)) << 4)) = make_float4(
                                tf32_lo(__uint_as_float(ov[4 * c]) * inv), tf32_lo(__uint_as_float(ov[4 * c + 1]) * inv),
                                tf32_lo(__uint_as_float(ov[4 * c + 2]) * inv), tf32_lo(__uint_as_float(ov[4 * c + 3]) * inv));
                        }
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_3d(&tmOlo, stg, col0, t0, n);
                        ptx::tma_store_3d(&tmOlo, stg + A3_STG, col0 + 32, t0, n);
                        ptx::bulk_commit_group();
                    }
                }
            }
        }
        ptx::tc_fence_before();
        __syncthreads();
        if (*abort_flag) break;   // the same value for every thread after the barrier
    }

    // teardown: every MMA issued has finished, every copy issued has landed and every
    // store issued has completed
    if (warp >= A3_HELP_WARP && warp < A3_HELP_WARP + 4 && lane == 0) ptx::bulk_wait_group<0>();
    if (issuer) {
        ptx::mma_commit(&bars->fin);
        if (!ptx::mbar_wait_bounded(&bars->fin, 0, nullptr)) a3_error(p.err, ERRBIT_TIMEOUT_TEARDOWN);
    }
    if (loader) {
        if (pend_q && !ptx::mbar_wait_bounded(&bars->q_full, pph_q, nullptr)) a3_error(p.err, ERRBIT_TIMEOUT_TEARDOWN);
        if (pend_k && !ptx::mbar_wait_bounded(&bars->k_full, pph_k, nullptr)) a3_error(p.err, ERRBIT_TIMEOUT_TEARDOWN);
        if (pend_v && !ptx::mbar_wait_bounded(&bars->v_full, pph_v, nullptr)) a3_error(p.err, ERRBIT_TIMEOUT_TEARDOWN);
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == A3_MMA_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn a3_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* q = nullptr;
        cudaDriverEntryPointQueryResult r;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault,
                                             &r) == cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(q);
    });
    return fn;
}

}  // namespace

// VIT_ATTN_F32_TC=0 keeps these shapes on the CUDA-core kernel.
bool attention_tf32_supported(int64_t N, int64_t T, int64_t D, int64_t H, const void* qkv, const void* o) {
    if (H <= 0 || D % H != 0 || D / H != A3_DH || T < 1 || T > A3_MAX_KEYS || N < 1) return false;
    if ((reinterpret_cast<uintptr_t>(qkv) & 15) || (reinterpret_cast<uintptr_t>(o) & 15)) return false;
    if (N * H * 2 > 0x7fffffff || 3 * D > 0x7fffffff) return false;
    static const bool off = [] {
        const char* e = std::getenv("VIT_ATTN_F32_TC");
        return e && e[0] == '0';
    }();
    return !off && a3_encode_fn() != nullptr;
}

cudaError_t launch_attention_tf32(const void* qkv, void* o, int64_t N, int64_t T, int64_t D, int64_t H,
                                  const DeviceInfo& dev, cudaStream_t s, float* o_lo) {
    if (N <= 0 || T <= 0) return cudaSuccess;
    if (!attention_tf32_supported(N, T, D, H, qkv, o)) return cudaErrorInvalidValue;
    if (o_lo && (reinterpret_cast<uintptr_t>(o_lo) & 15)) return cudaErrorInvalidValue;
    EncodeTiledFn fn = a3_encode_fn();
    const int ns = (int)((T + 15) / 16 * 16);
    alignas(64) CUtensorMap tq, tkv;
    cuuint64_t dims[3] = {(cuuint64_t)(3 * D), (cuuint64_t)T, (cuuint64_t)N};
    cuuint64_t strides[2] = {(cuuint64_t)(3 * D * 4), (cuuint64_t)(T * 3 * D * 4)};
    cuuint32_t estr[3] = {1, 1, 1};
    cuuint32_t bq[3] = {32, A3_ROWS, 1}, bkv[3] = {32, (cuuint32_t)ns, 1};
    if (fn(&tq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(qkv), dims, strides, bq, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        fn(&tkv, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(qkv), dims, strides, bkv, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // o and o_lo over (column, token, sequence), box 32 x 32 x 1 (128-byte rows), for stores
    alignas(64) CUtensorMap to, tol;
    cuuint64_t odims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)N};
    cuuint64_t ostr[2] = {(cuuint64_t)(D * 4), (cuuint64_t)(T * D * 4)};
    cuuint32_t obox[3] = {32, 32, 1};
    if (fn(&to, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, o, odims, ostr, obox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
            CUDA_SUCCESS ||
        fn(&tol, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, o_lo ? static_cast<void*>(o_lo) : o, odims, ostr, obox, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    A3Params p;
    p.T = (int)T;
    p.D = (int)D;
    p.H = (int)H;
    p.ns = ns;
    p.nq = (int)((T + A3_ROWS - 1) / A3_ROWS);
    p.units = (int)(N * H * p.nq);
    p.sl2 = 1.4426950408889634f / 8.0f;   // log2(e) / sqrt(64)
    p.o = static_cast<float*>(o);
    p.lo = o_lo != nullptr;
    p.err = dev.err_word;
    static std::atomic<uint64_t> attr{0};
    cudaError_t ae = set_smem_limit_once(attention_tf32_kernel, A3_SMEM, attr);
    if (ae != cudaSuccess) return ae;
    const int grid = p.units < dev.num_sms ? p.units : dev.num_sms;
    return launch_dependent(attention_tf32_kernel, dim3(grid), dim3(A3_THREADS), A3_SMEM, s, tq, tkv, to, tol, p);
}

}  // namespace vit
