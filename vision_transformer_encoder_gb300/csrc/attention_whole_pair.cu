// attention_whole_pair.cu -- bidirectional multi-head attention for head width 64 and at
// most 224 tokens per sequence, on CTA pairs (tcgen05 cta_group::2).
//
// "ViT Encoder Block" (crackedaicode), "Multi-head attention": per sequence n and head
// h, out_h = softmax(Q_h K_h^T / sqrt(D/H)) V_h with every key visible; heads written
// side by side in order, Q, K and V read in place from the fused (N, T, 3D) buffer.
//
// The mathematics and the softmax are those of the single-CTA whole-row kernel: with
// T <= 224 all keys of a query row fit in one S tile (ns = T rounded up to 16 columns),
// so the row maximum is known before any exponent and the softmax is one exact pass.
// What changes is who runs the MMAs. An item is one (sequence, head); the two CTAs of a
// cluster (one TPC's two SMs) take its two 128-row query tiles -- CTA r owns query rows
// [128 r, 128 r + 128) -- and every MMA is a pair MMA (M 256), which runs at twice the
// per-SM rate of the single-CTA M 128 form and halves the MMA time of the S -> softmax ->
// P.V chain:
//   S = Q K^T   A = each CTA's Q tile, B = K with its ns keys split ns/2 + ns/2 between
//               the CTAs' shared memory, D = each CTA's 128 rows x ns columns of TMEM.
//   O = P V     A = P from each CTA's TMEM, B = V with its 64 columns split 32 + 32
//               (64-byte swizzle), D = each CTA's 128 rows x 64 columns of TMEM.
// Warps of each CTA (768 threads):
//   0-7 / 8-15  softmax of the even / odd items of the pair ("groups"), as in the
//               single-CTA kernel: two warps per TMEM lane quarter split the keys, pass 1
//               takes the row maximum, pass 2 writes bf16 P over the consumed S columns.
//   16-19       epilogue: O into registers, the O slot released, O / l to global memory.
//   20          TMEM (pair allocation); in the even CTA also the MMA issuer. MMA stream:
//               S(0), S(1), PV(0), S(2), PV(1), ...
//   21-23       TMA loads of Q, K and V, double-buffered per item; the loads of
//               both CTAs complete on the even CTA's barriers.
// The MMA issuer waits on barriers in the even CTA only: the odd CTA's softmax and
// epilogue warps gather on a local barrier and one thread forwards a single arrive (a
// cluster-scope arrive costs far more than a local one).
// TMEM of each CTA, 512 columns: S / P of group 0 at [0, 224), of group 1 at [224, 448),
// O at [448, 512). Every wait is bounded; on expiry the kernel records an error bit and
// unwinds.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace vit {
namespace {

constexpr int WP_DH = 64;
constexpr int WP_ROWS = 128;                // query rows per CTA (TMEM lanes)
constexpr int WP_MAX_KEYS = 224;            // S columns per group
constexpr int WP_THREADS = 768;             // 24 warps
constexpr int WP_EPI_WARP = 16, WP_MMA_WARP = 20, WP_LOAD_WARP = 21;
constexpr int WP_Q_BYTES = WP_ROWS * 128;           // 128 rows x 64 columns, 128B swizzle
constexpr int WP_K_BYTES = (WP_MAX_KEYS / 2) * 128; // up to 112 keys x 64 columns
constexpr int WP_V_BYTES = WP_MAX_KEYS * 64;        // up to 224 keys x 32 columns, 64B swizzle
constexpr int WP_NBUF = 2;                                    // Q / K / V buffers (items ahead)
constexpr int WP_OFF_Q = 0;                                   // [buffer]
constexpr int WP_OFF_K = WP_OFF_Q + WP_NBUF * WP_Q_BYTES;     // [buffer]
constexpr int WP_OFF_V = WP_OFF_K + WP_NBUF * 16384;          // [buffer], 1 KB aligned
constexpr int WP_OFF_L = WP_OFF_V + WP_NBUF * 16384;          // row sums [item % 4][half][row]
constexpr int WP_OFF_MX = WP_OFF_L + 4 * 2 * WP_ROWS * 4;     // row maxima [group][half][row]
constexpr int WP_OFF_BAR = WP_OFF_MX + 2 * 2 * WP_ROWS * 4;
constexpr int WP_SMEM = WP_OFF_BAR + 512 + 1024;              // + alignment slack
constexpr uint32_t WP_TMEM_O = 448;
static_assert(WP_K_BYTES <= 16384 && WP_V_BYTES <= 16384, "K / V buffers");

struct WpParams {
    int T, D, H;
    int ns;        // S columns: T rounded up to 16
    int split;     // keys of softmax half 0: a multiple of 32
    int items;     // N * H
    float scale_log2;
    __nv_bfloat16* o;
    uint32_t* err;
};

struct WpBars {
    // in the even CTA: loads of both CTAs, P and O hand-offs of both CTAs
    uint64_t q_full[WP_NBUF], k_full[WP_NBUF], v_full[WP_NBUF];
    uint64_t p_full[2], o_free;
    // in each CTA
    uint64_t q_empty[WP_NBUF], k_empty[WP_NBUF], v_empty[WP_NBUF];
    uint64_t s_full[2], o_done, l_full[4];
    uint64_t mx_full[2][4];   // [group][lane quarter]: both halves' maxima written
    uint64_t p_gather[2], o_gather;
    uint64_t done;
    uint32_t tmem_slot;
    int abort_flag;
};
static_assert(sizeof(WpBars) <= 512, "barrier block");
static_assert(WP_SMEM <= 227 * 1024, "shared memory");

__device__ __forceinline__ void wp_error(uint32_t* err, uint32_t bit) {
    if (err) atomicOr(err, bit);
}

template <int W>
__device__ __forceinline__ void wp_mask_tail(uint32_t (&v)[W], int lim) {
    if (lim < W) {
#pragma unroll
        for (int e = 0; e < W; ++e)
            if (e >= lim) v[e] = __float_as_uint(-INFINITY);
    }
}

template <int W>
__device__ __forceinline__ float wp_chunk_max(const uint32_t (&v)[W], float m) {
    float a[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) a[e] = __uint_as_float(v[e]);
#pragma unroll
    for (int e = 8; e < W; ++e) a[e & 7] = fmaxf(a[e & 7], __uint_as_float(v[e]));
    return fmaxf(m, fmaxf(fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3])), fmaxf(fmaxf(a[4], a[5]), fmaxf(a[6], a[7]))));
}

template <int W>
__device__ __forceinline__ void wp_chunk_exp(const uint32_t (&v)[W], float sl2, float m, uint32_t (&pk)[W / 2],
                                   unsigned long long (&ls)[4]) {
    // exponent arguments and the row sums in packed fp32 pairs: half the instructions
    const unsigned long long s2 = f2_pack(sl2, sl2), nm = f2_pack(-m, -m);
#pragma unroll
    for (int e = 0; e < W; e += 2) {
        float x0, x1;
        f2_unpack(f2_fma(f2_pack(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), s2, nm), x0, x1);
        const float p0 = exp2_approx(x0);
        const float p1 = exp2_approx(x1);
        ls[(e >> 1) & 3] = f2_add(ls[(e >> 1) & 3], f2_pack(p0, p1));
        pk[e >> 1] = pack_bf16x2(p0, p1);
    }
}

// Pair MMA with A read from tensor memory (each CTA's lanes) and B from shared memory.
__device__ __forceinline__ void mma_bf16_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(WP_THREADS, 1)
attention_whole_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const WpParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem + WP_OFF_Q;
    uint8_t* sK = smem + WP_OFF_K;
    uint8_t* sV = smem + WP_OFF_V;
    float* sL = reinterpret_cast<float*>(smem + WP_OFF_L);
    float* sMx = reinterpret_cast<float*>(smem + WP_OFF_MX);
    WpBars* bars = reinterpret_cast<WpBars*>(smem + WP_OFF_BAR);
    volatile int* abort_flag = &bars->abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const int n_items = p.items > cluster ? (p.items - 1 - cluster) / nclusters + 1 : 0;
    const int khalf = p.ns >> 1;   // keys of S's B operand in each CTA

    if (threadIdx.x == 0) {
        for (int b = 0; b < WP_NBUF; ++b) {
            ptx::mbar_init(&bars->q_full[b], 1);
            ptx::mbar_init(&bars->k_full[b], 1);
            ptx::mbar_init(&bars->v_full[b], 1);
            ptx::mbar_init(&bars->q_empty[b], 1);
            ptx::mbar_init(&bars->k_empty[b], 1);
            ptx::mbar_init(&bars->v_empty[b], 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&bars->s_full[b], 1);
            ptx::mbar_init(&bars->p_full[b], 2);     // one forwarded arrive per CTA
            ptx::mbar_init(&bars->p_gather[b], 8);   // the eight softmax warps of a group
            for (int q = 0; q < 4; ++q) ptx::mbar_init(&bars->mx_full[b][q], 2);
        }
        for (int i = 0; i < 4; ++i) ptx::mbar_init(&bars->l_full[i], 8);
        ptx::mbar_init(&bars->o_done, 1);
        ptx::mbar_init(&bars->o_free, 2);            // one forwarded arrive per CTA
        ptx::mbar_init(&bars->o_gather, 4);          // the four epilogue warps
        ptx::mbar_init(&bars->done, 1);
        bars->abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == WP_LOAD_WARP && lane == 0) {
        ptx::prefetch_tensormap(&tmQ);
        ptx::prefetch_tensormap(&tmK);
        ptx::prefetch_tensormap(&tmV);
    }
    if (warp == WP_MMA_WARP) {
        ptx::tmem_alloc_pair(&bars->tmem_slot, 512);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();   // barriers of both CTAs exist before any remote arrive
    ptx::tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;

    auto leader = [&](const void* local) {   // shared::cluster address in the even CTA
        return ptx::mapa_shared(ptx::smem_addr(local), 0);
    };

    if (warp >= WP_LOAD_WARP) {
        if (lane == 0) {
            // --------------------------------------------------- TMA producers (both CTAs)
            const int role = warp - WP_LOAD_WARP;   // 0 Q, 1 K, 2 V
            uint64_t* full = role == 0 ? bars->q_full : role == 1 ? bars->k_full : bars->v_full;
            uint64_t* empty = role == 0 ? bars->q_empty : role == 1 ? bars->k_empty : bars->v_empty;
            uint8_t* ring = role == 0 ? sQ : role == 1 ? sK : sV;
            const int ring_bytes = role == 0 ? WP_Q_BYTES : 16384;
            const uint32_t bytes = role == 0 ? WP_Q_BYTES : role == 1 ? (uint32_t)khalf * 128 : (uint32_t)p.ns * 64;
            const CUtensorMap* tm = role == 0 ? &tmQ : role == 1 ? &tmK : &tmV;
            int k = 0;
            bool ok = true;
            for (; k < n_items; ++k) {
                const int item = cluster + k * nclusters;
                const int n = item / p.H, h = item - n * p.H;
                const int b = k % WP_NBUF;
                if (!ptx::mbar_wait_bounded<true>(&empty[b], ((k / WP_NBUF) & 1) ^ 1, abort_flag)) { ok = false; break; }
                if (rank == 0) ptx::mbar_arrive_expect_tx(&full[b], 2 * bytes);
                const uint32_t fb = leader(&full[b]);
                if (role == 0)
                    ptx::tma_load_3d_pair(ring + b * ring_bytes, tm, fb, h * WP_DH, (int)rank * WP_ROWS, n);
                else if (role == 1)
                    ptx::tma_load_3d_pair(ring + b * ring_bytes, tm, fb, p.D + h * WP_DH, (int)rank * khalf, n);
                else
                    ptx::tma_load_3d_pair(ring + b * ring_bytes, tm, fb, 2 * p.D + h * WP_DH + (int)rank * 32, 0, n);
            }
            if (!ok) {
                wp_error(p.err, ERRBIT_TIMEOUT_ATTENTION);
                *abort_flag = 1;
            }
            // let the copies in flight (of both CTAs) land before the pair can exit
            if (rank == 0)
                for (int b = 0; b < WP_NBUF; ++b)
                    if (k > b && !ptx::mbar_wait_bounded(&full[b], ((k - 1 - b) / WP_NBUF) & 1, nullptr))
                        wp_error(p.err, ERRBIT_TIMEOUT_TEARDOWN);
        }
    } else if (warp == WP_MMA_WARP) {
        if (lane == 0 && rank == 0) {
            // ------------------------------------------------------ pair MMA issuer
            const uint32_t idS = ptx::idesc_bf16_f32(2 * WP_ROWS, p.ns, false, false);
            constexpr uint32_t idO = ptx::idesc_bf16_f32(2 * WP_ROWS, WP_DH, false, true);
            const int ksteps = p.ns >> 4, ksplit = p.split >> 4;
            bool ok = true;
            for (int s = 0; s <= n_items && ok; ++s) {
                if (s < n_items) {
                    // S(s) = Q K^T into the item's S slot
                    const int b = s % WP_NBUF, g = s & 1;
                    if (!ptx::mbar_wait_bounded(&bars->q_full[b], (s / WP_NBUF) & 1, abort_flag) ||
                        !ptx::mbar_wait_bounded(&bars->k_full[b], (s / WP_NBUF) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t qa = ptx::smem_addr(sQ + b * WP_Q_BYTES);
                    const uint32_t ka = ptx::smem_addr(sK + b * 16384);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {   // 64 columns: 128-byte rows, 32 bytes per step
                        const uint64_t ad = ptx::smem_desc(qa + kk * 32, 16, 1024, ptx::kLayoutSw128);
                        const uint64_t bd = ptx::smem_desc(ka + kk * 32, 16, 1024, ptx::kLayoutSw128);
                        ptx::mma_bf16_ss_pair(tmem + g * WP_MAX_KEYS, ad, bd, idS, kk > 0 ? 1u : 0u);
                    }
                    ptx::mma_commit_pair_mc(&bars->s_full[g], 0x3);
                    ptx::mma_commit_pair_mc(&bars->q_empty[b], 0x3);
                    ptx::mma_commit_pair_mc(&bars->k_empty[b], 0x3);
                }
                if (s >= 1) {
                    // PV(s - 1): O = P V, P read from tensor memory
                    const int u = s - 1, b = u % WP_NBUF, g = u & 1;
                    if (!ptx::mbar_wait_bounded(&bars->p_full[g], (u >> 1) & 1, abort_flag) ||
                        !ptx::mbar_wait_bounded(&bars->v_full[b], (u / WP_NBUF) & 1, abort_flag) ||
                        (u >= 1 && !ptx::mbar_wait_bounded(&bars->o_free, (u - 1) & 1, abort_flag))) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t va = ptx::smem_addr(sV + b * 16384);
                    const uint32_t tP = tmem + g * WP_MAX_KEYS;
                    for (int kk = 0; kk < ksteps; ++kk) {
                        // V half: 32 columns = 64-byte rows, 16 keys = 1 KB, 8-row groups 512 B
                        // apart; P: 16 keys = 8 columns of bf16 pairs, half 0's keys from the
                        // slot's first column, half 1's from column `split`
                        const uint64_t bd = ptx::smem_desc(va + kk * 1024, 16, 512, ptx::kLayoutSw64);
                        const uint32_t pa = kk < ksplit ? tP + kk * 8 : tP + p.split + (kk - ksplit) * 8;
                        mma_bf16_ts_pair(tmem + WP_TMEM_O, pa, bd, idO, kk > 0 ? 1u : 0u);
                    }
                    ptx::mma_commit_pair_mc(&bars->o_done, 0x3);
                    ptx::mma_commit_pair_mc(&bars->v_empty[b], 0x3);
                }
            }
            if (!ok) {
                wp_error(p.err, ERRBIT_TIMEOUT_MMA);
                *abort_flag = 1;
            }
            ptx::mma_commit_pair(&bars->done);
            if (!ptx::mbar_wait_bounded(&bars->done, 0, nullptr)) wp_error(p.err, ERRBIT_TIMEOUT_TEARDOWN);
        }
    } else if (warp < WP_EPI_WARP) {
        // ------------------------------------------------------------------- softmax
        const int g = warp >> 3;                // 0: even items, 1: odd items
        const int half = (warp >> 2) & 1;       // which keys of the rows
        const int quarter = warp & 3;           // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;
        const uint32_t tS = tmem + g * WP_MAX_KEYS + ((uint32_t)(quarter * 32) << 16);
        const float sl2 = p.scale_log2;
        const int T = p.T;
        const int c0 = half ? p.split >> 5 : 0, c1 = half ? p.ns >> 5 : p.split >> 5;
        const bool tail = half && (p.ns & 16) != 0;
        const uint32_t pbase = half ? (uint32_t)p.split : 0u;
        float* mx_mine = sMx + (g * 2 + half) * WP_ROWS;
        const float* mx_other = sMx + (g * 2 + (half ^ 1)) * WP_ROWS;
        const bool forwarder = half == 0 && quarter == 0;   // forwards the group's P hand-off
        const uint32_t p_full0 = leader(&bars->p_full[g]);
        // a warp whose 32 query rows all lie past T has no output; it keeps the protocol
        const bool live = (int)rank * WP_ROWS + quarter * 32 < T;
        bool ok = true;
        for (int u = g; u < n_items; u += 2) {
            const uint32_t ph = (uint32_t)(u >> 1) & 1;
            ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(&bars->s_full[g], ph, abort_flag));
            if (!ok) break;
            ptx::tc_fence_after();
            float mx = -INFINITY;
            if (live) {
                // pass 1: maximum over this half's keys < T, one 32-key chunk per TMEM wait
#pragma unroll
                for (int c = 0; c < 7; ++c) {
                    const int cc = c0 + c;
                    if (cc < c1) {
                        uint32_t v0[32];
                        if (T - cc * 32 >= 32) {
                            const float cm = ptx::tmem_ld_red_max_32x32b_x32(tS + cc * 32, v0);
                            ptx::tmem_ld_wait();
                            ptx::regs_keep(v0);
                            mx = fmaxf(mx, cm);
                        } else {
                            ptx::tmem_ld_32x32b_x32(tS + cc * 32, v0);
                            ptx::tmem_ld_wait();
                            wp_mask_tail(v0, T - cc * 32);
                            mx = wp_chunk_max(v0, mx);
                        }
                    }
                }
                if (tail) {
                    uint32_t v0[16];
                    ptx::tmem_ld_32x32b_x16(tS + c1 * 32, v0);
                    ptx::tmem_ld_wait();
                    wp_mask_tail(v0, T - c1 * 32);
                    mx = wp_chunk_max(v0, mx);
                }
                mx_mine[row] = mx;
            }
            // exchange the two halves' maxima
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bars->mx_full[g][quarter]);
            ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(&bars->mx_full[g][quarter], ph, abort_flag));
            if (!ok) break;
            if (live) {
                const float m = fmaxf(mx, mx_other[row]) * sl2;
                // pass 2: P over this half's consumed S columns
                unsigned long long ls[4] = {0ull, 0ull, 0ull, 0ull};   // packed pairs of +0.0f
#pragma unroll
                for (int c = 0; c < 7; ++c) {
                    const int cc = c0 + c;
                    if (cc < c1) {
                        uint32_t v0[32], pk0[16];
                        ptx::tmem_ld_32x32b_x32(tS + cc * 32, v0);
                        ptx::tmem_ld_wait();
                        wp_mask_tail(v0, T - cc * 32);
                        wp_chunk_exp(v0, sl2, m, pk0, ls);
                        ptx::tmem_st_32x32b_x16(tS + pbase + c * 16, pk0);
                    }
                }
                if (tail) {
                    uint32_t v0[16], pk0[8];
                    ptx::tmem_ld_32x32b_x16(tS + c1 * 32, v0);
                    ptx::tmem_ld_wait();
                    wp_mask_tail(v0, T - c1 * 32);
                    wp_chunk_exp(v0, sl2, m, pk0, ls);
                    ptx::tmem_st_32x32b_x8(tS + pbase + (c1 - c0) * 16, pk0);
                }
                ptx::tmem_st_wait();
                sL[((u & 3) * 2 + half) * WP_ROWS + row] = [&] {
                    float a[8];
                    f2_unpack(ls[0], a[0], a[1]);
                    f2_unpack(ls[1], a[2], a[3]);
                    f2_unpack(ls[2], a[4], a[5]);
                    f2_unpack(ls[3], a[6], a[7]);
                    return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
                }();
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(&bars->p_gather[g]);
                ptx::mbar_arrive(&bars->l_full[u & 3]);
            }
            if (forwarder) {
                // all eight warps of the group have written P: one arrive in the even CTA
                ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(&bars->p_gather[g], ph, abort_flag));
                if (!ok) break;
                if (lane == 0) {
                    ptx::tc_fence_before();
                    ptx::mbar_arrive_cluster_relaxed(p_full0);
                }
            }
        }
        if (!ok) {
            if (lane == 0) wp_error(p.err, ERRBIT_TIMEOUT_ATTENTION);
            *abort_flag = 1;
        }
    } else if (warp < WP_MMA_WARP) {
        // ------------------------------------------------------------------ epilogue
        const int quarter = warp & 3;
        const uint32_t tO = tmem + WP_TMEM_O + ((uint32_t)(quarter * 32) << 16);
        const int D = p.D;
        const uint32_t o_free0 = leader(&bars->o_free);
        const int row = quarter * 32 + lane;
        const int t = (int)rank * WP_ROWS + row;   // this thread's query row
        const bool live = (int)rank * WP_ROWS + quarter * 32 < p.T;
        bool ok = true;
        for (int u = 0; u < n_items; ++u) {
            const int item = cluster + u * nclusters;
            const int n = item / p.H, h = item - n * p.H;
            // the row sums are in before O (PV waited for them): take 1 / l first
            ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(&bars->l_full[u & 3], (u >> 2) & 1, abort_flag));
            if (!ok) break;
            const float inv = 1.f / (sL[((u & 3) * 2) * WP_ROWS + row] + sL[((u & 3) * 2 + 1) * WP_ROWS + row]);
            ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(&bars->o_done, u & 1, abort_flag));
            if (!ok) break;
            ptx::tc_fence_after();
            uint32_t ov[64];
            if (live) {
                ptx::tmem_ld_32x32b_x32(tO, *reinterpret_cast<uint32_t(*)[32]>(&ov[0]));
                ptx::tmem_ld_32x32b_x32(tO + 32, *reinterpret_cast<uint32_t(*)[32]>(&ov[32]));
                ptx::tmem_ld_wait();
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bars->o_gather);
            if (quarter == 0) {
                // the four epilogue warps have read O: one arrive in the even CTA
                ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(&bars->o_gather, u & 1, abort_flag));
                if (!ok) break;
                if (lane == 0) ptx::mbar_arrive_cluster_relaxed(o_free0);
            }
            if (live && t < p.T) {
                __nv_bfloat16* orow = p.o + ((int64_t)n * p.T + t) * D + h * WP_DH;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(ov[8 * c + 0]) * inv, __uint_as_float(ov[8 * c + 1]) * inv);
                    w.y = pack_bf16x2(__uint_as_float(ov[8 * c + 2]) * inv, __uint_as_float(ov[8 * c + 3]) * inv);
                    w.z = pack_bf16x2(__uint_as_float(ov[8 * c + 4]) * inv, __uint_as_float(ov[8 * c + 5]) * inv);
                    w.w = pack_bf16x2(__uint_as_float(ov[8 * c + 6]) * inv, __uint_as_float(ov[8 * c + 7]) * inv);
                    *reinterpret_cast<uint4*>(orow + c * 8) = w;
                }
            }
        }
        if (!ok) {
            if (lane == 0) wp_error(p.err, ERRBIT_TIMEOUT_ATTENTION);
            *abort_flag = 1;
        }
    }

    __syncthreads();
    ptx::cluster_sync();   // neither CTA leaves while its peer may still touch its memory
    if (warp == WP_MMA_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem, 512);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn wp_encode_fn() {
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

// Opt-in (VIT_ATTN_WHOLE_PAIR=1): at T = 197 the pair kernel's cross-CTA hand-offs (the
// O slot and P of both CTAs must be released to the even CTA's MMA issuer) cost about what
// its faster MMAs save, and the single-CTA kernel measures 2-3 % faster.
bool attention_whole_pair_supported(int64_t T, int64_t D, int64_t H, const DeviceInfo& dev) {
    if (H <= 0 || D % H != 0 || D / H != WP_DH || T < 1 || T > WP_MAX_KEYS || dev.num_sms < 2) return false;
    static const bool on = [] {
        const char* e = std::getenv("VIT_ATTN_WHOLE_PAIR");
        return e && e[0] == '1';
    }();
    return on && wp_encode_fn() != nullptr;
}

cudaError_t launch_attention_whole_pair(const void* qkv, void* o, int64_t N, int64_t T, int64_t D, int64_t H,
                                        const DeviceInfo& dev, cudaStream_t s) {
    if (N <= 0 || T <= 0) return cudaSuccess;
    if (!attention_whole_pair_supported(T, D, H, dev) || N * H > 0x7fffffff) return cudaErrorInvalidValue;
    EncodeTiledFn fn = wp_encode_fn();
    const int ns = (int)((T + 15) / 16 * 16);
    alignas(64) CUtensorMap tq, tk, tv;
    cuuint64_t dims[3] = {(cuuint64_t)(3 * D), (cuuint64_t)T, (cuuint64_t)N};
    cuuint64_t strides[2] = {(cuuint64_t)(3 * D * 2), (cuuint64_t)(T * 3 * D * 2)};
    cuuint32_t estr[3] = {1, 1, 1};
    cuuint32_t bq[3] = {WP_DH, WP_ROWS, 1}, bk[3] = {WP_DH, (cuuint32_t)(ns / 2), 1}, bv[3] = {32, (cuuint32_t)ns, 1};
    if (fn(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(qkv), dims, strides, bq, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        fn(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(qkv), dims, strides, bk, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        fn(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(qkv), dims, strides, bv, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    WpParams p;
    p.T = (int)T;
    p.D = (int)D;
    p.H = (int)H;
    p.ns = ns;
    p.split = (ns >> 5) / 2 * 32;   // half 0: the first floor(full chunks / 2) chunks
    p.items = (int)(N * H);
    p.scale_log2 = 1.4426950408889634f / 8.0f;   // log2(e) / sqrt(64)
    p.o = static_cast<__nv_bfloat16*>(o);
    p.err = dev.err_word;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(attention_whole_pair_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, WP_SMEM);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const int64_t pairs = p.items < dev.num_sms / 2 ? p.items : dev.num_sms / 2;
    if (pairs < 1) return cudaErrorInvalidValue;
    attention_whole_pair_kernel<<<(unsigned)(2 * pairs), WP_THREADS, WP_SMEM, s>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace vit
