// attention_whole.cu -- bidirectional multi-head attention for head width 64 and at most
// 224 tokens per sequence, on the sm_103a tensor cores (tcgen05 / TMEM / TMA).
//
// "ViT Encoder Block" (crackedaicode), "Multi-head attention": per sequence n and head
// h, out_h = softmax(Q_h K_h^T / sqrt(D/H)) V_h with every key visible; heads written
// side by side in order, Q, K and V read in place from the fused (N, T, 3D) buffer.
//
// With T <= 224, all keys of a query row fit in one S tile: S = Q K^T for 128 query
// rows is a single M 128 x N ns MMA chain (ns = T rounded up to 16), so the row maximum
// is in TMEM before any exponent is taken. The softmax is one pass per row with no
// rescaling of O, and O = P V is one MMA chain over ns keys.
//
// A unit is (sequence, head, 128-row query tile); the units of one (sequence, head)
// item share its K and V. Persistent kernel, one CTA per SM, 24 warps:
//   warps 0-7 / 8-15  softmax of even / odd units. Two warps per TMEM lane quarter
//                    split the keys of their 32 rows: warp "half" 0 takes the first
//                    `split` keys, half 1 the rest. One pass over S: P = exp2(S
//                    log2(e)/sqrt(dh) - r) in bf16, written into the half's own S columns
//                    already consumed (32 keys fill 16 columns), and the half's row sum to
//                    shared memory. Softmax is unchanged by any common offset r; r starts
//                    as the maximum over keys [0, 32), which both halves read, and a half
//                    raises its own r, by whole log2 units, only when a chunk's maximum
//                    passes r by more than 8 (so P <= 2^8); the P it has written is then
//                    rescaled by an exact power of two. At the end the two halves take the
//                    larger of their offsets (a named barrier per quarter; a warp whose
//                    wait fails still passes it for each remaining unit, as its partner
//                    does, so it never waits for a warp that has left); the one below
//                    rescales. With typical scores no chunk passes the start by 8 and the
//                    row costs one read of S, each P rounded once.
//   warps 16-19      epilogue, one per TMEM lane quarter: O into registers, O's slot
//                    released at once, then O / (l0 + l1) in bf16 through a swizzled
//                    staging tile to one TMA store per warp and unit.
//   warps 20, 21     MMA issuers, one per group (warp 20 also owns TMEM): group g's
//                    stream is S(g), PV(g), S(g + 2), PV(g + 2), ...: S of a unit runs
//                    while the other group's softmax works, and PV(u) follows as soon as
//                    P(u) is in. (One thread issues an MMA only every ~120 cycles while
//                    the softmax warps move tensor memory: one issuer for both groups
//                    reached each P late.) PV reads P of keys below `split` from the
//                    slot's first columns and P of the rest from the columns from `split`.
//   warps 22, 23     TMA loads: Q then K of each item (warp 22), V (warp 23); one issuing
//                    thread per stream, as a thread's TMA copies go one after another.
//                    Each is double-buffered per item; a 3-D tensor map (column, token,
//                    sequence) zero-fills tokens past T.
// TMEM, 512 columns: S / P of even units at [0, 224), of odd units at [224, 448), O at
// [448, 512). S(u + 2) overwrites P(u) only after PV(u) in the same in-order MMA stream.
// Every wait is bounded; on expiry the kernel records an error bit and unwinds.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "ptx.cuh"

namespace vit {
namespace {

constexpr int AW_DH = 64;
constexpr int AW_ROWS = 128;               // query rows per unit (TMEM lanes)
constexpr int AW_MAX_KEYS = 224;           // S columns per unit
constexpr int AW_THREADS = 768;            // 24 warps
constexpr int AW_EPI_WARP = 16, AW_MMA_WARP = 20, AW_LOAD_WARP = 22;   // MMA: warps 20, 21
constexpr int AW_BOX = AW_ROWS * 128;      // 128 rows x 64 bf16 columns, 128B swizzle: 16 KB
constexpr int AW_OFF_Q = 0;                        // [buffer][query tile]
constexpr int AW_OFF_K = AW_OFF_Q + 4 * AW_BOX;    // [buffer][128-key box]
constexpr int AW_OFF_V = AW_OFF_K + 4 * AW_BOX;    // [buffer][128-key box]
constexpr int AW_OFF_L = AW_OFF_V + 4 * AW_BOX;    // row sums [unit % 4][half][row]
constexpr int AW_OFF_MX = AW_OFF_L + 4 * 2 * AW_ROWS * 4;   // row maxima [group][half][row]
constexpr int AW_OFF_BAR = AW_OFF_MX + 2 * 2 * AW_ROWS * 4;
constexpr int AW_STG = 32 * 128;                   // one 32-row x 64-column bf16 staging tile
constexpr int AW_OFF_STG = (AW_OFF_BAR + 256 + 1023) / 1024 * 1024;   // [epilogue warp]
constexpr int AW_SMEM = AW_OFF_STG + 4 * AW_STG + 1024;               // + alignment slack
static_assert(AW_SMEM <= 227 * 1024, "shared memory");
constexpr uint32_t AW_TMEM_O = 448;

struct AwParams {
    int T, D, H;
    int nq;        // query tiles per item: 1 or 2
    int nkb;       // 128-key boxes per item: 1 or 2
    int ns;        // S columns: T rounded up to 16
    int split;     // keys of softmax half 0: a multiple of 32
    int items;     // N * H
    float scale_log2;
    __nv_bfloat16* o;
    uint32_t* err;
};

struct AwBars {
    uint64_t q_full[2], q_empty[2], k_full[2], k_empty[2], v_full[2], v_empty[2];
    uint64_t s_full[2], p_full[2], l_full[4];
    uint64_t o_done, o_free[2], done;   // o_free[u & 1]: the epilogue has read O(u)
    uint32_t tmem_slot;
    int abort_flag;
};
static_assert(sizeof(AwBars) <= 256, "barrier block");
static_assert(AW_SMEM <= 227 * 1024, "shared memory");

__device__ __forceinline__ void aw_error(uint32_t* err, uint32_t bit) {
    if (err) atomicOr(err, bit);
}

// Masks keys at or past `lim` (chunk-relative) to -inf.
template <int W>
__device__ __forceinline__ void mask_tail(uint32_t (&v)[W], int lim) {
    if (lim < W) {
#pragma unroll
        for (int e = 0; e < W; ++e)
            if (e >= lim) v[e] = __float_as_uint(-INFINITY);
    }
}

// Eight independent chains: the reductions are latency-bound otherwise.
template <int W>
__device__ __forceinline__ float chunk_max(const uint32_t (&v)[W], float m) {
    float a[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) a[e] = __uint_as_float(v[e]);
#pragma unroll
    for (int e = 8; e < W; ++e) a[e & 7] = fmaxf(a[e & 7], __uint_as_float(v[e]));
    return fmaxf(m, fmaxf(fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3])), fmaxf(fmaxf(a[4], a[5]), fmaxf(a[6], a[7]))));
}

// P for W keys: W / 2 packed bf16 pairs, added to the eight partial row sums ls.
template <int W>
__device__ __forceinline__ void chunk_exp(const uint32_t (&v)[W], float sl2, float m, uint32_t (&pk)[W / 2],
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

// An offset is raised only when a chunk's maximum passes it by more than this (log2
// units), so P stays at most 2^kRaise and is seldom rescaled.
constexpr float kRaise = 8.f;

// 2^k for an integer-valued k <= 0, exactly (0 below the normal range).
__device__ __forceinline__ float pow2_int(float k) {
    return k < -126.f ? 0.f : __int_as_float(((int)k + 127) << 23);
}

__device__ __forceinline__ void f2_scale(unsigned long long (&ls)[4], float f) {
    const unsigned long long ff = f2_pack(f, f);
#pragma unroll
    for (int i = 0; i < 4; ++i) ls[i] = f2_mul(ls[i], ff);
}

// Multiplies the bf16 P this thread's half has written -- `full` 16-column chunks from
// tP on, then 8 columns if `tail` -- by f, a power of two <= 1 (exact but for values
// pushed below the normal range). Rare: only when an offset changes.
__device__ __noinline__ void rescale_p(uint32_t tP, int full, bool tail, float f) {
    ptx::tmem_st_wait();   // the P stores being read back have landed
    for (int i = 0; i < full; ++i) {
        uint32_t r[16];
        ptx::tmem_ld_32x32b_x16(tP + i * 16, r);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const float2 a = unpack_bf16x2(r[e]);
            r[e] = pack_bf16x2(a.x * f, a.y * f);
        }
        ptx::tmem_st_32x32b_x16(tP + i * 16, r);
    }
    if (tail) {
        uint32_t r[8];
        ptx::tmem_ld_32x32b_x8(tP + full * 16, r);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float2 a = unpack_bf16x2(r[e]);
            r[e] = pack_bf16x2(a.x * f, a.y * f);
        }
        ptx::tmem_st_32x32b_x8(tP + full * 16, r);
    }
}

// P of W keys (maximum cm, masked keys at -inf) for chunk j of this half: if cm sl2
// passes the offset by more than kRaise, raises the offset by the whole number of log2
// units that brings it to cm sl2 or above (the partial row sums and, after this chunk,
// the P already written are scaled by the exact power of two), then writes
// exp2(s sl2 - mrun) in bf16 to the W / 2 columns from tP + 16 j.
template <int W>
__device__ __forceinline__ void p_chunk(const uint32_t (&v)[W], float cm, float sl2, float& mrun,
                                        unsigned long long (&ls)[4], uint32_t tP, int j) {
    const float cms = cm * sl2;
    const bool up = cms > mrun + kRaise;
    const bool any_up = __any_sync(0xffffffffu, up);
    float f = 1.f;
    if (any_up) {
        const float n = up ? ceilf(cms - mrun) : 0.f;
        f = pow2_int(-n);
        f2_scale(ls, f);
        mrun += n;
    }
    {
        uint32_t pk[W / 2];
        chunk_exp(v, sl2, mrun, pk, ls);
        if constexpr (W == 32)
            ptx::tmem_st_32x32b_x16(tP + j * 16, pk);
        else
            ptx::tmem_st_32x32b_x8(tP + j * 16, pk);
    }
    // the chunks written under the old offset, once this chunk's values are no longer live
    if (any_up) rescale_p(tP, j, false, f);
}

__global__ void __launch_bounds__(AW_THREADS, 1)
attention_whole_kernel(const __grid_constant__ CUtensorMap tm, const __grid_constant__ CUtensorMap tmO,
                       const AwParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem + AW_OFF_Q;
    uint8_t* sK = smem + AW_OFF_K;
    uint8_t* sV = smem + AW_OFF_V;
    float* sL = reinterpret_cast<float*>(smem + AW_OFF_L);
    float* sMx = reinterpret_cast<float*>(smem + AW_OFF_MX);
    AwBars* bars = reinterpret_cast<AwBars*>(smem + AW_OFF_BAR);
    volatile int* abort_flag = &bars->abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nq = p.nq;
    const int n_items = p.items > (int)blockIdx.x ? (p.items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int units = n_items * nq;

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&bars->q_full[b], 1);
            ptx::mbar_init(&bars->q_empty[b], 2);    // both MMA issuers
            ptx::mbar_init(&bars->k_full[b], 1);
            ptx::mbar_init(&bars->k_empty[b], 2);
            ptx::mbar_init(&bars->v_full[b], 1);
            ptx::mbar_init(&bars->v_empty[b], 2);
            ptx::mbar_init(&bars->s_full[b], 1);
            ptx::mbar_init(&bars->p_full[b], 8);     // the eight softmax warps of a group
        }
        for (int i = 0; i < 4; ++i) ptx::mbar_init(&bars->l_full[i], 8);
        ptx::mbar_init(&bars->o_done, 1);
        ptx::mbar_init(&bars->o_free[0], 4);         // the four epilogue warps
        ptx::mbar_init(&bars->o_free[1], 4);
        ptx::mbar_init(&bars->done, 2);
        bars->abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == AW_LOAD_WARP && lane == 0) ptx::prefetch_tensormap(&tm);
    if (warp == AW_MMA_WARP) {
        ptx::tmem_alloc(&bars->tmem_slot, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;
    // the set-up above overlaps the previous kernel's tail; Q, K and V are its output
    griddep_wait();
    griddep_launch_dependents();

    if (warp >= AW_LOAD_WARP) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producers
            // (one issuing thread per stream, as a thread's copies go one after another):
            // warp 22 each item's query tiles, then its keys; warp 23 its values
            const bool qk = warp == AW_LOAD_WARP;
            int issued[3] = {0, 0, 0};   // items whose copies each stream has issued
            bool ok = true;
            for (int k = 0; k < n_items && ok; ++k) {
                const int item = (int)blockIdx.x + k * (int)gridDim.x;
                const int n = item / p.H, h = item - n * p.H;
                const int b = k & 1;
                for (int role = qk ? 0 : 2; role <= (qk ? 1 : 2) && ok; ++role) {   // 0 Q, 1 K, 2 V
                    uint64_t* full = role == 0 ? bars->q_full : role == 1 ? bars->k_full : bars->v_full;
                    uint64_t* empty = role == 0 ? bars->q_empty : role == 1 ? bars->k_empty : bars->v_empty;
                    uint8_t* ring = role == 0 ? sQ : role == 1 ? sK : sV;
                    const int boxes = role == 0 ? nq : p.nkb;
                    if (!ptx::mbar_wait_bounded<true>(&empty[b], ((k >> 1) & 1) ^ 1, abort_flag)) { ok = false; break; }
                    ptx::mbar_arrive_expect_tx(&full[b], boxes * AW_BOX);
                    for (int r = 0; r < boxes; ++r)   // Q at column 0, K at D, V at 2D
                        ptx::tma_load_3d(ring + (b * 2 + r) * AW_BOX, &tm, &full[b], role * p.D + h * AW_DH,
                                         r * AW_ROWS, n);
                    issued[role] = k + 1;
                }
            }
            if (!ok) {
                aw_error(p.err, ERRBIT_TIMEOUT_ATTENTION);
                *abort_flag = 1;
            }
            // let the copies in flight land before the CTA can exit
            for (int role = qk ? 0 : 2; role <= (qk ? 1 : 2); ++role) {
                uint64_t* full = role == 0 ? bars->q_full : role == 1 ? bars->k_full : bars->v_full;
                const int kk = issued[role];
                for (int b = 0; b < 2; ++b)
                    if (kk > b && !ptx::mbar_wait_bounded(&full[b], ((kk - 1 - b) >> 1) & 1, nullptr))
                        aw_error(p.err, ERRBIT_TIMEOUT_TEARDOWN);
            }
        }
    } else if (warp >= AW_MMA_WARP) {
        if (lane == 0) {
            // --------------------------------------- MMA issuers, one per softmax group
            // (warp 20: units 0, 2, 4, ...; warp 21: units 1, 3, 5, ...). One thread issues an
            // MMA only every ~120 cycles while the softmax warps move tensor memory, so each
            // group's chain S -> P.V gets its own thread. Both use an item's Q, K and V
            // buffers and release each once (their empty barriers count two); with one
            // query tile per item (nq == 1) an issuer releases the other's items too, after
            // their full barriers, so that it never runs a phase ahead.
            const int g = warp - AW_MMA_WARP;
            const uint32_t idS = ptx::idesc_bf16_f32(AW_ROWS, p.ns, false, false);
            constexpr uint32_t idO = ptx::idesc_bf16_f32(AW_ROWS, AW_DH, false, true);
            const int ksteps = p.ns >> 4, ksplit = p.split >> 4;
            bool ok = true;
            for (int k = 0; k < n_items && ok; ++k) {
                const int b = k & 1;
                const uint32_t ph = (uint32_t)(k >> 1) & 1;
                if (nq == 1 && (k & 1) != g) {
                    if (!ptx::mbar_wait_bounded(&bars->q_full[b], ph, abort_flag) ||
                        !ptx::mbar_wait_bounded(&bars->k_full[b], ph, abort_flag) ||
                        !ptx::mbar_wait_bounded(&bars->v_full[b], ph, abort_flag)) {
                        ok = false;
                        break;
                    }
                    ptx::mma_commit(&bars->q_empty[b]);
                    ptx::mma_commit(&bars->k_empty[b]);
                    ptx::mma_commit(&bars->v_empty[b]);
                    continue;
                }
                const int u = nq == 2 ? 2 * k + g : k;   // this issuer's unit of the item
                const int qt = u - k * nq;
                // S(u) = Q K^T into slot g (S(u) follows P.V(u - 2) in this thread's stream,
                // which has read P(u - 2) from the same columns)
                if (!ptx::mbar_wait_bounded(&bars->q_full[b], ph, abort_flag) ||
                    !ptx::mbar_wait_bounded(&bars->k_full[b], ph, abort_flag)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t qa = ptx::smem_addr(sQ + (b * 2 + qt) * AW_BOX);
                const uint32_t ka = ptx::smem_addr(sK + b * 2 * AW_BOX);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {   // 64 columns: 128-byte rows, 32 bytes per step
                    const uint64_t ad = ptx::smem_desc(qa + kk * 32, 16, 1024, ptx::kLayoutSw128);
                    const uint64_t bd = ptx::smem_desc(ka + kk * 32, 16, 1024, ptx::kLayoutSw128);
                    ptx::mma_bf16_ss(tmem + g * AW_MAX_KEYS, ad, bd, idS, kk > 0 ? 1u : 0u);
                }
                ptx::mma_commit(&bars->s_full[g]);
                ptx::mma_commit(&bars->q_empty[b]);
                ptx::mma_commit(&bars->k_empty[b]);
                // P.V(u): O = P V, P read from tensor memory. O is one accumulator for both
                // groups: P.V(u) waits until the epilogue has read O(u - 1), on o_free[(u - 1)
                // & 1], which only the other issuer's units advance: O(u - 3) was read before
                // this thread issued P.V(u - 2), and O(u + 1) cannot be read before P.V(u),
                // so the barrier is within one phase of unit u - 1.
                if (!ptx::mbar_wait_bounded(&bars->p_full[g], (u >> 1) & 1, abort_flag) ||
                    !ptx::mbar_wait_bounded(&bars->v_full[b], ph, abort_flag) ||
                    (u >= 1 && !ptx::mbar_wait_bounded(&bars->o_free[(u - 1) & 1], ((u - 1) >> 1) & 1, abort_flag))) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t va = ptx::smem_addr(sV + b * 2 * AW_BOX);
                const uint32_t tP = tmem + g * AW_MAX_KEYS;
                for (int kk = 0; kk < ksteps; ++kk) {
                    // V: keys are the K dimension (rows of 128 bytes), head columns the
                    // N dimension (MN-major); P: 16 keys = 8 columns of bf16 pairs, at
                    // the start of the slot for half 0's keys, from column `split` on
                    // for half 1's
                    const uint64_t bd = ptx::smem_desc(va + kk * 2048, 16, 1024, ptx::kLayoutSw128);
                    const uint32_t pa = kk < ksplit ? tP + kk * 8 : tP + p.split + (kk - ksplit) * 8;
                    ptx::mma_bf16_ts(tmem + AW_TMEM_O, pa, bd, idO, kk > 0 ? 1u : 0u);
                }
                ptx::mma_commit(&bars->o_done);
                ptx::mma_commit(&bars->v_empty[b]);
            }
            if (!ok) {
                aw_error(p.err, ERRBIT_TIMEOUT_MMA);
                *abort_flag = 1;
            }
            ptx::mma_commit(&bars->done);
            if (!ptx::mbar_wait_bounded(&bars->done, 0, nullptr)) aw_error(p.err, ERRBIT_TIMEOUT_TEARDOWN);
        }
    } else if (warp < AW_EPI_WARP) {
        // ------------------------------------------------------------------- softmax
        const int g = warp >> 3;                // 0: even units, 1: odd units
        const int half = (warp >> 2) & 1;       // which keys of the rows
        const int quarter = warp & 3;           // TMEM lane quarter this warp may access
        const int row = quarter * 32 + lane;
        const uint32_t tS = tmem + g * AW_MAX_KEYS + ((uint32_t)(quarter * 32) << 16);
        const float sl2 = p.scale_log2;
        const int T = p.T;
        // this half's keys: 32-key chunks [c0, c1), then a 16-key tail (half 1 only)
        const int c0 = half ? p.split >> 5 : 0, c1 = half ? p.ns >> 5 : p.split >> 5;
        const bool tail = half && (p.ns & 16) != 0;
        const uint32_t pbase = half ? (uint32_t)p.split : 0u;   // P columns of this half
        float* mx_mine = sMx + (g * 2 + half) * AW_ROWS;
        const float* mx_other = sMx + (g * 2 + (half ^ 1)) * AW_ROWS;
        bool ok = true;
        const uint32_t bar_id = 1 + g * 4 + quarter;   // named barrier of this quarter's two halves
        for (int u = g; u < units; u += 2) {
            const int k = u / nq, qt = u - k * nq;
            ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(&bars->s_full[g], (u >> 1) & 1, abort_flag));
            if (!ok) {
                // The named barrier below waits without limit: pass it for this and every
                // later unit the quarter works on, as the other half does, then leave.
                for (int v = u; v < units; v += 2)
                    if ((v - (v / nq) * nq) * AW_ROWS + quarter * 32 < T) {
                        ptx::named_bar_sync(bar_id, 64);
                        ptx::named_bar_sync(bar_id, 64);
                    }
                break;
            }
            ptx::tc_fence_after();
            // a warp whose 32 query rows all lie past T has no output; it only keeps the
            // barrier protocol (both halves of a lane quarter agree on this)
            const bool live = qt * AW_ROWS + quarter * 32 < T;
            if (live) {
                const uint32_t tP = tS + pbase;                  // this half's P columns
                unsigned long long ls[4] = {0ull, 0ull, 0ull, 0ull};   // packed pairs of +0.0f
                float mrun;        // this half's offset (log2 units): the start + whole steps
                int j = 0;         // 32-key chunks of this half whose P is written
                int cfirst = c0;   // first chunk still to load
                {
                    // the common starting offset: the maximum over keys [0, 32), read by
                    // both halves from the same columns
                    uint32_t vr[32];
                    float cm;
                    if (T >= 32) {
                        cm = ptx::tmem_ld_red_max_32x32b_x32(tS, vr);
                        ptx::tmem_ld_wait();
                    } else {
                        ptx::tmem_ld_32x32b_x32(tS, vr);
                        ptx::tmem_ld_wait();
                        mask_tail(vr, T);
                        cm = chunk_max(vr, -INFINITY);
                    }
                    mrun = cm * sl2;
                    // both halves hold it before P overwrites the columns of keys [0, 32)
                    ptx::named_bar_sync(bar_id, 64);
                    if (c0 == 0 && c1 > 0) {   // this half owns keys [0, 32): no second load
                        p_chunk(vr, cm, sl2, mrun, ls, tP, 0);
                        j = 1;
                        cfirst = 1;
                    } else {
                        ptx::regs_keep(vr);
                    }
                }
#pragma unroll
                for (int c = 0; c < 7; ++c) {
                    const int cc = cfirst + c;
                    if (cc < c1) {
                        uint32_t v0[32];
                        float cm;
                        if (T - cc * 32 >= 32) {
                            cm = ptx::tmem_ld_red_max_32x32b_x32(tS + cc * 32, v0);
                            ptx::tmem_ld_wait();
                        } else {
                            ptx::tmem_ld_32x32b_x32(tS + cc * 32, v0);
                            ptx::tmem_ld_wait();
                            mask_tail(v0, T - cc * 32);
                            cm = chunk_max(v0, -INFINITY);
                        }
                        p_chunk(v0, cm, sl2, mrun, ls, tP, j);
                        ++j;
                    }
                }
                if (tail) {
                    uint32_t v0[16];
                    ptx::tmem_ld_32x32b_x16(tS + c1 * 32, v0);
                    ptx::tmem_ld_wait();
                    mask_tail(v0, T - c1 * 32);
                    p_chunk(v0, chunk_max(v0, -INFINITY), sl2, mrun, ls, tP, j);
                }
                // one offset for the row: the larger of the two halves' (they differ only
                // where a half has raised its own, and then by whole steps)
                mx_mine[row] = mrun;
                ptx::named_bar_sync(bar_id, 64);
                const float mo = mx_other[row];
                if (__any_sync(0xffffffffu, mo > mrun + 0.5f)) {
                    const float f = mo > mrun + 0.5f ? pow2_int(-rintf(mo - mrun)) : 1.f;
                    rescale_p(tP, j, tail, f);
                    f2_scale(ls, f);
                }
                ptx::tmem_st_wait();
                sL[((u & 3) * 2 + half) * AW_ROWS + row] = [&] {
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
                ptx::mbar_arrive(&bars->p_full[g]);
                ptx::mbar_arrive(&bars->l_full[u & 3]);
            }
        }
        if (!ok) {
            if (lane == 0) aw_error(p.err, ERRBIT_TIMEOUT_ATTENTION);
            *abort_flag = 1;
        }
    } else if (warp < AW_MMA_WARP) {
        // ------------------------------------------------------------------ epilogue
        const int quarter = warp & 3;
        const uint32_t tO = tmem + AW_TMEM_O + ((uint32_t)(quarter * 32) << 16);
        bool ok = true;
        for (int u = 0; u < units; ++u) {
            const int k = u / nq, qt = u - k * nq;
            const int item = (int)blockIdx.x + k * (int)gridDim.x;
            const int n = item / p.H, h = item - n * p.H;
            // the row sums are in before O (PV waited for them): take 1 / l first
            ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(&bars->l_full[u & 3], (u >> 2) & 1, abort_flag));
            if (!ok) break;
            const int row = quarter * 32 + lane;
            const float inv = 1.f / (sL[((u & 3) * 2) * AW_ROWS + row] + sL[((u & 3) * 2 + 1) * AW_ROWS + row]);
            ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded<true>(&bars->o_done, u & 1, abort_flag));
            if (!ok) break;
            ptx::tc_fence_after();
            const bool live = qt * AW_ROWS + quarter * 32 < p.T;
            uint32_t ov[64];
            if (live) {
                ptx::tmem_ld_32x32b_x32(tO, *reinterpret_cast<uint32_t(*)[32]>(&ov[0]));
                ptx::tmem_ld_32x32b_x32(tO + 32, *reinterpret_cast<uint32_t(*)[32]>(&ov[32]));
                ptx::tmem_ld_wait();
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&bars->o_free[u & 1]);
            if (live) {
                // O / l in bf16 through a 32 x 64 staging tile (128-byte rows, 16-byte unit c
                // of row r at c ^ (r % 8)) to one TMA store over (column, token, sequence):
                // rows past T lie outside the tensor and are not written
                uint8_t* stg = smem + AW_OFF_STG + quarter * AW_STG;
                uint8_t* srow = stg + lane * 128;
                if (lane == 0) ptx::bulk_wait_group_read<0>();   // the previous store has read the tile
                __syncwarp();
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(ov[8 * c + 0]) * inv, __uint_as_float(ov[8 * c + 1]) * inv);
                    w.y = pack_bf16x2(__uint_as_float(ov[8 * c + 2]) * inv, __uint_as_float(ov[8 * c + 3]) * inv);
                    w.z = pack_bf16x2(__uint_as_float(ov[8 * c + 4]) * inv, __uint_as_float(ov[8 * c + 5]) * inv);
                    w.w = pack_bf16x2(__uint_as_float(ov[8 * c + 6]) * inv, __uint_as_float(ov[8 * c + 7]) * inv);
                    *reinterpret_cast<uint4*>(srow + ((c ^ (lane & 7)) << 4)) = w;
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ptx::tma_store_3d(&tmO, stg, h * AW_DH, qt * AW_ROWS + quarter * 32, n);
                    ptx::bulk_commit_group();
                }
            }
        }
        if (lane == 0) ptx::bulk_wait_group<0>();   // stores complete before the CTA exits
        if (!ok) {
            if (lane == 0) aw_error(p.err, ERRBIT_TIMEOUT_ATTENTION);
            *abort_flag = 1;
        }
    }

    __syncthreads();
    if (warp == AW_MMA_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn aw_encode_fn() {
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

// VIT_ATTN_WHOLE=0 sends these shapes to the key-streaming kernel instead.
bool attention_whole_supported(int64_t T, int64_t D, int64_t H) {
    if (H <= 0 || D % H != 0 || D / H != AW_DH || T < 1 || T > AW_MAX_KEYS) return false;
    static const bool off = [] {
        const char* e = std::getenv("VIT_ATTN_WHOLE");
        return e && e[0] == '0';
    }();
    return !off && aw_encode_fn() != nullptr;
}

cudaError_t launch_attention_whole(const void* qkv, void* o, int64_t N, int64_t T, int64_t D, int64_t H,
                                   const DeviceInfo& dev, cudaStream_t s) {
    if (N <= 0 || T <= 0) return cudaSuccess;
    if (!attention_whole_supported(T, D, H) || N * H > 0x7fffffff) return cudaErrorInvalidValue;
    EncodeTiledFn fn = aw_encode_fn();
    alignas(64) CUtensorMap tm;
    cuuint64_t dims[3] = {(cuuint64_t)(3 * D), (cuuint64_t)T, (cuuint64_t)N};
    cuuint64_t strides[2] = {(cuuint64_t)(3 * D * 2), (cuuint64_t)(T * 3 * D * 2)};
    cuuint32_t box[3] = {AW_DH, AW_ROWS, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    if (fn(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(qkv), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // o over (column, token, sequence), box 64 x 32 x 1 (128-byte rows), for the stores
    alignas(64) CUtensorMap to;
    cuuint64_t odims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)N};
    cuuint64_t ostr[2] = {(cuuint64_t)(D * 2), (cuuint64_t)(T * D * 2)};
    cuuint32_t obox[3] = {AW_DH, 32, 1};
    if (fn(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, o, odims, ostr, obox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    AwParams p;
    p.T = (int)T;
    p.D = (int)D;
    p.H = (int)H;
    p.nq = (int)((T + AW_ROWS - 1) / AW_ROWS);
    p.ns = (int)((T + 15) / 16 * 16);
    p.nkb = (p.ns + AW_ROWS - 1) / AW_ROWS;
    {
        // half 0 takes the first ceil((full chunks + 1) / 2) 32-key chunks (it reads key
        // chunk 0 once; half 1 reads it for the offset and then takes the rest and the
        // 16-key tail)
        const int full = p.ns >> 5;
        const int sc = (full + 2) / 2 < full ? (full + 2) / 2 : full;
        p.split = sc * 32;
    }
    p.items = (int)(N * H);
    p.scale_log2 = 1.4426950408889634f / 8.0f;   // log2(e) / sqrt(64)
    p.o = static_cast<__nv_bfloat16*>(o);
    p.err = dev.err_word;
    static std::atomic<uint64_t> attr{0};
    cudaError_t ae = set_smem_limit_once(attention_whole_kernel, AW_SMEM, attr);
    if (ae != cudaSuccess) return ae;
    const int grid = p.items < dev.num_sms ? p.items : dev.num_sms;
    return launch_dependent(attention_whole_kernel, dim3(grid), dim3(AW_THREADS), AW_SMEM, s, tm, to, p);
}

}  // namespace vit
