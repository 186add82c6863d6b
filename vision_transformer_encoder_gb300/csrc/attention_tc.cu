// attention_tc.cu -- bidirectional multi-head attention on the sm_103a tensor cores
// (tcgen05 / TMEM / TMA), bf16 in and out, fp32 softmax.
//
// "ViT Encoder Block" (crackedaicode), "Multi-head attention": per sequence n and head
// h, out_h = softmax(Q_h K_h^T / sqrt(D/H)) V_h with every key visible (no mask);
// heads written side by side in order. Q, K and V are read in place from the fused
// (N, T, 3D) buffer [Q | K | V] (head h at columns h*dh of each block, as in
// "vision1 reference transcript" (nipunbatra.github.io), Page 106).
//
// Persistent kernel, one CTA per SM. A work item is (sequence, head, pair of 128-row
// query tiles), so one pass over the keys serves 256 queries (T = 197 is one item).
//   warps 10,11 TMA: each item's query tiles and then its 128-key K tiles (warp 10), V
//               tiles (warp 11) into a ring; one thread issues its copies one at a time,
//               so the streams come from two warps. A 3-D tensor map (column, token, sequence) zero-fills tokens past
//               T, so tiles never read the next sequence. A head slice is one 64-column
//               box with the 128-byte swizzle, plus, for dh = 80, one 16-column box with
//               the 32-byte swizzle for Q and K (the S MMAs for that part use a second
//               descriptor) and a second 64-column box for V, so that P.V is one N 80 MMA
//               per 16 keys over two MN-major atoms rather than an N 64 and an N 16 one.
//   warps 1, 0  MMA, one issuing thread per softmax group g (warp 1: g = 0, warp 0: g = 1;
//               one thread issues at most one MMA per ~100 cycles while the softmax warps
//               move tensor memory): S_g = Q_g K^T (M 128, N 128, K dh) into TMEM, then O_g += P_g V
//               (M 128, N dh, K 128) with V read MN-major. S and O live in TMEM. For
//               dh = 64, P also lives in TMEM (the MMA reads A from tensor memory), which
//               frees shared memory for two query buffers and four K/V stages, so the
//               loads run a whole work item ahead; for dh = 80, P is staged in shared
//               memory and the ring is one query buffer and two K/V stages.
//   warps 2-5   softmax group 0 (query tile 0), warps 6-9 group 1 (query tile 1): one
//               query row per thread. Pass 1 takes the row maximum of the valid keys,
//               pass 2 writes P = exp2(S*log2(e)/sqrt(dh) - m) in bf16 (to TMEM, or to a
//               128B-swizzled K-major shared tile), keys past T get P = 0. When the running maximum grows, the
//               thread rescales its O row in TMEM first (online softmax). At the end it
//               divides by the row sum and stores bf16.
// Each group has its own MMA issuer, and S(g, j + 1) is issued before P.V(g, j): one
// group's softmax overlaps the other's MMAs, and the next tile's scores are made while
// P.V runs (the softmax makes P in registers and waits for P.V only to store it).
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

constexpr int AT_ROWS = 128;       // query rows per tile (TMEM lanes)
constexpr int AT_KEYS = 128;       // keys per K/V tile
constexpr int AT_MAX_KV = 4;
constexpr int AT_THREADS = 384;    // 12 warps: 0-1 MMA, 2-9 softmax, 10 Q and K loads, 11 V loads
constexpr int AT_BOX64 = AT_ROWS * 128;  // 64 columns x 128 rows, 128B swizzle: 16 KB
constexpr int AT_BOX16 = AT_ROWS * 32;   // 16 columns x 128 rows, 32B swizzle: 4 KB

// PT: P kept in TMEM (dh = 64). Otherwise P is staged in shared memory.
template <int DH, bool PT>
struct AtLayout {
    static_assert(DH == 64 || DH == 80, "head width 64 or 80");
    static constexpr bool TAIL = DH == 80;          // a 16-column second box
    static constexpr int TILE = AT_BOX64 + (TAIL ? AT_BOX16 : 0);   // one Q or K tile
    // one V tile: for dh = 80 two 64-column boxes with the 128-byte swizzle (the second
    // holds columns 64..79 and 48 columns the MMA does not read), so that one N 80 MMA per
    // 16 keys reads V as two MN-major atoms
    static constexpr int VTILE = TAIL ? 2 * AT_BOX64 : AT_BOX64;
    static constexpr int QBUF = PT ? 2 : 1;         // query-pair buffers
    static constexpr int KVS = PT ? 4 : 2;          // K/V ring stages
    static constexpr int P_BYTES = PT ? 0 : AT_ROWS * AT_KEYS * 2;
    // O staged for its TMA store: a 64-column 128B-swizzled box (+ for dh = 80 a 16-column
    // box of 32-byte rows); with P in TMEM its own tile per group, otherwise the group's
    // P tile, free once the item's last P.V is done
    static constexpr int OST_BYTES = PT ? AT_BOX64 : 0;
    static constexpr int OFF_Q = 0;                 // QBUF x 2 query tiles
    static constexpr int OFF_K = OFF_Q + QBUF * 2 * TILE;
    static constexpr int OFF_V = OFF_K + KVS * TILE;
    static constexpr int OFF_P = OFF_V + KVS * VTILE;  // 2 groups: P (if staged) or O staging
    static constexpr int GROUP_BYTES = P_BYTES + OST_BYTES;
    static constexpr int OFF_BAR = OFF_P + 2 * GROUP_BYTES;
    static constexpr int SMEM = OFF_BAR + 512 + 1024;
    static_assert(KVS <= AT_MAX_KV, "ring too deep");
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(GROUP_BYTES >= AT_BOX64 + (TAIL ? AT_ROWS * 32 : 0), "O staging");
    static_assert(!PT || DH <= 64, "O and P share a 128-column TMEM slot");
};

struct AtParams {
    int tail_maps;   // 1 when the 16-column map is used (dh = 80)
    int N, T, D, H;
    int npairs;      // query-tile pairs per (sequence, head)
    int nkt;         // key tiles per sequence
    int items;
    float scale_log2;
    __nv_bfloat16* o;
    uint32_t* err;
};

struct AtBars {
    uint64_t q_full[2], q_empty[2];
    uint64_t kv_full[AT_MAX_KV], kv_empty[AT_MAX_KV];
    uint64_t s_full[2], s_read[2], p_full[2], o_done[2], o_free[2];
    uint64_t ost_full[2], ost_free[2];   // O staging written by the group / read by its store
    uint64_t done;
    uint32_t tmem_slot;
    int abort_flag;
};

__device__ __forceinline__ void at_error(uint32_t* err, uint32_t bit) {
    if (err) atomicOr(err, bit);
}

__device__ __forceinline__ void item_decode(const AtParams& p, int item, int& n, int& h, int& q0,
                                            int& nact) {
    const int pair = item % p.npairs;
    h = (item / p.npairs) % p.H;
    n = item / (p.npairs * p.H);
    q0 = pair * 2 * AT_ROWS;
    nact = (q0 + AT_ROWS < p.T) ? 2 : 1;
}

template <int DH, bool PT>
__global__ void __launch_bounds__(AT_THREADS, 1)
attention_tc_kernel(const __grid_constant__ CUtensorMap tm, const __grid_constant__ CUtensorMap tm16,
                    const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmO16,
                    const AtParams p) {
    using L = AtLayout<DH, PT>;
    constexpr int KVS = L::KVS, QB = L::QBUF;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem + L::OFF_Q;
    uint8_t* sK = smem + L::OFF_K;
    uint8_t* sV = smem + L::OFF_V;
    uint8_t* sP = smem + L::OFF_P;
    AtBars* bars = reinterpret_cast<AtBars*>(smem + L::OFF_BAR);
    volatile int* abort_flag = &bars->abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(&bars->q_full[b], 1);
            ptx::mbar_init(&bars->q_empty[b], 2);     // both MMA issuers
        }
        for (int s = 0; s < AT_MAX_KV; ++s) {
            ptx::mbar_init(&bars->kv_full[s], 1);
            ptx::mbar_init(&bars->kv_empty[s], 2);    // both MMA issuers
        }
        for (int g = 0; g < 2; ++g) {
            ptx::mbar_init(&bars->s_full[g], 1);
            ptx::mbar_init(&bars->s_read[g], 4);     // one arrival per softmax warp
            ptx::mbar_init(&bars->ost_full[g], 4);
            ptx::mbar_init(&bars->ost_free[g], 1);
            ptx::mbar_init(&bars->p_full[g], 4);     // one arrival per softmax warp
            ptx::mbar_init(&bars->o_done[g], 1);
            ptx::mbar_init(&bars->o_free[g], 4);
        }
        ptx::mbar_init(&bars->done, 2);
        bars->abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 10 && lane == 0) {
        ptx::prefetch_tensormap(&tm);
        ptx::prefetch_tensormap(&tmO);
        if (L::TAIL) {
            ptx::prefetch_tensormap(&tm16);
            ptx::prefetch_tensormap(&tmO16);
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc(&bars->tmem_slot, 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bars->tmem_slot;
    // the set-up above overlaps the previous kernel's tail; qkv is its output
    griddep_wait();
    griddep_launch_dependents();
    // TMEM columns: S_g at [128 g, 128 g + 128); O_g at 256 + 128 g; with PT, P_g (64
    // columns of bf16 pairs) right after O_g at 256 + 128 g + 64.
    const int D = p.D;

    if (warp >= 10) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producers: one thread
            // issues its boxes one after another, so K (with each item's query tiles) and V
            // come from two warps
            const bool kq = warp == 10;   // Q and K; warp 11: V
            uint32_t kv_it = 0, ii = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < p.items && ok; item += gridDim.x, ++ii) {
                int n, h, q0, nact;
                item_decode(p, item, n, h, q0, nact);
                if (kq) {
                    const uint32_t qb = ii % QB, qu = ii / QB;
                    if (!ptx::mbar_wait_bounded(&bars->q_empty[qb], (qu & 1) ^ 1, abort_flag)) { ok = false; break; }
                    ptx::mbar_arrive_expect_tx(&bars->q_full[qb], nact * L::TILE);
                    for (int g = 0; g < nact; ++g) {
                        uint8_t* dq = sQ + (qb * 2 + g) * L::TILE;
                        ptx::tma_load_3d(dq, &tm, &bars->q_full[qb], h * DH, q0 + g * AT_ROWS, n);
                        if (L::TAIL)
                            ptx::tma_load_3d(dq + AT_BOX64, &tm16, &bars->q_full[qb], h * DH + 64, q0 + g * AT_ROWS, n);
                    }
                }
                const int col = (kq ? D : 2 * D) + h * DH;
                uint8_t* ring = kq ? sK : sV;
                for (int j = 0; j < p.nkt; ++j, ++kv_it) {
                    const uint32_t st = kv_it % KVS, u = kv_it / KVS;
                    if (!ptx::mbar_wait_bounded(&bars->kv_empty[st], (u & 1) ^ 1, abort_flag)) { ok = false; break; }
                    if (kq) ptx::mbar_arrive_expect_tx(&bars->kv_full[st], L::TILE + L::VTILE);
                    uint8_t* dst = ring + st * (kq ? L::TILE : L::VTILE);
                    ptx::tma_load_3d(dst, &tm, &bars->kv_full[st], col, j * AT_KEYS, n);
                    if (L::TAIL) {
                        if (kq)
                            ptx::tma_load_3d(dst + AT_BOX64, &tm16, &bars->kv_full[st], col + 64, j * AT_KEYS, n);
                        else   // columns past the last head's 80 read as zero
                            ptx::tma_load_3d(dst + AT_BOX64, &tm, &bars->kv_full[st], col + 64, j * AT_KEYS, n);
                    }
                }
            }
            if (!ok) {
                at_error(p.err, ERRBIT_TIMEOUT_ATTENTION);
                *abort_flag = 1;
            }
            // let in-flight copies land before the CTA can exit
            if (kq)
                for (uint32_t b = 0; b < (uint32_t)QB; ++b)
                    if (ii > b && !ptx::mbar_wait_bounded(&bars->q_full[b], ((ii - 1 - b) / QB) & 1, nullptr))
                        at_error(p.err, ERRBIT_TIMEOUT_TEARDOWN);
            for (uint32_t s2 = 0; s2 < (uint32_t)KVS; ++s2)
                if (kv_it > s2 && !ptx::mbar_wait_bounded(&bars->kv_full[s2], ((kv_it - 1 - s2) / KVS) & 1, nullptr))
                    at_error(p.err, ERRBIT_TIMEOUT_TEARDOWN);
        }
    } else if (warp <= 1) {
        if (lane == 0) {
            // -------------------------------------------- MMA issuers, one per softmax group
            // (warp 1: group 0, warp 0: group 1). One thread issues an MMA only every
            // ~100-130 cycles while the softmax warps move tensor memory, so each group's
            // chain S -> P.V gets its own thread. The groups share the K/V stages and the
            // query buffer: each issuer releases them once (their empty barriers count two).
            const int g = warp == 1 ? 0 : 1;
            constexpr uint32_t idS = ptx::idesc_bf16_f32(AT_ROWS, AT_KEYS, false, false);
            constexpr uint32_t idO64 = ptx::idesc_bf16_f32(AT_ROWS, 64, false, true);
            constexpr uint32_t idO80 = ptx::idesc_bf16_f32(AT_ROWS, 80, false, true);
            uint32_t kv_base = 0, ii = 0, pc = 0, ic = 0;
            bool ok = true;
            uint32_t qb = 0;
            auto kv_wait = [&](int j) -> bool {
                const uint32_t kv = kv_base + j;
                return ptx::mbar_wait_bounded(&bars->kv_full[kv % KVS], (kv / KVS) & 1, abort_flag);
            };
            auto issue_S = [&](int j) -> bool {
                if (!kv_wait(j)) return false;
                // S_g is free again: S(g, j) is only issued after s_read(g, j - 1), which
                // the softmax warps signal once their loads of S(g, j - 1) have completed.
                ptx::tc_fence_after();
                const uint32_t st = (kv_base + j) % KVS;
                const uint32_t qa = ptx::smem_addr(sQ + (qb * 2 + g) * L::TILE);
                const uint32_t ka = ptx::smem_addr(sK + st * L::TILE);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {   // 64 columns: 128-byte rows, 32 bytes per step
                    const uint64_t ad = ptx::smem_desc(qa + kk * 32, 16, 1024, ptx::kLayoutSw128);
                    const uint64_t bd = ptx::smem_desc(ka + kk * 32, 16, 1024, ptx::kLayoutSw128);
                    ptx::mma_bf16_ss(tmem + g * AT_KEYS, ad, bd, idS, kk > 0);
                }
                if (L::TAIL) {                     // columns 64..79: one 32-byte-row step
                    const uint64_t ad = ptx::smem_desc(qa + AT_BOX64, 16, 256, ptx::kLayoutSw32);
                    const uint64_t bd = ptx::smem_desc(ka + AT_BOX64, 16, 256, ptx::kLayoutSw32);
                    ptx::mma_bf16_ss(tmem + g * AT_KEYS, ad, bd, idS, 1u);
                }
                ptx::mma_commit(&bars->s_full[g]);
                return true;
            };
            for (int item = blockIdx.x; item < p.items && ok; item += gridDim.x, ++ii) {
                int n, h, q0, nact;
                item_decode(p, item, n, h, q0, nact);
                qb = ii % QB;
                if (!ptx::mbar_wait_bounded(&bars->q_full[qb], (ii / QB) & 1, abort_flag)) { ok = false; break; }
                if (g >= nact) {
                    // no query tile for this group: release the query buffer and each K/V
                    // stage once it holds this item's tile, as the other issuer does after
                    // its products (never ahead of a stage's current phase)
                    ptx::mma_commit(&bars->q_empty[qb]);
                    for (int j = 0; j < p.nkt && ok; ++j) {
                        if (!kv_wait(j)) { ok = false; break; }
                        ptx::mma_commit(&bars->kv_empty[(kv_base + j) % KVS]);
                    }
                    kv_base += p.nkt;
                    continue;
                }
                ok = issue_S(0);
                if (p.nkt == 1 && ok) ptx::mma_commit(&bars->q_empty[qb]);
                for (int j = 0; j < p.nkt && ok; ++j) {
                    const uint32_t st = (kv_base + j) % KVS;
                    // S(g, j + 1) as soon as the softmax has read S(g, j) into registers: the
                    // next tile's scores are made while the softmax works on this one
                    if (!ptx::mbar_wait_bounded(&bars->s_read[g], pc & 1, abort_flag)) { ok = false; break; }
                    if (j + 1 < p.nkt) {
                        if (!issue_S(j + 1)) { ok = false; break; }
                        if (j + 1 == p.nkt - 1) ptx::mma_commit(&bars->q_empty[qb]);
                    }
                    if (!ptx::mbar_wait_bounded(&bars->p_full[g], pc & 1, abort_flag)) { ok = false; break; }
                    if (j == 0 && ic > 0 && !ptx::mbar_wait_bounded(&bars->o_free[g], (ic - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t va = ptx::smem_addr(sV + st * L::VTILE);
                    const uint32_t tO = tmem + 256 + g * 128;
#pragma unroll
                    for (int kk = 0; kk < AT_KEYS / 16; ++kk) {
                        // V: keys are the K dimension (rows), head columns the N dimension
                        // (MN-major); 16 keys = 16 rows of 128 bytes
                        const uint64_t bd = ptx::smem_desc(va + kk * 2048, 16, 1024, ptx::kLayoutSw128);
                        const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
                        if (PT) {
                            // P: 16 keys = 8 columns of bf16 pairs per k step
                            ptx::mma_bf16_ts(tO, tO + 64 + kk * 8, bd, idO64, acc);
                        } else {
                            const uint32_t pa = ptx::smem_addr(sP + g * L::P_BYTES);
                            const uint64_t ad = ptx::smem_desc(pa + (kk >> 2) * (AT_ROWS * 128) + (kk & 3) * 32,
                                                               16, 1024, ptx::kLayoutSw128);
                            if (L::TAIL) {
                                // N 80: two MN-major atoms of 64 columns, a box (16 KB) apart
                                const uint64_t b80 = ptx::smem_desc(va + kk * 2048, AT_BOX64, 1024, ptx::kLayoutSw128);
                                ptx::mma_bf16_ss(tO, ad, b80, idO80, acc);
                            } else {
                                ptx::mma_bf16_ss(tO, ad, bd, idO64, acc);
                            }
                        }
                    }
                    ptx::mma_commit(&bars->o_done[g]);
                    ++pc;
                    ptx::mma_commit(&bars->kv_empty[st]);
                }
                ++ic;
                kv_base += p.nkt;
            }
            if (!ok) {
                at_error(p.err, ERRBIT_TIMEOUT_MMA);
                *abort_flag = 1;
            }
            ptx::mma_commit(&bars->done);
            if (!ptx::mbar_wait_bounded(&bars->done, 0, nullptr)) at_error(p.err, ERRBIT_TIMEOUT_TEARDOWN);
        }
    } else if (warp >= 2 && warp <= 9) {
        // -------------------------------------------------------- softmax groups
        const int g = (warp - 2) >> 2;          // 0: warps 2-5, 1: warps 6-9
        const int quarter = warp & 3;           // TMEM lane quarter this warp may access
        const int r = quarter * 32 + lane;      // query row within the tile
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + g * AT_KEYS + lane_off;
        const uint32_t tO = tmem + 256 + g * 128 + lane_off;
        const uint32_t tP = tO + 64;
        uint8_t* prow = sP + g * L::P_BYTES + r * 128;   // + chunk * 16 KB (staged P)
        uint32_t ec = 0;                                    // epilogues of this group so far
        const float sl2 = p.scale_log2;
        uint32_t tt = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < p.items && ok; item += gridDim.x) {
            int n, h, q0, nact;
            item_decode(p, item, n, h, q0, nact);
            if (g >= nact) continue;
            // a warp whose 32 query rows all lie past T has no output: it only keeps the
            // barrier protocol (its rows of P and O are never read back)
            const bool live = q0 + g * AT_ROWS + quarter * 32 < p.T;
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < p.nkt; ++j, ++tt) {
                ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(&bars->s_full[g], tt & 1, abort_flag));
                if (!ok) break;
                ptx::tc_fence_after();
                // P of this tile is made in registers first; only the O rescale and the P
                // store wait for P.V of the previous tile, which runs meanwhile
                uint32_t sv[AT_KEYS];   // S, then P packed in place (bf16 pairs in sv[0, 64))
                float m_new = m, alpha = 1.f, lsum = 0.f;
                if (!live) {
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&bars->s_read[g]);
                } else {
#pragma unroll
                    for (int c = 0; c < AT_KEYS / 32; ++c)
                        ptx::tmem_ld_32x32b_x32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[c * 32]));
                    ptx::tmem_ld_wait();
                    // S(g, j) is in registers: the issuer may write S(g, j + 1) over it
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&bars->s_read[g]);
                    const int valid = min(AT_KEYS, p.T - j * AT_KEYS);
                    if (valid < AT_KEYS) {
#pragma unroll
                        for (int e = 0; e < AT_KEYS; ++e)
                            if (e >= valid) sv[e] = __float_as_uint(-INFINITY);
                    }
                    // row maximum, eight independent chains
                    float mx[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) mx[e] = __uint_as_float(sv[e]);
#pragma unroll
                    for (int e = 8; e < AT_KEYS; ++e) mx[e & 7] = fmaxf(mx[e & 7], __uint_as_float(sv[e]));
                    const float mrow = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
                    m_new = fmaxf(m, mrow * sl2);
                    alpha = exp2_approx(m - m_new);
                    // P = exp2(s * scale - m) (masked keys give exp2(-inf) = 0) in bf16, the
                    // exponent arguments and row sums in packed fp32 pairs; pair e / 2 goes to
                    // sv[e / 2], whose S value has been read already
                    const unsigned long long s2 = f2_pack(sl2, sl2), nm = f2_pack(-m_new, -m_new);
                    unsigned long long ls[4] = {0ull, 0ull, 0ull, 0ull};   // packed pairs of +0.0f
#pragma unroll
                    for (int e = 0; e < AT_KEYS; e += 2) {
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), s2, nm), x0, x1);
                        const float p0 = exp2_approx(x0);
                        const float p1 = exp2_approx(x1);
                        ls[(e >> 1) & 3] = f2_add(ls[(e >> 1) & 3], f2_pack(p0, p1));
                        sv[e >> 1] = pack_bf16x2(p0, p1);
                    }
                    float a0, a1, b0, b1;
                    f2_unpack(f2_add(ls[0], ls[1]), a0, a1);
                    f2_unpack(f2_add(ls[2], ls[3]), b0, b1);
                    lsum = (a0 + a1) + (b0 + b1);
                }
                if (j > 0) {
                    // P.V of the previous tile must be done: it reads P, and O is rescaled
                    ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(&bars->o_done[g], (tt - 1) & 1, abort_flag));
                    if (!ok) break;
                    ptx::tc_fence_after();
                } else if (!PT && ec > 0) {
                    // P shares its shared memory with the previous item's O staging
                    ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(&bars->ost_free[g], (ec - 1) & 1, abort_flag));
                    if (!ok) break;
                }
                if (live) {
                    if (j > 0 && __any_sync(0xffffffffu, alpha < 1.f)) {
                        // rescale this row of O, 16 columns at a time
#pragma unroll
                        for (int c = 0; c < DH / 16; ++c) {
                            uint32_t ov[16];
                            ptx::tmem_ld_32x32b_x16(tO + c * 16, ov);
                            ptx::tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                            ptx::tmem_st_32x32b_x16(tO + c * 16, ov);
                        }
                    }
                    m = m_new;
#pragma unroll
                    for (int c = 0; c < AT_KEYS / 32; ++c) {
                        if (PT) {
                            ptx::tmem_st_32x32b_x16(tP + c * 16, *reinterpret_cast<uint32_t(*)[16]>(&sv[c * 16]));
                        } else {
                            // four 16-byte units of the 128B-swizzled row (64 keys per row)
                            uint8_t* base = prow + (c >> 1) * (AT_ROWS * 128);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const int unit = (c & 1) * 4 + q;
                                *reinterpret_cast<uint4*>(base + ((unit ^ (r & 7)) << 4)) =
                                    make_uint4(sv[c * 16 + 4 * q], sv[c * 16 + 4 * q + 1], sv[c * 16 + 4 * q + 2],
                                               sv[c * 16 + 4 * q + 3]);
                            }
                        }
                    }
                    l = l * alpha + lsum;
                    ptx::tmem_st_wait();
                }
                ptx::tc_fence_before();
                if (!PT) ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&bars->p_full[g]);
            }
            if (!ok) break;
            // epilogue: O / l -> bf16, staged in shared memory and written by one TMA store
            // per group (rows past T fall outside the tensor and are not written)
            ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(&bars->o_done[g], (tt - 1) & 1, abort_flag));
            if (!ok) break;
            ptx::tc_fence_after();
            uint8_t* stage = sP + g * L::GROUP_BYTES;                        // this group's O staging
            const bool storer = quarter == ((2 + 4 * g) & 3) && lane == 0;   // the group's first warp
            if (PT && ec > 0) {   // the previous store has read the staging tile
                ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(&bars->ost_free[g], (ec - 1) & 1, abort_flag));
                if (!ok) break;
            }
            if (live) {
                uint32_t ov[DH];
#pragma unroll
                for (int c = 0; c < DH / 16; ++c)
                    ptx::tmem_ld_32x32b_x16(tO + c * 16, *reinterpret_cast<uint32_t(*)[16]>(&ov[c * 16]));
                ptx::tmem_ld_wait();
                const float inv = 1.f / l;
                // the staging addresses depend on the row alone; made opaque here, they are
                // computed in the epilogue instead of being held through the tile loop
                uint32_t rr = (uint32_t)r;
                asm volatile("" : "+r"(rr));
                uint8_t* srow = stage + rr * 128;   // 16-byte unit c of row r at c ^ (r % 8)
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(ov[8 * c + 0]) * inv, __uint_as_float(ov[8 * c + 1]) * inv);
                    w.y = pack_bf16x2(__uint_as_float(ov[8 * c + 2]) * inv, __uint_as_float(ov[8 * c + 3]) * inv);
                    w.z = pack_bf16x2(__uint_as_float(ov[8 * c + 4]) * inv, __uint_as_float(ov[8 * c + 5]) * inv);
                    w.w = pack_bf16x2(__uint_as_float(ov[8 * c + 6]) * inv, __uint_as_float(ov[8 * c + 7]) * inv);
                    *reinterpret_cast<uint4*>(srow + ((c ^ (rr & 7)) << 4)) = w;
                }
                if (L::TAIL) {   // columns 64..79: rows of 32 bytes, no swizzle
                    uint8_t* trow = stage + AT_BOX64 + rr * 32;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int b = 64 + 8 * c;
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(ov[b + 0]) * inv, __uint_as_float(ov[b + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(ov[b + 2]) * inv, __uint_as_float(ov[b + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(ov[b + 4]) * inv, __uint_as_float(ov[b + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(ov[b + 6]) * inv, __uint_as_float(ov[b + 7]) * inv);
                        *reinterpret_cast<uint4*>(trow + c * 16) = w;
                    }
                }
            }
            ptx::fence_proxy_async_smem();   // these writes before the store reads them
            // O has been read: P.V of the group's next item may overwrite it
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(&bars->o_free[g]);
                ptx::mbar_arrive(&bars->ost_full[g]);
            }
            bool sok = true;
            if (storer) {
                sok = ptx::mbar_wait_bounded(&bars->ost_full[g], ec & 1, abort_flag);
                if (sok) {
                    const int32_t row0 = q0 + g * AT_ROWS;
                    ptx::tma_store_3d(&tmO, stage, h * DH, row0, n);
                    if (L::TAIL) ptx::tma_store_3d(&tmO16, stage + AT_BOX64, h * DH + 64, row0, n);
                    ptx::bulk_commit_group();
                    ptx::bulk_wait_group_read<0>();
                    ptx::mbar_arrive(&bars->ost_free[g]);
                }
            }
            ok = __all_sync(0xffffffffu, sok);
            ++ec;
        }
        if (quarter == 2 && lane == 0) ptx::bulk_wait_group<0>();   // the group's last store has completed
        if (!ok) {
            if (lane == 0) at_error(p.err, ERRBIT_TIMEOUT_ATTENTION);
            *abort_flag = 1;
        }
    }

    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}


typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn at_encode_fn() {
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

template <int DH, bool PT>
cudaError_t launch_tc_dh(const void* qkv, void* o, int64_t N, int64_t T, int64_t D, int64_t H,
                         const DeviceInfo& dev, cudaStream_t s) {
    using L = AtLayout<DH, PT>;
    EncodeTiledFn fn = at_encode_fn();
    if (!fn) return cudaErrorNotSupported;
    alignas(64) CUtensorMap tm, tm16;
    cuuint64_t dims[3] = {(cuuint64_t)(3 * D), (cuuint64_t)T, (cuuint64_t)N};
    cuuint64_t strides[2] = {(cuuint64_t)(3 * D * 2), (cuuint64_t)(T * 3 * D * 2)};
    cuuint32_t box[3] = {64, AT_ROWS, 1};
    cuuint32_t box16[3] = {16, AT_ROWS, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    if (fn(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(qkv), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (fn(&tm16, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(qkv), dims, strides, box16, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // the output (N, T, D): 64-column boxes with the 128-byte swizzle of the staging tile,
    // and for dh = 80 16-column boxes of unswizzled 32-byte rows
    alignas(64) CUtensorMap tmO, tmO16;
    cuuint64_t odims[3] = {(cuuint64_t)D, (cuuint64_t)T, (cuuint64_t)N};
    cuuint64_t ostrides[2] = {(cuuint64_t)(D * 2), (cuuint64_t)(T * D * 2)};
    if (fn(&tmO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, o, odims, ostrides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    if (fn(&tmO16, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, o, odims, ostrides, box16, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    AtParams p;
    p.tail_maps = DH == 80;
    p.N = (int)N;
    p.T = (int)T;
    p.D = (int)D;
    p.H = (int)H;
    const int qt = (int)((T + AT_ROWS - 1) / AT_ROWS);
    p.npairs = (qt + 1) / 2;
    p.nkt = (int)((T + AT_KEYS - 1) / AT_KEYS);
    p.items = (int)(N * H * p.npairs);
    p.scale_log2 = 1.4426950408889634f / sqrtf((float)DH);
    p.o = static_cast<__nv_bfloat16*>(o);
    p.err = dev.err_word;
    static std::atomic<uint64_t> attr{0};
    cudaError_t ae = set_smem_limit_once(attention_tc_kernel<DH, PT>, L::SMEM, attr);
    if (ae != cudaSuccess) return ae;
    const int grid = p.items < dev.num_sms ? p.items : dev.num_sms;
    return launch_dependent(attention_tc_kernel<DH, PT>, dim3(grid), dim3(AT_THREADS), L::SMEM, s, tm, tm16, tmO,
                            tmO16, p);
}

}  // namespace

bool attention_tc_supported(int64_t N, int64_t T, int64_t D, int64_t H, const void* qkv, const void* o) {
    if (H <= 0 || D % H != 0) return false;
    const int64_t dh = D / H;
    if (dh != 64 && dh != 80) return false;
    if ((reinterpret_cast<uintptr_t>(qkv) & 15) || (reinterpret_cast<uintptr_t>(o) & 15)) return false;
    if ((3 * D * 2) % 16 != 0 || N * H * ((T + 255) / 256) > 0x7fffffff || T > (1 << 20)) return false;
    const char* e = std::getenv("VIT_ATTN_TC");
    if (e && e[0] == '0') return false;
    return at_encode_fn() != nullptr;
}

cudaError_t launch_attention_tc(const void* qkv, void* o, int64_t N, int64_t T, int64_t D, int64_t H,
                                const DeviceInfo& dev, cudaStream_t s) {
    if (N <= 0 || T <= 0) return cudaSuccess;
    switch (D / H) {
        case 64:
            if (attention_whole_supported(T, D, H)) return launch_attention_whole(qkv, o, N, T, D, H, dev, s);
            return launch_tc_dh<64, true>(qkv, o, N, T, D, H, dev, s);
        case 80: return launch_tc_dh<80, false>(qkv, o, N, T, D, H, dev, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace vit
