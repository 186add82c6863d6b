// gemm_tc.cu -- persistent tcgen05 GEMM with fused epilogues, for the four dense
// contractions of the block ("ViT Encoder Block" (crackedaicode): the Q/K/V and
// output projections of "Multi-head attention", the two MLP matrices of
// "Feed-forward stage"):
//
//   QKV : qkv = xn @ [w_q | w_k | w_v]           epilogue: store bf16
//   Wo  : y   = x + o @ w_o                       epilogue: + residual (bf16) -> fp32
//   W1  : h   = GELU_tanh(yn @ w_mlp1 [+ b1])     epilogue: GELU -> bf16
//   W2  : out = y + h @ w_mlp2 [+ b2]             epilogue: + residual (fp32) -> bf16
//
// Default kernel (sm_103a): gemm_tc_pair_kernel, a persistent CTA-pair GEMM. The two
// CTAs of a cluster (one TPC) compute a 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M 256 split 128/128 across the CTAs, N 256 split 128/128 in
// their shared memory, K 16 per instruction, bf16 in, fp32 accumulators in TMEM):
//   warps 0, 2, 3, 4  TMA producers, one 8 KB box each per ring stage (A rows 0-63, A
//                     rows 64-127, weight columns 0-63, 64-127 of this CTA's half); the
//                     completions of both CTAs are counted on the leader's barrier. Five
//                     or six ring stages of 32 KB per CTA.
//   warp 1            allocates 512 TMEM columns (two 256-column accumulators) on both
//                     CTAs; the leader's lane 0 issues the pair MMAs and multicasts its
//                     commits (ring slot free, accumulator ready) to both CTAs.
//   warps 5-12        epilogue, two warps per TMEM lane quarter (128 columns each):
//                     tcgen05.ld 32 columns at a time, bias / GELU / residual in packed
//                     fp32 pairs, a swizzled 32 x 32 staging tile in shared memory and a
//                     TMA store; residual tiles arrive by TMA one chunk ahead.
// GEMMs whose tiles fill at most half of the CTA pairs split K over the pairs and reduce
// the fp32 slices in a second kernel that applies the epilogue.
// The weights are read in their (in, out) storage order directly: the B operand is
// MN-major, so no transposed copy is made. Every wait is bounded; on expiry the
// kernel sets a bit in the device error word, lets its copies and MMAs drain, frees
// TMEM and returns.
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

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int B_BOX_BYTES = 64 * BK * 2;    // 8 KB: 64 N columns x 64 K rows
constexpr int ACC_COLS = BN;                // fp32 columns per accumulator
constexpr int TMEM_COLS = 2 * ACC_COLS;     // double-buffered
constexpr int BAR_BYTES = 256;

struct Params {
    int M, N, K;
    int n_per_w, n_w;
    const __nv_bfloat16* bias;
    const void* residual;
    int64_t ldr;
    void* out;
    int64_t ldo;
    uint32_t* err;
    TcLnFold fold;
    float2* parts_out;   // extra outputs: row partials (mean, M2), 2 per 256-column tile
    int parts_stride;
    // split K (pair kernel): work item w is tile w / ksplit over k blocks
    // [ks kb_per, (ks + 1) kb_per) with ks = w % ksplit; ksplit > 1 stores the raw fp32
    // sums of slice ks at depth ks of a 3-D output map
    int ksplit, kb_per;
};

__device__ __forceinline__ void load32(const __nv_bfloat16* p, float (&v)[32]) {
    const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint4 u = __ldg(q + i);
        float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y), c = unpack_bf16x2(u.z),
               d = unpack_bf16x2(u.w);
        v[8 * i + 0] = a.x; v[8 * i + 1] = a.y; v[8 * i + 2] = b.x; v[8 * i + 3] = b.y;
        v[8 * i + 4] = c.x; v[8 * i + 5] = c.y; v[8 * i + 6] = d.x; v[8 * i + 7] = d.y;
    }
}

__device__ __forceinline__ void load32(const float* p, float (&v)[32]) {
    const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float4 u = __ldg(q + i);
        v[4 * i + 0] = u.x; v[4 * i + 1] = u.y; v[4 * i + 2] = u.z; v[4 * i + 3] = u.w;
    }
}

__device__ __forceinline__ void set_error(uint32_t* err, uint32_t bit) {
    if (err) atomicOr(err, bit);
}


// Residual values of 32 columns of one row (nothing for other epilogues or past M/N).
template <int EPI, typename ResT>
__device__ __forceinline__ void epilogue_prefetch(const Params& p, int row, int col, float (&rv)[32]) {
    if (EPI == TC_EPI_RESID && row < p.M && col < p.N)
        load32(reinterpret_cast<const ResT*>(p.residual) + (int64_t)row * p.ldr + col, rv);
}

// 32 values of one output row inside a 32-row staging tile that a TMA store writes
// out. fp32: 128-byte rows with the 128-byte swizzle (16-byte unit u of row r at
// u ^ (r % 8)); bf16: 64-byte rows with the 64-byte swizzle (unit u at u ^ (r / 2 % 4)).
// Each group of eight rows touches eight distinct 16-byte bank groups: no conflicts.
template <typename T> struct StageIO;
template <> struct StageIO<float> {
    static constexpr int ROW_BYTES = 128;
    __device__ static void write(uint8_t* buf, int r, const float (&v)[32]) {
        uint8_t* row = buf + r * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u)
            *reinterpret_cast<float4*>(row + ((u ^ (r & 7)) << 4)) =
                make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
    }
    // the inverse: row r of a tile a TMA load wrote with the same swizzle
    __device__ static void read(const uint8_t* buf, int r, float (&v)[32]) {
        const uint8_t* row = buf + r * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float4 f = *reinterpret_cast<const float4*>(row + ((u ^ (r & 7)) << 4));
            v[4 * u] = f.x; v[4 * u + 1] = f.y; v[4 * u + 2] = f.z; v[4 * u + 3] = f.w;
        }
    }
};
template <> struct StageIO<__nv_bfloat16> {
    static constexpr int ROW_BYTES = 64;
    __device__ static void write(uint8_t* buf, int r, const float (&v)[32]) {
        uint8_t* row = buf + r * 64;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            uint4 w;
            w.x = pack_bf16x2(v[8 * u + 0], v[8 * u + 1]);
            w.y = pack_bf16x2(v[8 * u + 2], v[8 * u + 3]);
            w.z = pack_bf16x2(v[8 * u + 4], v[8 * u + 5]);
            w.w = pack_bf16x2(v[8 * u + 6], v[8 * u + 7]);
            *reinterpret_cast<uint4*>(row + ((u ^ ((r >> 1) & 3)) << 4)) = w;
        }
    }
    __device__ static void read(const uint8_t* buf, int r, float (&v)[32]) {
        const uint8_t* row = buf + r * 64;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const uint4 w = *reinterpret_cast<const uint4*>(row + ((u ^ ((r >> 1) & 3)) << 4));
            const float2 a = unpack_bf16x2(w.x), b = unpack_bf16x2(w.y), c = unpack_bf16x2(w.z),
                         d = unpack_bf16x2(w.w);
            v[8 * u + 0] = a.x; v[8 * u + 1] = a.y; v[8 * u + 2] = b.x; v[8 * u + 3] = b.y;
            v[8 * u + 4] = c.x; v[8 * u + 5] = c.y; v[8 * u + 6] = d.x; v[8 * u + 7] = d.y;
        }
    }
};

constexpr int EPI_STAGE_BYTES = 32 * 128;   // one 32 x 32 staging tile (fp32 size)

// Epilogue of this warp's 32 rows x 256 columns: TMEM -> registers (bias, GELU or
// residual) -> swizzled shared staging -> TMA store, 32 columns at a time, two staging
// tiles per warp so a store drains while the next chunk is computed. The residual
// of the next chunk is loaded into registers while the current one is processed.
template <typename T> __device__ __forceinline__ void load32f(const float* p, float (&v)[32]) {
    const float4* q = reinterpret_cast<const float4*>(p);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 u = __ldg(q + i);
        v[4 * i + 0] = u.x; v[4 * i + 1] = u.y; v[4 * i + 2] = u.z; v[4 * i + 3] = u.w;
    }
}

// Residual tiles through TMA (pair kernel): each epilogue warp keeps one 32 x 32 residual
// tile in shared memory (the swizzle of StageIO). A chunk's tile is copied into registers
// as soon as it lands, and the load of the next chunk's tile (or of the next output tile's
// first one) is issued into the same buffer while the chunk is computed and stored.
struct ResStream {
    const CUtensorMap* tm = nullptr;
    uint8_t* buf = nullptr;
    uint64_t* bar = nullptr;
    volatile int* abort = nullptr;
    uint32_t phase = 0;
    int inflight = 0;          // loads issued and not yet waited for (0 or 1)
    bool failed = false;       // a wait ran out: no further loads, residual values invalid
    bool next = false;         // after the last chunk, load the next output tile's first
    int next_col = 0, next_row0 = 0;
};

// Mean and 1/sqrt(var + eps) of one row from its partials (mean_k, M2_k) over column
// ranges of part_cols (the last one may be shorter), merged with Chan's formula.
__device__ __forceinline__ float2 merge_row_stats(const TcLnFold& f, int row) {
    float n = 0.f, mean = 0.f, m2 = 0.f;
    for (int k = 0; k < f.nparts; ++k) {
        const int rest = f.D - k * f.part_cols;
        if (rest <= 0) break;
        const float nb = (float)(rest < f.part_cols ? rest : f.part_cols);
        const float2 pb = f.parts[(int64_t)row * f.nparts + k];
        const float nt = n + nb;
        const float delta = pb.x - mean;
        mean += delta * (nb / nt);
        m2 += pb.y + delta * delta * (n * nb / nt);
        n = nt;
    }
    return make_float2(mean, rsqrtf(m2 / (float)f.D + f.eps));
}

// Epilogue of this warp's 32 rows x (32 * CHUNKS) columns: TMEM -> registers (folded
// LayerNorm or bias, GELU or residual) -> swizzled shared staging -> TMA store, 32
// columns at a time. The residual of the next chunk is loaded into registers while the
// current one is processed. With EXTRA, the same values are also stored as bf16 through
// tmOut2 and the row's (mean, M2) over these columns is written to p.parts_out.
template <int EPI, typename OutT, typename ResT, int CHUNKS, int BUFS, bool FOLD, bool EXTRA,
          int STG = EPI_STAGE_BYTES, bool RES_TMA = false>
__device__ __forceinline__ void epilogue_tile_tma(const Params& p, const CUtensorMap* tmOut,
                                                  const CUtensorMap* tmOut2, uint8_t* stage,
                                                  uint32_t t_row, int row, int row0, int n0,
                                                  int lane, int part_index, int zk, ResStream& rs) {
    float rv[32];
    if (!RES_TMA) epilogue_prefetch<EPI, ResT>(p, row, n0, rv);
    float2 st = make_float2(0.f, 1.f);
    if (FOLD && row < p.M) st = merge_row_stats(p.fold, row);
    float cnt = 0.f, cmean = 0.f, cm2 = 0.f;   // EXTRA: running statistics of this row
#pragma unroll 1
    for (int c = 0; c < CHUNKS; ++c) {
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(t_row + c * 32, r);
        const int col = n0 + c * 32;
        float rnext[32];
        if constexpr (RES_TMA) {
            if (!rs.failed) {
                const bool landed = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(rs.bar, rs.phase, rs.abort));
                rs.phase ^= 1;
                rs.inflight = 0;
                if (!landed) {
                    rs.failed = true;
                    if (lane == 0) set_error(p.err, ERRBIT_TIMEOUT_EPILOGUE);
                    *rs.abort = 1;
                }
            }
            StageIO<ResT>::read(rs.buf, lane, rv);
            ptx::fence_proxy_async_smem();   // these reads before the next copy into the buffer
            __syncwarp();
            const bool more = c + 1 < CHUNKS || rs.next;
            if (more && !rs.failed) {
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(rs.bar, 32 * StageIO<ResT>::ROW_BYTES);
                    if (c + 1 < CHUNKS)
                        ptx::tma_load_2d(rs.buf, rs.tm, rs.bar, col + 32, row0);
                    else
                        ptx::tma_load_2d(rs.buf, rs.tm, rs.bar, rs.next_col, rs.next_row0);
                }
                rs.inflight = 1;
            }
        } else if (c + 1 < CHUNKS) {
            epilogue_prefetch<EPI, ResT>(p, row, col + 32, rnext);
        }
        ptx::tmem_ld_wait();
        float val[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) val[j] = __uint_as_float(r[j]);
        if (col < p.N) {
            if (FOLD) {
                float cs[32], cb[32];
                load32f<float>(p.fold.colsum + col, cs);
                load32f<float>(p.fold.colbias + col, cb);
#pragma unroll
                for (int j = 0; j < 32; ++j) val[j] = fmaf(st.y, fmaf(-st.x, cs[j], val[j]), cb[j]);
            } else if (p.bias) {
                float b[32];
                load32(p.bias + col, b);
#pragma unroll
                for (int j = 0; j < 32; j += 2) f2_add_to(val[j], val[j + 1], b[j], b[j + 1]);
            }
            if (EPI == TC_EPI_GELU) {
#pragma unroll
                for (int j = 0; j < 32; j += 2) gelu_tanh_fast2(val[j], val[j + 1]);
            } else if (EPI == TC_EPI_RESID) {
#pragma unroll
                for (int j = 0; j < 32; j += 2) f2_add_to(val[j], val[j + 1], rv[j], rv[j + 1]);
            }
        }
        if (EPI == TC_EPI_RESID && !RES_TMA && c + 1 < CHUNKS) {
#pragma unroll
            for (int j = 0; j < 32; ++j) rv[j] = rnext[j];
        }
        if (col < p.N) {
            uint8_t* buf = stage + (c % BUFS) * STG;
            // the store issued from this buffer BUFS chunks ago must have read it
            if (lane == 0) ptx::bulk_wait_group_read<BUFS - 1>();
            __syncwarp();
            StageIO<OutT>::write(buf, lane, val);
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (zk >= 0)
                    ptx::tma_store_3d(tmOut, buf, col, row0, zk);
                else
                    ptx::tma_store_2d(tmOut, buf, col, row0);
                ptx::bulk_commit_group();
            }
            if (EXTRA) {
                // chunk statistics, merged into this row's running (count, mean, M2)
                float sm = 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) sm += val[j];
                const float mb = sm * (1.f / 32.f);
                float qb = 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float d = val[j] - mb;
                    qb = fmaf(d, d, qb);
                }
                const float nt = cnt + 32.f;
                const float delta = mb - cmean;
                cmean += delta * (32.f / nt);
                cm2 += qb + delta * delta * (cnt * 32.f / nt);
                cnt = nt;
                // bf16 copy through the same staging tile once the fp32 store has read it
                if (lane == 0) ptx::bulk_wait_group_read<0>();
                __syncwarp();
                StageIO<__nv_bfloat16>::write(buf, lane, val);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ptx::tma_store_2d(tmOut2, buf, col, row0);
                    ptx::bulk_commit_group();
                }
            }
        }
    }
    if (EXTRA && row < p.M && cnt > 0.f)
        p.parts_out[(int64_t)row * p.parts_stride + part_index] = make_float2(cmean, cm2);
}

// Ring depth and epilogue staging per epilogue and output type: a bf16 staging tile is
// half the size of an fp32 one, which leaves room for a sixth ring stage; epilogues that
// read a residual keep five (their residual tiles take the shared memory of the sixth).
template <int EPI, typename OutT> struct PairCfg {
    static constexpr int STAGES = sizeof(OutT) == 2 && EPI != TC_EPI_RESID ? 6 : 5;
    static constexpr int STAGE_TILE = sizeof(OutT) == 2 ? 32 * 64 : 32 * 128;
};
constexpr int P_EPI_WARPS = 8;
constexpr int P_THREADS = 416;  // warp 0, 2, 3, 4: TMA (one 8 KB box each per stage);
                                // warp 1: MMA; warps 5-12: epilogue
constexpr int P_A_BYTES = BM * BK * 2;          // 16 KB: this CTA's 128 rows
constexpr int P_B_BYTES = (BN / 2) * BK * 2;    // 16 KB: this CTA's 128 weight columns
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;
constexpr int P_EPI_BUFS = 1;   // staging tiles per epilogue warp
template <int EPI, typename OutT> __host__ __device__ constexpr int pair_epi_bytes() {
    return P_EPI_WARPS * P_EPI_BUFS * PairCfg<EPI, OutT>::STAGE_TILE;
}
// one 32 x 32 residual tile per epilogue warp (residual epilogues)
template <int EPI, typename ResT> __host__ __device__ constexpr int pair_res_tile() {
    return EPI == TC_EPI_RESID ? 32 * StageIO<ResT>::ROW_BYTES : 0;
}
template <int EPI, typename OutT, typename ResT> __host__ __device__ constexpr int pair_smem_bytes() {
    return PairCfg<EPI, OutT>::STAGES * P_STAGE_BYTES + pair_epi_bytes<EPI, OutT>() +
           P_EPI_WARPS * pair_res_tile<EPI, ResT>() + BAR_BYTES + 1024;
}

template <int EPI, typename OutT, typename ResT, bool FOLD, bool EXTRA>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(P_THREADS, 1)
gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2,
                    const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ CUtensorMap tmOut2,
                    const __grid_constant__ CUtensorMap tmRes, const Params p) {
    constexpr int P_STAGES = PairCfg<EPI, OutT>::STAGES;
    constexpr int P_STG = PairCfg<EPI, OutT>::STAGE_TILE;
    constexpr int RES_TILE = pair_res_tile<EPI, ResT>();
    constexpr bool RES_TMA = EPI == TC_EPI_RESID;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + P_STAGES * P_A_BYTES;
    uint8_t* sEpi = smem + P_STAGES * P_STAGE_BYTES;
    uint8_t* sRes = sEpi + pair_epi_bytes<EPI, OutT>();   // 1 KB aligned
    uint64_t* full = reinterpret_cast<uint64_t*>(sRes + P_EPI_WARPS * RES_TILE);
    uint64_t* empty = full + P_STAGES;
    uint64_t* tfull = empty + P_STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* done = tempty + 2;
    uint64_t* rbar = done + 1;   // [epilogue warp]: residual tile landed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rbar + P_EPI_WARPS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const int m_tiles = (p.M + 2 * BM - 1) / (2 * BM);
    const int n_tiles = (p.N + BN - 1) / BN;
    const int num_tiles = m_tiles * n_tiles;
    const int kblocks = p.K / BK;
    const int num_items = num_tiles * p.ksplit;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            ptx::mbar_init(full + s, 1);
            ptx::mbar_init(empty + s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(tfull + a, 1);
            ptx::mbar_init(tempty + a, 2 * P_EPI_WARPS);
        }
        ptx::mbar_init(done, 1);
        for (int e = 0; e < P_EPI_WARPS; ++e) ptx::mbar_init(rbar + e, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmB0);
        if (p.n_w > 1) ptx::prefetch_tensormap(&tmB1);
        if (p.n_w > 2) ptx::prefetch_tensormap(&tmB2);
        ptx::prefetch_tensormap(&tmOut);
        if (EXTRA) ptx::prefetch_tensormap(&tmOut2);
        if (RES_TMA) ptx::prefetch_tensormap(&tmRes);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(tmem_slot, TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();  // barriers of both CTAs initialised before any remote arrive
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the set-up above overlaps the previous kernel's tail; A and the residual are its output
    griddep_wait();
    griddep_launch_dependents();

    // TMA issue from one thread is serialised (roughly one box at a time), so four warps
    // each issue one 64-row box per stage: A rows 0-63, A rows 64-127, weight columns
    // 0-63 and 64-127 of this CTA's half.
    const int prod = warp == 0 ? 0 : (warp >= 2 && warp <= 4) ? warp - 1 : -1;
    if (prod >= 0) {
        if (lane == 0) {
            // -------------------------------------------- TMA producers (both ranks)
            const uint32_t full0 = ptx::mapa_shared(ptx::smem_addr(full), 0);  // leader's
            uint32_t it = 0;
            bool ok = true;
            for (int w = cluster; w < num_items && ok; w += nclusters) {
                const int tile = w / p.ksplit, ks = w - tile * p.ksplit;
                const int m0 = (tile / n_tiles) * 2 * BM + (int)rank * BM;
                const int n0 = (tile % n_tiles) * BN + (int)rank * (BN / 2);
                const int kb0 = ks * p.kb_per, kb1 = min(kblocks, kb0 + p.kb_per);
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const uint32_t s = it % P_STAGES, u = it / P_STAGES;
                    if (!ptx::mbar_wait_bounded<true>(empty + s, (u & 1) ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (prod == 0 && rank == 0) ptx::mbar_arrive_expect_tx(full + s, 2 * P_STAGE_BYTES);
                    const uint32_t fb = full0 + s * 8;
                    if (prod < 2) {
                        ptx::tma_load_2d_pair(sA + s * P_A_BYTES + prod * (P_A_BYTES / 2), &tmA, fb, kb * BK,
                                              m0 + prod * (BM / 2));
                    } else {
                        const int j = prod - 2;
                        const int col = n0 + 64 * j;
                        int wi = col / p.n_per_w;
                        if (wi > p.n_w - 1) wi = p.n_w - 1;  // past N: zero-filled box
                        const int lc = col - wi * p.n_per_w;
                        const CUtensorMap* tb = wi == 0 ? &tmB0 : (wi == 1 ? &tmB1 : &tmB2);
                        ptx::tma_load_2d_pair(sB + s * P_B_BYTES + j * B_BOX_BYTES, tb, fb, lc, kb * BK);
                    }
                }
            }
            if (!ok) {
                set_error(p.err, ERRBIT_TIMEOUT_PRODUCER);
                *abort_flag = 1;
            }
            if (prod == 0 && rank == 0) {
                // every copy of both CTAs completes on these barriers: let them land
                for (uint32_t s = 0; s < P_STAGES; ++s) {
                    if (it > s) {
                        const uint32_t u_last = (it - 1 - s) / P_STAGES;
                        if (!ptx::mbar_wait_bounded(full + s, u_last & 1, nullptr))
                            set_error(p.err, ERRBIT_TIMEOUT_TEARDOWN);
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // -------------------------------------------- pair MMA issuer (leader)
            constexpr uint32_t idesc = ptx::idesc_bf16_f32(2 * BM, BN, false, true);
            uint32_t it = 0;
            int local = 0;
            bool ok = true;
            for (int w = cluster; w < num_items; w += nclusters, ++local) {
                const int ks = w % p.ksplit;
                const int kb0 = ks * p.kb_per, kb1 = min(kblocks, kb0 + p.kb_per);
                const int acc = local & 1;
                const uint32_t v = (uint32_t)(local >> 1);
                if (!ptx::mbar_wait_bounded(tempty + acc, (v & 1) ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const uint32_t s = it % P_STAGES, u = it / P_STAGES;
                    if (!ptx::mbar_wait_bounded(full + s, u & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t a_base = ptx::smem_addr(sA + s * P_A_BYTES);
                    const uint32_t b_base = ptx::smem_addr(sB + s * P_B_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        const uint64_t adesc = ptx::smem_desc_sw128(a_base + k * 32, 16, 1024);
                        const uint64_t bdesc =
                            ptx::smem_desc_sw128(b_base + k * 2048, B_BOX_BYTES, 1024);
                        ptx::mma_bf16_ss_pair(d_tmem, adesc, bdesc, idesc, kb != kb0 || k != 0);
                    }
                    ptx::mma_commit_pair_mc(empty + s, 0x3);
                }
                if (!ok) break;
                ptx::mma_commit_pair_mc(tfull + acc, 0x3);
            }
            if (!ok) {
                set_error(p.err, ERRBIT_TIMEOUT_MMA);
                *abort_flag = 1;
            }
            ptx::mma_commit_pair(done);
            if (!ptx::mbar_wait_bounded(done, 0, nullptr)) set_error(p.err, ERRBIT_TIMEOUT_TEARDOWN);
        }
    } else {
        // ---------------------------------------------- epilogue warps 5..12 (both ranks)
        const int quarter = warp & 3;               // TMEM lane quarter this warp may read
        const int half = (warp - 5) >> 2;           // which 128 of the 256 columns
        const uint32_t tempty0 = ptx::mapa_shared(ptx::smem_addr(tempty), 0);  // leader's
        // this warp's residual rows and columns of item w
        auto res_row0 = [&](int w) { return ((w / p.ksplit) / n_tiles) * 2 * BM + (int)rank * BM + quarter * 32; };
        auto res_col = [&](int w) { return ((w / p.ksplit) % n_tiles) * BN + half * 128; };
        ResStream rs;
        if constexpr (RES_TMA) {
            rs.tm = &tmRes;
            rs.buf = sRes + (warp - 5) * RES_TILE;
            rs.bar = rbar + (warp - 5);
            rs.abort = abort_flag;
            if (cluster < num_items) {   // the first tile's first residual chunk
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(rs.bar, RES_TILE);
                    ptx::tma_load_2d(rs.buf, rs.tm, rs.bar, res_col(cluster), res_row0(cluster));
                }
                rs.inflight = 1;
            }
        }
        int local = 0;
        for (int w = cluster; w < num_items; w += nclusters, ++local) {
            const int tile = w / p.ksplit, ks = w - tile * p.ksplit;
            const int acc = local & 1;
            const uint32_t v = (uint32_t)(local >> 1);
            const int m0 = (tile / n_tiles) * 2 * BM + (int)rank * BM;
            const int n0 = (tile % n_tiles) * BN;
            const int row0 = m0 + quarter * 32;
            const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded<true>(tfull + acc, v & 1, abort_flag));
            if (!ok) {
                if (lane == 0) set_error(p.err, ERRBIT_TIMEOUT_EPILOGUE);
                *abort_flag = 1;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t t_row = tmem_base + acc * ACC_COLS + half * 128 + ((uint32_t)(quarter * 32) << 16);
            if constexpr (RES_TMA) {
                rs.next = w + nclusters < num_items;
                if (rs.next) {
                    rs.next_col = res_col(w + nclusters);
                    rs.next_row0 = res_row0(w + nclusters);
                }
            }
            epilogue_tile_tma<EPI, OutT, ResT, 4, P_EPI_BUFS, FOLD, EXTRA, P_STG, RES_TMA>(
                p, &tmOut, &tmOut2, sEpi + (warp - 5) * P_EPI_BUFS * P_STG, t_row, row0 + lane, row0,
                n0 + half * 128, lane, (n0 / BN) * 2 + half, p.ksplit > 1 ? ks : -1, rs);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster_relaxed(tempty0 + acc * 8);   // orders TMEM reads only
        }
        if (lane == 0) ptx::bulk_wait_group<0>();   // stores complete before the CTA exits
        if (RES_TMA && rs.inflight && !rs.failed) {
            // a residual copy issued before an early exit lands before the CTA leaves
            if (!__all_sync(0xffffffffu, ptx::mbar_wait_bounded(rs.bar, rs.phase, nullptr)) && lane == 0)
                set_error(p.err, ERRBIT_TIMEOUT_TEARDOWN);
        }
    }

    __syncthreads();
    ptx::cluster_sync();  // no CTA leaves while its peer may still touch its memory
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Row-major bf16 matrix (rows, cols) with row stride `ld` elements; box (box_cols, box_rows).
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld,
              uint32_t box_cols, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Output (rows, cols) of fp32 or bf16, row stride ld elements; 32 x 32 boxes with the
// swizzle matching StageIO (128B for fp32 rows of 128 bytes, 64B for bf16).
bool make_map_out(CUtensorMap* m, void* base, int64_t rows, int64_t cols, int64_t ld, bool f32) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const int es = f32 ? 4 : 2;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * es)};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int EPI, typename OutT, typename ResT, bool FOLD, bool EXTRA>
cudaError_t launch_inst_pair(const CUtensorMap& a, const CUtensorMap* b, const CUtensorMap& out,
                             const CUtensorMap& out2, const CUtensorMap& res, const Params& p, int grid,
                             cudaStream_t s) {
    auto k = gemm_tc_pair_kernel<EPI, OutT, ResT, FOLD, EXTRA>;
    static std::atomic<uint64_t> attr{0};
    cudaError_t e = set_smem_limit_once(k, pair_smem_bytes<EPI, OutT, ResT>(), attr);
    if (e != cudaSuccess) return e;
    return launch_dependent(k, dim3(grid), dim3(P_THREADS), pair_smem_bytes<EPI, OutT, ResT>(), s, a, b[0], b[1],
                            b[2], out, out2, res, p);
}

template <int EPI, typename OutT, typename ResT>
cudaError_t launch_any(const CUtensorMap& a, const CUtensorMap* b, const CUtensorMap& out,
                       const CUtensorMap& out2, const CUtensorMap& res, const Params& p, int grid,
                       cudaStream_t s) {
    if (p.fold.parts)
        return launch_inst_pair<EPI, OutT, ResT, true, false>(a, b, out, out2, res, p, grid, s);
    if (p.parts_out)
        return launch_inst_pair<EPI, OutT, ResT, false, true>(a, b, out, out2, res, p, grid, s);
    return launch_inst_pair<EPI, OutT, ResT, false, false>(a, b, out, out2, res, p, grid, s);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Split K (VIT_GEMM_SPLITK=0 turns it off): a pair-kernel GEMM whose output tiles fill at
// most half of the CTA pairs is cut along K so that every pair gets work, with at least
// two 64-deep k blocks per slice.
bool split_k_enabled() {
    static int v = -1;
    if (v < 0) {
        const char* e = std::getenv("VIT_GEMM_SPLITK");
        v = (e && e[0] == '0') ? 0 : 1;
    }
    return v == 1;
}

struct SplitK {
    int ksplit = 1, kb_per = 0;
};

SplitK split_k_for(int64_t M, int64_t N, int64_t K, int num_sms) {
    SplitK r;
    const int kblocks = (int)(K / BK);
    r.kb_per = kblocks;
    if (!split_k_enabled() || num_sms < 4) return r;
    const int64_t tiles = ((M + 2 * BM - 1) / (2 * BM)) * ((N + BN - 1) / BN);
    const int64_t pairs = num_sms / 2;
    if (tiles * 2 > pairs || kblocks < 4) return r;
    int64_t ks = pairs / tiles;
    if (ks > kblocks / 2) ks = kblocks / 2;
    if (ks < 2) return r;
    r.kb_per = (int)((kblocks + ks - 1) / ks);
    r.ksplit = (kblocks + r.kb_per - 1) / r.kb_per;
    return r;
}

// out[m, n] = epi(sum over slices k of part[k][m][n] (+ bias[n])) (+ residual[m, n]), the
// slices added in order; four columns per thread (N % 64 == 0).
template <int EPI, typename OutT, typename ResT>
__global__ void __launch_bounds__(256)
split_reduce_kernel(const float* __restrict__ part, int ksplit, int M, int N, const __nv_bfloat16* __restrict__ bias,
                    const ResT* __restrict__ residual, int64_t ldr, OutT* __restrict__ out, int64_t ldo) {
    const int nq = N / 4;
    const int64_t total = (int64_t)M * nq, slice = (int64_t)M * N;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int m = (int)(i / nq), n = (int)(i - (int64_t)m * nq) * 4;
        const float* src = part + (int64_t)m * N + n;
        float4 a = *reinterpret_cast<const float4*>(src);
        for (int k = 1; k < ksplit; ++k) {
            const float4 b = *reinterpret_cast<const float4*>(src + k * slice);
            a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
        }
        float v[4] = {a.x, a.y, a.z, a.w};
        if (bias) {
            const uint2 u = *reinterpret_cast<const uint2*>(bias + n);
            const float2 b0 = unpack_bf16x2(u.x), b1 = unpack_bf16x2(u.y);
            v[0] += b0.x; v[1] += b0.y; v[2] += b1.x; v[3] += b1.y;
        }
        if (EPI == TC_EPI_GELU) {
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = gelu_tanh_fast(v[j]);
        } else if (EPI == TC_EPI_RESID) {
            const ResT* r = residual + (int64_t)m * ldr + n;
            if constexpr (sizeof(ResT) == 4) {
                const float4 q = *reinterpret_cast<const float4*>(r);
                v[0] += q.x; v[1] += q.y; v[2] += q.z; v[3] += q.w;
            } else {
                const uint2 u = *reinterpret_cast<const uint2*>(r);
                const float2 q0 = unpack_bf16x2(u.x), q1 = unpack_bf16x2(u.y);
                v[0] += q0.x; v[1] += q0.y; v[2] += q1.x; v[3] += q1.y;
            }
        }
        OutT* o = out + (int64_t)m * ldo + n;
        if constexpr (sizeof(OutT) == 4) {
            *reinterpret_cast<float4*>(o) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
            uint2 u;
            u.x = pack_bf16x2(v[0], v[1]);
            u.y = pack_bf16x2(v[2], v[3]);
            *reinterpret_cast<uint2*>(o) = u;
        }
    }
}

template <int EPI, typename OutT, typename ResT>
cudaError_t launch_split_reduce(const TcGemmDesc& d, int ksplit, const DeviceInfo& dev, cudaStream_t s) {
    const int64_t total = d.M * (d.N / 4);
    int64_t blocks = (total + 255) / 256;
    if (blocks > 8 * (int64_t)dev.num_sms) blocks = 8 * (int64_t)dev.num_sms;
    split_reduce_kernel<EPI, OutT, ResT><<<(unsigned)blocks, 256, 0, s>>>(
        d.split_ws, ksplit, (int)d.M, (int)d.N, static_cast<const __nv_bfloat16*>(d.bias),
        static_cast<const ResT*>(d.residual), d.ldr, static_cast<OutT*>(d.out), d.ldo);
    return cudaGetLastError();
}

// fp32 partial sums (ksplit, rows, cols), contiguous; 32 x 32 x 1 boxes, 128B swizzle.
bool make_map_split(CUtensorMap* m, void* base, int64_t rows, int64_t cols, int ksplit) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)ksplit};
    cuuint64_t strides[2] = {(cuuint64_t)(cols * 4), (cuuint64_t)(rows * cols * 4)};
    cuuint32_t box[3] = {32, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

int64_t tc_split_ws_bytes(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev) {
    if (M <= 0 || N <= 0 || K <= 0 || K % BK != 0) return 0;
    const SplitK sk = split_k_for(M, N, K, dev.num_sms);
    return sk.ksplit > 1 ? (int64_t)sk.ksplit * M * N * 4 : 0;
}

bool tc_pair_enabled(const DeviceInfo& dev) { return dev.num_sms >= 2; }

bool tc_gemm_supported(const TcGemmDesc& d) {
    if (d.M <= 0 || d.N <= 0 || d.K <= 0) return false;
    if (d.K % BK != 0 || d.n_per_w % 64 != 0 || d.N != d.n_w * d.n_per_w) return false;
    if (d.n_w < 1 || d.n_w > 3) return false;
    if (d.M > 0x7fffffff || d.N > 0x7fffffff || d.K > 0x7fffffff) return false;
    if (!aligned16(d.a) || (d.lda * 2) % 16 != 0) return false;
    for (int i = 0; i < d.n_w; ++i)
        if (!aligned16(d.w[i])) return false;
    if (!aligned16(d.out) || (d.ldo * (d.out_f32 ? 4 : 2)) % 16 != 0) return false;
    if (d.bias && !aligned16(d.bias)) return false;
    if (d.epi == TC_EPI_RESID &&
        (!d.residual || !aligned16(d.residual) || (d.ldr * (d.residual_f32 ? 4 : 2)) % 16 != 0))
        return false;
    return encode_fn() != nullptr;
}

cudaError_t launch_gemm_tc(const TcGemmDesc& d, const DeviceInfo& dev, cudaStream_t s) {
    alignas(64) CUtensorMap ma;
    alignas(64) CUtensorMap mb[3];
    if (dev.num_sms < 2) return cudaErrorNotSupported;   // CTA pairs need two SMs
    // A is loaded as two 64-row boxes from two warps
    if (!make_map(&ma, d.a, d.M, d.K, d.lda, BK, BM / 2)) return cudaErrorInvalidValue;
    for (int i = 0; i < 3; ++i) {
        const void* w = d.w[i < d.n_w ? i : 0];
        if (!make_map(&mb[i], w, d.K, d.n_per_w, d.n_per_w, 64, BK)) return cudaErrorInvalidValue;
    }
    alignas(64) CUtensorMap mo, mo2;
    if (!make_map_out(&mo, d.out, d.M, d.N, d.ldo, d.out_f32)) return cudaErrorInvalidValue;
    if (d.extra.parts) {
        if (!make_map_out(&mo2, d.extra.out_bf16, d.M, d.N, d.N, false)) return cudaErrorInvalidValue;
    } else {
        mo2 = mo;
    }
    // split K: raw fp32 slices into split_ws, then the reduction applies the epilogue
    SplitK sk;
    sk.kb_per = (int)(d.K / BK);
    if (!d.fold.parts && !d.extra.parts && d.split_ws && d.N % 64 == 0 && aligned16(d.split_ws)) {
        const SplitK c = split_k_for(d.M, d.N, d.K, dev.num_sms);
        if (c.ksplit > 1 && (int64_t)c.ksplit * d.M * d.N * 4 <= d.split_ws_bytes) sk = c;
    }
    if (sk.ksplit > 1 && !make_map_split(&mo, d.split_ws, d.M, d.N, sk.ksplit)) return cudaErrorInvalidValue;
    // residual tiles for the pair kernel's TMA-fed residual epilogue (same boxes and swizzle
    // as the output staging tiles)
    alignas(64) CUtensorMap mres = mo;
    if (d.epi == TC_EPI_RESID && sk.ksplit == 1 &&
        !make_map_out(&mres, const_cast<void*>(d.residual), d.M, d.N, d.ldr, d.residual_f32))
        return cudaErrorInvalidValue;
    Params p;
    p.M = (int)d.M;
    p.N = (int)d.N;
    p.K = (int)d.K;
    p.n_per_w = (int)d.n_per_w;
    p.n_w = d.n_w;
    p.bias = reinterpret_cast<const __nv_bfloat16*>(d.bias);
    p.residual = d.residual;
    p.ldr = d.ldr;
    p.out = d.out;
    p.ldo = d.ldo;
    p.err = dev.err_word;
    p.fold = d.fold;
    p.parts_out = d.extra.parts;
    p.parts_stride = (int)(2 * ((d.N + BN - 1) / BN));
    p.ksplit = sk.ksplit;
    p.kb_per = sk.kb_per;
    const int64_t tiles = ((d.M + 2 * BM - 1) / (2 * BM)) * ((d.N + BN - 1) / BN) * sk.ksplit;
    const int64_t clusters = tiles < dev.num_sms / 2 ? tiles : dev.num_sms / 2;
    const int grid = (int)(2 * clusters);
    if (sk.ksplit > 1) {
        p.bias = nullptr;
        cudaError_t e = launch_any<TC_EPI_STORE, float, float>(ma, mb, mo, mo2, mres, p, grid, s);
        if (e != cudaSuccess) return e;
        switch (d.epi) {
            case TC_EPI_STORE:
                return d.out_f32 ? launch_split_reduce<TC_EPI_STORE, float, float>(d, sk.ksplit, dev, s)
                                 : launch_split_reduce<TC_EPI_STORE, __nv_bfloat16, float>(d, sk.ksplit, dev, s);
            case TC_EPI_GELU:
                return d.out_f32 ? launch_split_reduce<TC_EPI_GELU, float, float>(d, sk.ksplit, dev, s)
                                 : launch_split_reduce<TC_EPI_GELU, __nv_bfloat16, float>(d, sk.ksplit, dev, s);
            case TC_EPI_RESID:
                if (d.out_f32)
                    return d.residual_f32
                               ? launch_split_reduce<TC_EPI_RESID, float, float>(d, sk.ksplit, dev, s)
                               : launch_split_reduce<TC_EPI_RESID, float, __nv_bfloat16>(d, sk.ksplit, dev, s);
                return d.residual_f32
                           ? launch_split_reduce<TC_EPI_RESID, __nv_bfloat16, float>(d, sk.ksplit, dev, s)
                           : launch_split_reduce<TC_EPI_RESID, __nv_bfloat16, __nv_bfloat16>(d, sk.ksplit, dev, s);
        }
        return cudaErrorInvalidValue;
    }
    switch (d.epi) {
        case TC_EPI_STORE:
            return d.out_f32 ? launch_any<TC_EPI_STORE, float, float>(ma, mb, mo, mo2, mres, p, grid, s)
                             : launch_any<TC_EPI_STORE, __nv_bfloat16, float>(ma, mb, mo, mo2, mres, p, grid, s);
        case TC_EPI_GELU:
            return d.out_f32 ? launch_any<TC_EPI_GELU, float, float>(ma, mb, mo, mo2, mres, p, grid, s)
                             : launch_any<TC_EPI_GELU, __nv_bfloat16, float>(ma, mb, mo, mo2, mres, p, grid, s);
        case TC_EPI_RESID:
            if (d.out_f32)
                return d.residual_f32
                           ? launch_any<TC_EPI_RESID, float, float>(ma, mb, mo, mo2, mres, p, grid, s)
                           : launch_any<TC_EPI_RESID, float, __nv_bfloat16>(ma, mb, mo, mo2, mres, p, grid, s);
            return d.residual_f32
                       ? launch_any<TC_EPI_RESID, __nv_bfloat16, float>(ma, mb, mo, mo2, mres, p, grid, s)
                       : launch_any<TC_EPI_RESID, __nv_bfloat16, __nv_bfloat16>(ma, mb, mo, mo2, mres, p, grid, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace vit
