// gemm_tf32.cu -- fp32 GEMMs with fused epilogues on the sm_103a tensor cores, as three
// TF32 products per step ("3xTF32"):
//   A B = A_hi B_hi + A_hi B_lo + A_lo B_hi  (+ A_lo B_lo, of relative size 2^-20, dropped)
// where x_hi is x with its 13 low mantissa bits cleared -- the TF32 value the tensor core
// takes from an fp32 operand, which it truncates -- and x_lo = x - x_hi, exact in fp32.
// A single TF32 product per step would leave errors near 1e-3 in the block output.
//
// Serves the fp32 path of the block ("ViT Encoder Block" (crackedaicode): the Q, K, V,
// output and MLP products). Split kernels first write A_lo (same layout as A) and, for a
// weight stored (in, out), its transpose W^T and W^T_lo (out rows, K contiguous), so both
// operands are K-major. The GEMM is a persistent CTA-pair kernel: 256 x 256 output tiles,
// K blocks of 32 (one 128-byte swizzled row of fp32), three stages of four 16 KB TMA boxes
// per CTA (A, A_lo, W^T, W^T_lo), one box per producer warp; the leader's MMA thread issues
// per 8-element K step the three kind::tf32 pair MMAs into a double-buffered TMEM
// accumulator; eight epilogue warps per CTA add bias and residual or apply GELU (fp32
// tanh) and store fp32 rows. Every wait is bounded.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "launch.cuh"
#include "ptx.cuh"

namespace vit {
namespace {

constexpr int XM = 128, XK = 32, XSTAGES = 3;     // rows per CTA, K block, ring stages
constexpr int X_BOX = 128 * XK * 4;                  // 16 KB: 128 rows x 32 fp32
constexpr int X_STAGE = 4 * X_BOX;                   // A, A_lo, W^T, W^T_lo
constexpr int X_BAR_BYTES = 256;

struct XParams {
    int M, N, K;
    int epi;                 // TC_EPI_STORE, TC_EPI_GELU or TC_EPI_RESID
    const float* bias;       // N, or null
    const float* residual;   // M x N (ldr), for TC_EPI_RESID
    int64_t ldr;
    float* out;
    int64_t ldo;
    bool lo;                 // also store the low part of each output (out_lo)
    uint32_t* err;
};

__device__ __forceinline__ void x_error(uint32_t* err, uint32_t bit) {
    if (err) atomicOr(err, bit);
}

// Instruction descriptor, kind::tf32: D fp32 (bits 4-5 = 1), A and B TF32 (format 2 at
// bits 7-9 and 10-12), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ float tf32_hi(float v) { return __uint_as_float(__float_as_uint(v) & 0xFFFFE000u); }

// The two CTAs of a cluster compute a 256 x 256 output tile with
// tcgen05.mma.cta_group::2.kind::tf32 (M 256 split 128 / 128 over the CTAs, N 256 split
// 128 / 128 over their shared memory). Per K block of 32 each CTA stages four 16 KB boxes
// (its 128 rows of A and A_lo, its 128 rows of W^T and W^T_lo); the MMA reads both CTAs'
// halves of W^T, so each operand byte feeds twice the products of a single-CTA 128 x 128
// tile.
//   warps 0, 2, 3, 4  TMA producers (A, A_lo, W^T, W^T_lo), both CTAs; every copy of the
//                     pair completes on the leader's ring barrier
//   warp 1            allocates 512 TMEM columns (two 256-column accumulators) on both
//                     CTAs; the leader's lane 0 issues the pair MMAs and multicasts its
//                     commits (ring slot free, accumulator ready) to both CTAs
//   warps 5-12        epilogue, two warps per TMEM lane quarter (128 columns each): bias,
//                     fp32 tanh GELU or residual; each 32 x 32 fp32 chunk goes through a
//                     128B-swizzled staging tile to a TMA store (and, when asked, its low
//                     parts through the same tile to a second TMA store)
constexpr int XP_THREADS = 416;
constexpr int XP_EPI_WARPS = 8;
constexpr int XP_ACC_COLS = 256;
constexpr int XP_TMEM_COLS = 2 * XP_ACC_COLS;
constexpr int XP_STG = 32 * 128;                       // one 32 x 32 fp32 staging tile
constexpr int XP_OFF_STG = XSTAGES * X_STAGE + 1024;   // after the ring and the barriers, 1 KB aligned
constexpr int XP_SMEM = XP_OFF_STG + XP_EPI_WARPS * XP_STG + 1024;
static_assert(X_BAR_BYTES <= 1024, "barriers fit before the staging tiles");

__device__ __forceinline__ void mma_tf32_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(XP_THREADS, 1)
gemm_tf32x3_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAlo,
                        const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmBlo,
                        const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ CUtensorMap tmOutLo,
                        const XParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + XSTAGES * X_STAGE);
    uint64_t* empty = full + XSTAGES;
    uint64_t* tfull = empty + XSTAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* done = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const int m_tiles = (p.M + 2 * XM - 1) / (2 * XM);
    const int n_tiles = (p.N + XP_ACC_COLS - 1) / XP_ACC_COLS;
    const int num_tiles = m_tiles * n_tiles;
    const int kblocks = (p.K + XK - 1) / XK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < XSTAGES; ++s) {
            ptx::mbar_init(full + s, 1);    // the leader's expect-tx arrival; bytes of both CTAs
            ptx::mbar_init(empty + s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(tfull + a, 1);
            ptx::mbar_init(tempty + a, 2 * XP_EPI_WARPS);
        }
        ptx::mbar_init(done, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tmA);
        ptx::prefetch_tensormap(&tmAlo);
        ptx::prefetch_tensormap(&tmB);
        ptx::prefetch_tensormap(&tmBlo);
        ptx::prefetch_tensormap(&tmOut);
        if (p.lo) ptx::prefetch_tensormap(&tmOutLo);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(tmem_slot, XP_TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();  // barriers of both CTAs initialised before any remote arrive
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the set-up above overlaps the previous kernel's tail; A and A_lo are its output
    griddep_wait();
    griddep_launch_dependents();

    const int prod = warp == 0 ? 0 : (warp >= 2 && warp <= 4) ? warp - 1 : -1;   // 0 A, 1 A_lo, 2 W^T, 3 W^T_lo
    if (prod >= 0) {
        if (lane == 0) {
            // -------------------------------------------- TMA producers (both ranks)
            const CUtensorMap* tm = prod == 0 ? &tmA : prod == 1 ? &tmAlo : prod == 2 ? &tmB : &tmBlo;
            const uint32_t full0 = ptx::mapa_shared(ptx::smem_addr(full), 0);   // leader's
            uint32_t it = 0;
            bool ok = true;
            for (int tile = cluster; tile < num_tiles && ok; tile += nclusters) {
                const int r0 = prod < 2 ? (tile / n_tiles) * 2 * XM + (int)rank * XM
                                        : (tile % n_tiles) * XP_ACC_COLS + (int)rank * (XP_ACC_COLS / 2);
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const uint32_t s = it % XSTAGES, u = it / XSTAGES;
                    if (!ptx::mbar_wait_bounded<true>(empty + s, (u & 1) ^ 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (prod == 0 && rank == 0) ptx::mbar_arrive_expect_tx(full + s, 2 * X_STAGE);
                    ptx::tma_load_2d_pair(smem + s * X_STAGE + prod * X_BOX, tm, full0 + s * 8, kb * XK, r0);
                }
            }
            if (!ok) {
                x_error(p.err, ERRBIT_TIMEOUT_PRODUCER);
                *abort_flag = 1;
            }
            if (prod == 0 && rank == 0) {
                // every copy of both CTAs completes on these barriers: let them land
                for (uint32_t s = 0; s < XSTAGES; ++s) {
                    if (it > s) {
                        const uint32_t u_last = (it - 1 - s) / XSTAGES;
                        if (!ptx::mbar_wait_bounded(full + s, u_last & 1, nullptr))
                            x_error(p.err, ERRBIT_TIMEOUT_TEARDOWN);
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // -------------------------------------------- pair MMA issuer (leader)
            constexpr uint32_t idesc = idesc_tf32(2 * XM, XP_ACC_COLS);
            uint32_t it = 0;
            int local = 0;
            bool ok = true;
            for (int tile = cluster; tile < num_tiles; tile += nclusters, ++local) {
                const int acc = local & 1;
                const uint32_t v = (uint32_t)(local >> 1);
                if (!ptx::mbar_wait_bounded(tempty + acc, (v & 1) ^ 1, abort_flag)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * XP_ACC_COLS;
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const uint32_t s = it % XSTAGES, u = it / XSTAGES;
                    if (!ptx::mbar_wait_bounded(full + s, u & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t st = ptx::smem_addr(smem + s * X_STAGE);
#pragma unroll
                    for (int k = 0; k < XK / 8; ++k) {
                        // K-major, 128-byte swizzle: 8 fp32 = 32 bytes per K step
                        const uint64_t a = ptx::smem_desc(st + k * 32, 16, 1024, ptx::kLayoutSw128);
                        const uint64_t alo = ptx::smem_desc(st + X_BOX + k * 32, 16, 1024, ptx::kLayoutSw128);
                        const uint64_t b = ptx::smem_desc(st + 2 * X_BOX + k * 32, 16, 1024, ptx::kLayoutSw128);
                        const uint64_t blo = ptx::smem_desc(st + 3 * X_BOX + k * 32, 16, 1024, ptx::kLayoutSw128);
                        mma_tf32_pair(d_tmem, alo, b, idesc, (kb | k) != 0 ? 1u : 0u);
                        mma_tf32_pair(d_tmem, a, blo, idesc, 1u);
                        mma_tf32_pair(d_tmem, a, b, idesc, 1u);
                    }
                    ptx::mma_commit_pair_mc(empty + s, 0x3);
                }
                if (!ok) break;
                ptx::mma_commit_pair_mc(tfull + acc, 0x3);
            }
            if (!ok) {
                x_error(p.err, ERRBIT_TIMEOUT_MMA);
                *abort_flag = 1;
            }
            ptx::mma_commit_pair(done);
            if (!ptx::mbar_wait_bounded(done, 0, nullptr)) x_error(p.err, ERRBIT_TIMEOUT_TEARDOWN);
        }
    } else {
        // ---------------------------------------------- epilogue warps 5..12 (both ranks)
        const int quarter = warp & 3;               // TMEM lane quarter this warp may read
        const int half = (warp - 5) >> 2;           // which 128 of the 256 columns
        const uint32_t tempty0 = ptx::mapa_shared(ptx::smem_addr(tempty), 0);   // leader's
        uint8_t* stage = smem + XP_OFF_STG + (warp - 5) * XP_STG;
        uint8_t* srow = stage + lane * 128;   // 16-byte unit u of this lane's row at u ^ (lane % 8)
        int local = 0;
        for (int tile = cluster; tile < num_tiles; tile += nclusters, ++local) {
            const int acc = local & 1;
            const uint32_t v = (uint32_t)(local >> 1);
            const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded<true>(tfull + acc, v & 1, abort_flag));
            if (!ok) {
                if (lane == 0) x_error(p.err, ERRBIT_TIMEOUT_EPILOGUE);
                *abort_flag = 1;
                break;
            }
            ptx::tc_fence_after();
            const int row0 = (tile / n_tiles) * 2 * XM + (int)rank * XM + quarter * 32;
            const int row = row0 + lane;
            const int n0 = (tile % n_tiles) * XP_ACC_COLS + half * 128;
            const uint32_t t_row =
                tmem_base + acc * XP_ACC_COLS + half * 128 + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(t_row + c * 32, r);
                ptx::tmem_ld_wait();
                const int col0 = n0 + c * 32;
                if (row0 >= p.M || col0 >= p.N) continue;   // the whole chunk lies outside out
                const float* rrow = p.epi == TC_EPI_RESID && row < p.M ? p.residual + (int64_t)row * p.ldr : nullptr;
                float4 vv[8];
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const int col = col0 + 4 * j4;
                    float x[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) x[e] = __uint_as_float(r[4 * j4 + e]);
                    if (col < p.N) {   // N is a multiple of 4
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            if (p.bias) x[e] += p.bias[col + e];
                            if (p.epi == TC_EPI_GELU) x[e] = gelu_tanh_acc(x[e]);
                        }
                        if (rrow) {
                            const float4 rv = *reinterpret_cast<const float4*>(rrow + col);
                            x[0] += rv.x; x[1] += rv.y; x[2] += rv.z; x[3] += rv.w;
                        }
                    }
                    vv[j4] = make_float4(x[0], x[1], x[2], x[3]);
                }
                // the previous store from the staging tile has read it; rows past M and
                // columns past N fall outside the tensor and are not written
                if (lane == 0) ptx::bulk_wait_group_read<0>();
                __syncwarp();
#pragma unroll
                for (int u = 0; u < 8; ++u) *reinterpret_cast<float4*>(srow + ((u ^ (lane & 7)) << 4)) = vv[u];
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ptx::tma_store_2d(&tmOut, stage, col0, row0);
                    ptx::bulk_commit_group();
                }
                if (p.lo) {
                    if (lane == 0) ptx::bulk_wait_group_read<0>();
                    __syncwarp();
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        *reinterpret_cast<float4*>(srow + ((u ^ (lane & 7)) << 4)) =
                            make_float4(tf32_low_part(vv[u].x), tf32_low_part(vv[u].y), tf32_low_part(vv[u].z),
                                        tf32_low_part(vv[u].w));
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_2d(&tmOutLo, stage, col0, row0);
                        ptx::bulk_commit_group();
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster_relaxed(tempty0 + acc * 8);   // orders TMEM reads only
        }
        if (lane == 0) ptx::bulk_wait_group<0>();   // stores complete before the CTA exits
    }

    __syncthreads();
    ptx::cluster_sync();  // no CTA leaves while its peer may still touch its memory
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, XP_TMEM_COLS);
    }
}

// A_lo = A - A_hi, written contiguously (rows x cols); cols and lda multiples of 4.
__global__ void split_lo_kernel(const float* __restrict__ a, int64_t rows, int64_t cols, int64_t lda,
                                float* __restrict__ lo) {
    const int64_t q = cols / 4, total = rows * q;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / q, c = (i - r * q) * 4;
        const float4 v = *reinterpret_cast<const float4*>(a + r * lda + c);
        *reinterpret_cast<float4*>(lo + r * cols + c) =
            make_float4(v.x - tf32_hi(v.x), v.y - tf32_hi(v.y), v.z - tf32_hi(v.z), v.w - tf32_hi(v.w));
    }
}

// Up to kMaxSplitJobs weights per launch: job j is W_j (K x N, ldw) -> W_j^T and W_j^T_lo
// (N x K) at rows [row0, row0 + N) of its outputs, through 32 x 32 shared-memory tiles;
// the launch's CTAs cover the jobs' tiles one after another (first[j] = first CTA of j).
struct SplitWtBatch {
    SplitWtJob job[kMaxSplitJobs];
    int first[kMaxSplitJobs + 1];
    int njobs;
};

__global__ void split_wt_kernel(const __grid_constant__ SplitWtBatch b) {
    __shared__ float tile[32][33];
    int j = 0;
    while (j + 1 < b.njobs && (int)blockIdx.x >= b.first[j + 1]) ++j;
    const float* __restrict__ w = b.job[j].w;
    const int64_t K = b.job[j].K, N = b.job[j].N, ldw = b.job[j].ldw, row0 = b.job[j].row0;
    float* __restrict__ wt = b.job[j].wt;
    float* __restrict__ wt_lo = b.job[j].wt_lo;
    const int64_t ntx = (N + 31) / 32, t = (int64_t)blockIdx.x - b.first[j];
    const int64_t k0 = (t / ntx) * 32, n0 = (t % ntx) * 32;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int64_t k = k0 + i, n = n0 + threadIdx.x;
        tile[i][threadIdx.x] = (k < K && n < N) ? w[k * ldw + n] : 0.f;
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        const int64_t n = n0 + i, k = k0 + threadIdx.x;
        if (n < N && k < K) {
            const float v = tile[threadIdx.x][i];
            wt[(row0 + n) * K + k] = v;
            wt_lo[(row0 + n) * K + k] = v - tf32_hi(v);
        }
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn x_encode_fn() {
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

// fp32 rows x cols (ld elements), box 32 columns x box_rows, 128-byte swizzle, zero fill past
// the edges (loads) or clipped there (stores).
bool make_map_f32(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, uint32_t box_rows = 128) {
    EncodeTiledFn fn = x_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * 4)};
    cuuint32_t box[2] = {(cuuint32_t)XK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

bool tf32x3_supported(int64_t M, int64_t N, int64_t K, int64_t lda, const void* a) {
    return M > 0 && N > 0 && K > 0 && N % 4 == 0 && K % 4 == 0 && lda % 4 == 0 && aligned16(a) &&
           M <= 0x7fffffff && N <= 0x7fffffff && K <= 0x7fffffff && x_encode_fn() != nullptr;
}

cudaError_t launch_split_lo(const float* a, int64_t rows, int64_t cols, int64_t lda, float* lo, cudaStream_t s) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    const int64_t total = rows * (cols / 4);
    const int64_t blocks = (total + 255) / 256 < 65536 ? (total + 255) / 256 : 65536;
    split_lo_kernel<<<(unsigned)blocks, 256, 0, s>>>(a, rows, cols, lda, lo);
    return cudaGetLastError();
}

cudaError_t launch_split_wt(const SplitWtJob* jobs, int njobs, cudaStream_t s) {
    if (njobs <= 0 || njobs > kMaxSplitJobs) return cudaErrorInvalidValue;
    SplitWtBatch b;
    std::memset(&b, 0, sizeof(b));
    int64_t total = 0;
    b.njobs = njobs;
    for (int j = 0; j < njobs; ++j) {
        b.job[j] = jobs[j];
        b.first[j] = (int)total;
        if (jobs[j].K > 0 && jobs[j].N > 0) total += ((jobs[j].N + 31) / 32) * ((jobs[j].K + 31) / 32);
        if (total > 0x7fffffff) return cudaErrorInvalidValue;
    }
    b.first[njobs] = (int)total;
    if (total == 0) return cudaSuccess;
    split_wt_kernel<<<(unsigned)total, dim3(32, 8), 0, s>>>(b);
    return cudaGetLastError();
}

cudaError_t launch_gemm_tf32x3(const Tf32GemmDesc& d, const DeviceInfo& dev, cudaStream_t s) {
    if (d.M <= 0 || d.N <= 0) return cudaSuccess;
    if (!tf32x3_supported(d.M, d.N, d.K, d.lda, d.a) || !aligned16(d.a_lo) || !aligned16(d.wt) ||
        !aligned16(d.wt_lo) || !aligned16(d.out) || d.ldo % 4 != 0 || (d.out_lo && !aligned16(d.out_lo)) ||
        (d.epi == TC_EPI_RESID && (!aligned16(d.residual) || d.ldr % 4 != 0)))
        return cudaErrorInvalidValue;
    alignas(64) CUtensorMap ma, malo, mb, mblo, mo, molo;
    if (!make_map_f32(&ma, d.a, d.M, d.K, d.lda) || !make_map_f32(&malo, d.a_lo, d.M, d.K, d.K) ||
        !make_map_f32(&mb, d.wt, d.N, d.K, d.K) || !make_map_f32(&mblo, d.wt_lo, d.N, d.K, d.K) ||
        !make_map_f32(&mo, d.out, d.M, d.N, d.ldo, 32) ||
        !make_map_f32(&molo, d.out_lo ? d.out_lo : d.out, d.M, d.N, d.ldo, 32))
        return cudaErrorInvalidValue;
    XParams p;
    p.M = (int)d.M;
    p.N = (int)d.N;
    p.K = (int)d.K;
    p.epi = d.epi;
    p.bias = d.bias;
    p.residual = d.residual;
    p.ldr = d.ldr;
    p.out = d.out;
    p.ldo = d.ldo;
    p.lo = d.out_lo != nullptr;
    p.err = dev.err_word;
    static std::atomic<uint64_t> attr{0};
    cudaError_t ae = set_smem_limit_once(gemm_tf32x3_pair_kernel, XP_SMEM, attr);
    if (ae != cudaSuccess) return ae;
    const int64_t tiles = ((d.M + 2 * XM - 1) / (2 * XM)) * ((d.N + XP_ACC_COLS - 1) / XP_ACC_COLS);
    const int64_t pairs = dev.num_sms / 2;
    const int grid = 2 * (int)(tiles < pairs ? tiles : pairs);
    return launch_dependent(gemm_tf32x3_pair_kernel, dim3(grid), dim3(XP_THREADS), XP_SMEM, s, ma, malo, mb, mblo, mo, molo, p);
}

}  // namespace vit
