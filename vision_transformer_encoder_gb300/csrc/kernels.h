// kernels.h -- host-side launchers of the library's kernels (internal interface).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace vit {

// Element type tags (values match vit_dtype).
enum Dt : int { DT_F32 = 0, DT_BF16 = 1, DT_F64 = 2 };

inline size_t dt_size(int dt) { return dt == DT_F64 ? 8 : dt == DT_F32 ? 4 : 2; }

// Per-device facts the launchers need.
struct DeviceInfo {
    int device = -1;
    int num_sms = 0;
    int cc_major = 0, cc_minor = 0;
    uint32_t* err_word = nullptr;  // device address of the error word
};

// ---- bounded-wait self test (selftest.cu) -------------------------------------
// One CTA waits on an mbarrier nothing completes and sets ERRBIT_SELFTEST in *err when
// the wait gives up: after the library's wait limit, or at once with abort_first != 0.
cudaError_t launch_selftest_wait(int abort_first, uint32_t* err, cudaStream_t s);

// ---- LayerNorm (layernorm.cu) -------------------------------------------------
// out = LN(x) [* gamma + beta] row by row. Pairs: bf16->bf16, f32->bf16, f32->f32,
// f64->f64, bf16->f32. gamma/beta (either may be null) have element type gb_dt.
// fp32 LayerNorm that also writes the low part of each output (tf32_low_part) to lo,
// contiguous rows x D: the A_lo operand of a following 3xTF32 product.
cudaError_t launch_layernorm_f32_lo(const float* x, float* out, float* lo, const void* gamma, const void* beta,
                                    int gb_dt, int64_t rows, int64_t D, double eps, cudaStream_t s);
cudaError_t launch_layernorm(const void* x, int in_dt, void* out, int out_dt,
                             const void* gamma, const void* beta, int gb_dt, int64_t rows,
                             int64_t D, double eps, cudaStream_t s);

// ---- Tensor-core GEMM (gemm_tc.cu) --------------------------------------------
enum TcEpi : int { TC_EPI_STORE = 0, TC_EPI_GELU = 1, TC_EPI_RESID = 2 };

// LayerNorm folded into the GEMM (pair kernel only): A holds un-normalised rows; the
// epilogue computes rstd * (acc - mean * colsum_j) + colbias_j with mean and rstd merged
// from per-row partials (mean, M2) over ln_part_cols columns each.
struct TcLnFold {
    const float2* parts = nullptr;   // (M, nparts)
    int nparts = 0, part_cols = 0, D = 0;
    float eps = 0.f;
    const float* colsum = nullptr;   // (N)
    const float* colbias = nullptr;  // (N), includes the layer's own bias
};

// Extra outputs of the Wo epilogue (pair kernel only): a bf16 copy of the output and
// the output rows' partial statistics (mean, M2) per 128 columns.
struct TcExtraOut {
    void* out_bf16 = nullptr;        // (M, N) bf16, row stride N
    float2* parts = nullptr;         // (M, 2 * ceil(N / 256))
};


struct TcGemmDesc {
    const void* a;         // (M, K) bf16, row stride lda elements
    int64_t lda;
    const void* w[3];      // weights (K, n_per_w) bf16 row-major; N = n_w * n_per_w
    int n_w;
    int64_t n_per_w;
    int64_t M, N, K;
    int epi;
    const void* bias;      // (N) bf16 or nullptr
    const void* residual;  // (M, N) residual_f32 ? f32 : bf16, row stride ldr
    int64_t ldr;
    bool residual_f32;
    void* out;             // (M, N) out_f32 ? f32 : bf16, row stride ldo
    int64_t ldo;
    bool out_f32;
    TcLnFold fold;         // fold.parts != nullptr: LayerNorm folded (pair kernel)
    TcExtraOut extra;      // extra.parts != nullptr: extra outputs (pair kernel)
    // Split K for GEMMs with too few output tiles to fill the GPU (pair kernel, no fold or
    // extra outputs): with split_ws holding tc_split_ws_bytes(...) bytes, the K range is
    // cut into slices whose fp32 sums land in split_ws and a second kernel adds them in
    // slice order and applies the epilogue. nullptr: no split.
    float* split_ws;
    int64_t split_ws_bytes;
};

// True when the pair kernel is in use (the fused LayerNorm needs it).
bool tc_pair_enabled(const DeviceInfo& dev);

// ---- LayerNorm folding (fold.cu) ------------------------------------------------
// Row partials of x (bf16, D % 8 == 0, D <= 2048): one (mean, M2) per row.
bool row_parts_supported(int64_t D, const void* x);
cudaError_t launch_row_parts(const void* x, float2* parts, int64_t rows, int64_t D, cudaStream_t s);

// Column terms of a folded LayerNorm for weights (K, n_per_w) x n_w (concatenated
// columns, N = n_w * n_per_w): colsum_j = sum_i W'_ij, colbias_j = sum_i beta_i W_ij
// + bias_j, W' = diag(gamma) W written to w_scaled when gamma is given.
struct FoldPrep {
    const void* w[3];
    void* w_scaled[3];
    int64_t n_per_w, N, K;
    const void* gamma;
    const void* beta;
    const void* bias;
    float* colsum;
    float* colbias;
};
// scratch: fold_prep_scratch_bytes(N, K) bytes of per-chunk partial sums.
size_t fold_prep_scratch_bytes(int64_t N, int64_t K);
cudaError_t launch_fold_prep(const FoldPrep& d, float* scratch, cudaStream_t s);

// True when the tensor-core GEMM takes this shape and these pointers.
bool tc_gemm_supported(const TcGemmDesc& d);
// Bytes of split_ws a GEMM of this shape uses on this device (0: it is not split).
int64_t tc_split_ws_bytes(int64_t M, int64_t N, int64_t K, const DeviceInfo& dev);
cudaError_t launch_gemm_tc(const TcGemmDesc& d, const DeviceInfo& dev, cudaStream_t s);

// ---- CUDA-core GEMM (generic.cu) ----------------------------------------------
// out (M, N) = epi(a (M, K) @ w (K, N) [+ bias]), residual (M, N). Types:
//   a_dt / w_dt / bias_dt: input element types; acc is f64 when a_dt is f64, else f32.
struct SimtGemmDesc {
    const void* a; int a_dt; int64_t lda;
    const void* w; int w_dt; int64_t ldw;
    const void* bias; int bias_dt;
    const void* residual; int res_dt; int64_t ldr;
    void* out; int out_dt; int64_t ldo;
    int64_t M, N, K;
    int epi;  // TcEpi values
};
cudaError_t launch_gemm_simt(const SimtGemmDesc& d, cudaStream_t s);

// ---- Attention (attention.cu) -------------------------------------------------
// qkv (N, T, 3D) bf16 -> o (N, T, D) bf16 with tensor cores, for head widths the
// fast kernel covers (attention_fast_supported); otherwise the CUDA-core kernel.
bool attention_fast_supported(int64_t D, int64_t H, const void* qkv, const void* o);
cudaError_t launch_attention_fast(const void* qkv, void* o, int64_t N, int64_t T, int64_t D,
                                  int64_t H, cudaStream_t s);
// tcgen05 flash attention (attention_tc.cu): head widths 64 and 80, bf16, 16-byte
// aligned buffers. VIT_ATTN_TC=0 disables it (then the kernel above is used).
// fp32 GEMM as three TF32 tensor-core products per step. a_lo (M x K, contiguous) and
// wt / wt_lo (N x K, contiguous: the weight transposed) come from launch_split_lo /
// launch_split_wt. out (ldo), bias (N) and residual (ldr) are fp32.
struct Tf32GemmDesc {
    const float* a;
    int64_t lda;
    const float* a_lo;
    const float* wt;
    const float* wt_lo;
    int64_t M, N, K;
    int epi;
    const float* bias;
    const float* residual;
    int64_t ldr;
    float* out;
    int64_t ldo;
    float* out_lo;   // optional: the low part of each output (tf32_low_part), stride ldo
};
bool tf32x3_supported(int64_t M, int64_t N, int64_t K, int64_t lda, const void* a);
cudaError_t launch_split_lo(const float* a, int64_t rows, int64_t cols, int64_t lda, float* lo, cudaStream_t s);
// One weight of launch_split_wt: W (K x N, row stride ldw) -> W^T and W^T_lo (N x K) at
// rows [row0, row0 + N) of wt and wt_lo.
struct SplitWtJob {
    const float* w;
    int64_t K, N, ldw, row0;
    float* wt;
    float* wt_lo;
};
constexpr int kMaxSplitJobs = 6;
// All jobs in one launch (at most kMaxSplitJobs).
cudaError_t launch_split_wt(const SplitWtJob* jobs, int njobs, cudaStream_t s);
cudaError_t launch_gemm_tf32x3(const Tf32GemmDesc& d, const DeviceInfo& dev, cudaStream_t s);

// ---- Patch embedding (patch_embed.cu) ----------------------------------------
// images (N, C, Hi, Wi) -> A (N * NP, C P P) in the same dtype, flatten order 0 (c, p1, p2)
// or 1 (p1, p2, c); then tokens (N, NP + [cls], D) = [cls;] E (+ pos), E = A @ w (+ b) in
// e_dt (fp32 for bf16 tokens).
cudaError_t launch_patchify(const void* images, int dt, int64_t N, int64_t C, int64_t Hi, int64_t Wi, int64_t P,
                            int order, void* A, cudaStream_t s);
cudaError_t launch_patch_assemble(const void* E, int e_dt, const void* cls, const void* pos, int dt, int64_t N,
                                  int64_t NP, int64_t D, void* out, cudaStream_t s);

// fp32 qkv -> fp32 o on the CUDA cores (head widths 32, 48, 64, 80, 96, 128). With o_lo,
// the low part of o (tf32_low_part, contiguous (N T) x D) is written too.
bool attention_f32_supported(int64_t N, int64_t T, int64_t D, int64_t H, const void* qkv, const void* o);
cudaError_t launch_attention_f32(const void* qkv, void* o, int64_t N, int64_t T, int64_t D, int64_t H,
                                 const DeviceInfo& dev, cudaStream_t s, float* o_lo = nullptr);
// fp32 qkv -> fp32 o on the tensor cores, three TF32 products per step (attention_tf32.cu):
// head width 64, T <= 224. VIT_ATTN_F32_TC=0 turns it off.
bool attention_tf32_supported(int64_t N, int64_t T, int64_t D, int64_t H, const void* qkv, const void* o);
cudaError_t launch_attention_tf32(const void* qkv, void* o, int64_t N, int64_t T, int64_t D, int64_t H,
                                  const DeviceInfo& dev, cudaStream_t s, float* o_lo = nullptr);
// Head width 64 and T <= 224: all keys of a row in one S tile, exact one-pass softmax.
bool attention_whole_supported(int64_t T, int64_t D, int64_t H);
cudaError_t launch_attention_whole(const void* qkv, void* o, int64_t N, int64_t T, int64_t D, int64_t H,
                                   const DeviceInfo& dev, cudaStream_t s);
bool attention_tc_supported(int64_t N, int64_t T, int64_t D, int64_t H, const void* qkv,
                            const void* o);
cudaError_t launch_attention_tc(const void* qkv, void* o, int64_t N, int64_t T, int64_t D,
                                int64_t H, const DeviceInfo& dev, cudaStream_t s);
// One query row per sequence (attention_cls.cu): q row n at q + n ldq, keys / values of
// sequence n row u at k / v + (n T + u) ldkv, o row n at o + n ldo, all of type dt; heads
// are column blocks of D / H. Supported while the T scores fit in shared memory.
bool attention_cls_supported(int64_t N, int64_t T, int64_t D, int64_t H, int dt);
cudaError_t launch_attention_cls(const void* q, int64_t ldq, const void* k, const void* v, int64_t ldkv, int dt,
                                 int64_t N, int64_t T, int64_t D, int64_t H, void* o, int64_t ldo, cudaStream_t s);
// Any dtype (f32/bf16/f64 in and out, same type), any head width.
cudaError_t launch_attention_simt(const void* qkv, int dt, void* o, int64_t N, int64_t T,
                                  int64_t D, int64_t H, cudaStream_t s);

}  // namespace vit
