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

// ---- LayerNorm (layernorm.cu) -------------------------------------------------
// out = LN(x) [* gamma + beta] row by row. Pairs: bf16->bf16, f32->bf16, f32->f32,
// f64->f64, bf16->f32. gamma/beta (either may be null) have element type gb_dt.
cudaError_t launch_layernorm(const void* x, int in_dt, void* out, int out_dt,
                             const void* gamma, const void* beta, int gb_dt, int64_t rows,
                             int64_t D, double eps, cudaStream_t s);

// ---- Tensor-core GEMM (gemm_tc.cu) --------------------------------------------
enum TcEpi : int { TC_EPI_STORE = 0, TC_EPI_GELU = 1, TC_EPI_RESID = 2 };

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
};

// True when the tensor-core GEMM takes this shape and these pointers.
bool tc_gemm_supported(const TcGemmDesc& d);
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
bool attention_tc_supported(int64_t N, int64_t T, int64_t D, int64_t H, const void* qkv,
                            const void* o);
cudaError_t launch_attention_tc(const void* qkv, void* o, int64_t N, int64_t T, int64_t D,
                                int64_t H, const DeviceInfo& dev, cudaStream_t s);
// Any dtype (f32/bf16/f64 in and out, same type), any head width.
cudaError_t launch_attention_simt(const void* qkv, int dt, void* o, int64_t N, int64_t T,
                                  int64_t D, int64_t H, cudaStream_t s);

}  // namespace vit
