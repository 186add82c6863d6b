// vit_block.cu -- the C ABI (include/vit_block.h) and the host-side dispatcher.
//
// vit_block enqueues, on the caller's stream, the seven steps of one pre-LN ViT
// encoder block ("ViT Encoder Block" (crackedaicode): "Normalize before each
// stage", "Multi-head attention", "Feed-forward stage"):
//
//   1 LN1        x   -> xn
//   2 QKV GEMM   xn  -> qkv = xn @ [w_q | w_k | w_v]
//   3 attention  qkv -> o   (per sequence and head, unmasked softmax)
//   4 Wo GEMM    o   -> y   = x + o @ w_o
//   5 LN2        y   -> yn
//   6 W1 GEMM    yn  -> h   = GELU_tanh(yn @ w_mlp1 [+ b1])
//   7 W2 GEMM    h   -> out = y + h @ w_mlp2 [+ b2]
//
// bf16 shapes with D and F multiples of 64 take the tensor-core kernels (GEMMs on
// tcgen05/TMEM fed by TMA, attention on bf16 MMAs) with bf16 intermediates, except y,
// which stays fp32 between the two residual adds. Every other case (fp32, fp64, odd
// shapes) takes the CUDA-core kernels with intermediates in the accumulation type.
// Scratch comes from a library-owned stream-ordered pool and is returned on the
// same stream; nothing here synchronises unless VIT_DEBUG_SYNC=1.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "vit_block.h"

namespace vit {
namespace {

__device__ uint32_t g_err_word;

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    DeviceInfo info;
    cudaMemPool_t pool = nullptr;
    // vit_block_host's pipeline: host-to-device copies, compute (two streams, chunks
    // alternating), device-to-host copies
    cudaStream_t h2d = nullptr, comp = nullptr, comp2 = nullptr, d2h = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<int64_t> g_launches{0};

// ---- per-kernel timing -------------------------------------------------------
enum Kern { K_LN1 = 0, K_QKV, K_ATTN, K_WO, K_LN2, K_W1, K_W2, K_LN1_STATS, K_FOLD_PREP, K_TF32_SPLIT, K_FINAL_LN,
            K_PATCHIFY, K_PATCH_GEMM, K_PATCH_ASSEMBLE, K_KV, K_CLS_Q, K_CLS_ATTN, K_CLS_WO, K_CLS_LN2,
            K_CLS_W1, K_CLS_W2, K_COUNT };
const char* const kKernNames[K_COUNT] = {"ln1",          "qkv_gemm",         "attention",
                                         "wo_gemm_residual", "ln2",          "w1_gemm_gelu",
                                         "w2_gemm_residual", "ln1_row_stats", "ln_fold_prep",
                                         "tf32_weight_split", "final_ln", "patchify", "patch_gemm",
                                         "patch_assemble", "kv_gemm", "cls_q_gemm", "cls_attention",
                                         "cls_wo_gemm_residual", "cls_ln2", "cls_w1_gemm_gelu",
                                         "cls_w2_gemm_residual"};
struct Pending {
    int kind;
    cudaEvent_t a, b;
};
std::atomic<bool> g_timing{false};
std::mutex g_tmu;
std::vector<Pending> g_pending;
double g_total_ms[K_COUNT];
int64_t g_count[K_COUNT];

bool debug_sync() {
    static int v = -1;
    if (v < 0) {
        const char* e = std::getenv("VIT_DEBUG_SYNC");
        v = (e && e[0] == '1') ? 1 : 0;
    }
    return v == 1;
}

int status_from(cudaError_t e) {
    if (e == cudaSuccess) return VIT_OK;
    if (e == cudaErrorMemoryAllocation) return VIT_ERR_NOMEM;
    return VIT_ERR_CUDA;
}

// Sets up (once) and returns the state of the current device.
int current_device(DeviceState** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return VIT_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& st = g_dev[dev];
    if (!st.ready) {
        DeviceInfo info;
        info.device = dev;
        if (cudaDeviceGetAttribute(&info.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&info.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&info.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return VIT_ERR_CUDA;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return VIT_ERR_CUDA;
        info.err_word = static_cast<uint32_t*>(p);
        cudaMemPoolProps props;
        std::memset(&props, 0, sizeof(props));
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) return VIT_ERR_CUDA;
        uint64_t thr = UINT64_MAX;  // keep freed scratch for the next call
        cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &thr);
        st.info = info;
        st.pool = pool;
        st.ready = true;
    }
    *out = &st;
    return VIT_OK;
}

// Runs one kernel launcher; counts it and, with timing on, brackets it with events.
template <class F>
cudaError_t run(int kind, cudaStream_t s, F&& launch) {
    if (!g_timing.load(std::memory_order_relaxed)) {
        cudaError_t e = launch();
        if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
        return e;
    }
    cudaEvent_t a, b;
    if (cudaEventCreate(&a) != cudaSuccess) return cudaErrorUnknown;
    if (cudaEventCreate(&b) != cudaSuccess) {
        cudaEventDestroy(a);
        return cudaErrorUnknown;
    }
    cudaEventRecord(a, s);
    cudaError_t e = launch();
    cudaEventRecord(b, s);
    if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
    std::lock_guard<std::mutex> lk(g_tmu);
    g_pending.push_back({kind, a, b});
    return e;
}

inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Column terms of both LayerNorm folds (and the gain-scaled weights), prepared once
// per weight set by vit_weights_create.
struct FoldTerms {
    const float *colsum1, *colbias1, *colsum2, *colbias2;
    const void* wq_scaled;   // (3, D, D) diag(ln1_g) w_q, w_k, w_v in bf16, or null (no LN1 gain)
    const void* w1_scaled;   // (D, F) diag(ln2_g) w_mlp1 in bf16, or null (no LN2 gain)
};

struct BlockArgs {
    const void *x, *w_q, *w_k, *w_v, *w_o, *w1, *w2;
    const void *ln1_g, *ln1_b, *ln2_g, *ln2_b, *b1, *b2;
    int64_t N, T, D, F, H;
    double eps;
    int dt;
    void* out;
    // For blocks inside a stack: x and out may be the fp32 residual stream (-1: dt), and
    // the projection biases (dt) may be given; bias_scratch holds 3D elements of dt for
    // the concatenated [b_q | b_k | b_v] of the fused QKV product.
    int x_dt = -1, out_dt = -1;
    const void *b_q = nullptr, *b_k = nullptr, *b_v = nullptr, *b_o = nullptr;
    void* bias_scratch = nullptr;
    // Prepared weights: bias_scratch already holds [b_q | b_k | b_v]; fold_terms, when
    // set, replaces the per-call column terms of the folded path (whose [b_q | b_k | b_v]
    // and b1 are then inside colbias1 and colbias2).
    bool qkv_bias_ready = false;
    const FoldTerms* fold_terms = nullptr;
    // Prepared fp32 weights: transposed with their low parts once (tf32_weight_layout), so
    // the fp32 tensor-core path skips its per-call split.
    const float* tf32_wt = nullptr;
};

inline int x_dtype(const BlockArgs& a) { return a.x_dt < 0 ? a.dt : a.x_dt; }
inline int out_dtype(const BlockArgs& a) { return a.out_dt < 0 ? a.dt : a.out_dt; }
inline bool has_qkv_bias(const BlockArgs& a) { return a.b_q || a.b_k || a.b_v; }

// [b_q | b_k | b_v] into a.bias_scratch (absent ones zero), in stream order; nothing
// when prepared weights already hold it there.
cudaError_t concat_qkv_bias(const BlockArgs& a, cudaStream_t s) {
    if (a.qkv_bias_ready) return cudaSuccess;
    const size_t nb = (size_t)a.D * dt_size(a.dt);
    const void* b[3] = {a.b_q, a.b_k, a.b_v};
    for (int i = 0; i < 3; ++i) {
        uint8_t* dst = static_cast<uint8_t*>(a.bias_scratch) + i * nb;
        cudaError_t e = b[i] ? cudaMemcpyAsync(dst, b[i], nb, cudaMemcpyDeviceToDevice, s)
                             : cudaMemsetAsync(dst, 0, nb, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// out_bytes: the size of the caller's output (0: the block's (N, T, D) in dt).
int validate(const BlockArgs& a, size_t out_bytes = 0) {
    if (a.dt != DT_F32 && a.dt != DT_BF16 && a.dt != DT_F64) return VIT_ERR_DTYPE;
    if (!a.x || !a.w_q || !a.w_k || !a.w_v || !a.w_o || !a.w1 || !a.w2 || !a.out) return VIT_ERR_ARG;
    if (a.N <= 0 || a.T <= 0 || a.D <= 0 || a.F <= 0 || a.H <= 0 || a.D % a.H != 0) return VIT_ERR_ARG;
    const int64_t lim = (int64_t)1 << 40;
    if (a.N > lim / a.T || a.D > (1 << 20) || a.F > (1 << 22)) return VIT_ERR_ARG;
    const size_t es = dt_size(a.dt);
    const size_t xb = (size_t)(a.N * a.T * a.D) * es;
    const size_t dd = (size_t)(a.D * a.D) * es, df = (size_t)(a.D * a.F) * es;
    const void* in[] = {a.x, a.w_q, a.w_k, a.w_v, a.w_o, a.w1, a.w2,
                        a.ln1_g, a.ln1_b, a.ln2_g, a.ln2_b, a.b1, a.b2};
    const size_t nb[] = {xb, dd, dd, dd, dd, df, df,
                         (size_t)a.D * es, (size_t)a.D * es, (size_t)a.D * es, (size_t)a.D * es,
                         (size_t)a.F * es, (size_t)a.D * es};
    const size_t ob = out_bytes ? out_bytes : xb;
    for (int i = 0; i < 13; ++i)
        if (overlaps(a.out, ob, in[i], nb[i])) return VIT_ERR_ARG;
    return VIT_OK;
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

bool fast_path_ok(const BlockArgs& a) {
    if (a.dt != DT_BF16) return false;
    if (a.D % 64 != 0 || a.F % 64 != 0 || a.D > 2048) return false;
    if (a.N * a.T > 0x7fffffff) return false;
    const void* ps[] = {a.x, a.w_q, a.w_k, a.w_v, a.w_o, a.w1, a.w2, a.out, a.b1, a.b2};
    for (const void* p : ps)
        if (p && !al16(p)) return false;
    return true;
}

// Scratch layout of one block call, each piece rounded up to 256 bytes; every byte is
// written before it is read.
//  unfused paths: buf (xn, then o, then yn) | qkv | y | h
//  fused bf16 path (LayerNorm folded into the GEMMs): buf (o) | qkv | y | yb (bf16 copy
//  of y) | h | LN1 row partials | LN2 row partials | column terms of both folds |
//  gain-scaled weights when LN gains are given.
struct Workspace {
    bool fast, fused;
    int acc_dt;
    size_t sz_buf, sz_qkv, sz_y, sz_h;
    size_t sz_yb, sz_p1, sz_p2, sz_cols, sz_wq, sz_w1, sz_prep;
    bool tf32;                // fp32 path on the 3xTF32 tensor-core GEMM
    size_t sz_lo, sz_wt;      // its A_lo scratch and split, transposed weights
    int p2;   // LN2 partials per row
    size_t total;
};

// The fp32 path uses the 3xTF32 tensor-core GEMM unless VIT_FP32_TC=0.
bool tf32_requested() {
    static const bool on = [] {
        const char* e = std::getenv("VIT_FP32_TC");
        return !(e && e[0] == '0');
    }();
    return on;
}

// The fp32 tensor-core path's weights, each transposed (out rows, K contiguous) and
// followed by its low part: [w_q | w_k | w_v]^T, w_o^T, w_mlp1^T, w_mlp2^T.
struct Tf32Weights {
    float *wqkv_t, *wqkv_lo, *wo_t, *wo_lo, *w1_t, *w1_lo, *w2_t, *w2_lo;
};
size_t tf32_weight_bytes(int64_t D, int64_t F) { return round_up((size_t)(2 * (4 * D * D + 2 * D * F)) * 4, 256); }
Tf32Weights tf32_weight_layout(float* base, int64_t D, int64_t F) {
    Tf32Weights t;
    t.wqkv_t = base;
    t.wqkv_lo = t.wqkv_t + 3 * D * D;
    t.wo_t = t.wqkv_lo + 3 * D * D;
    t.wo_lo = t.wo_t + D * D;
    t.w1_t = t.wo_lo + D * D;
    t.w1_lo = t.w1_t + F * D;
    t.w2_t = t.w1_lo + F * D;
    t.w2_lo = t.w2_t + D * F;
    return t;
}
// The six transposes and splits, in one launch.
cudaError_t tf32_split_weights(const BlockArgs& a, const Tf32Weights& t, cudaStream_t s) {
    const int64_t D = a.D, F = a.F;
    const SplitWtJob jobs[6] = {
        {static_cast<const float*>(a.w_q), D, D, D, 0, t.wqkv_t, t.wqkv_lo},
        {static_cast<const float*>(a.w_k), D, D, D, D, t.wqkv_t, t.wqkv_lo},
        {static_cast<const float*>(a.w_v), D, D, D, 2 * D, t.wqkv_t, t.wqkv_lo},
        {static_cast<const float*>(a.w_o), D, D, D, 0, t.wo_t, t.wo_lo},
        {static_cast<const float*>(a.w1), D, F, F, 0, t.w1_t, t.w1_lo},
        {static_cast<const float*>(a.w2), F, D, D, 0, t.w2_t, t.w2_lo}};
    return launch_split_wt(jobs, 6, s);
}

Workspace workspace_layout(const BlockArgs& a, bool fused_ok) {
    Workspace w;
    const int64_t M = a.N * a.T, D = a.D, F = a.F;
    w.fast = fast_path_ok(a);
    w.fused = w.fast && fused_ok;
    w.acc_dt = w.fast ? DT_BF16 : (a.dt == DT_F64 ? DT_F64 : DT_F32);
    const size_t ea = dt_size(w.acc_dt);
    w.sz_buf = round_up((size_t)(M * D) * ea, 256);
    w.sz_qkv = round_up((size_t)(M * 3 * D) * ea, 256);
    w.sz_y = round_up((size_t)(M * D) * (w.fast ? 4 : ea), 256);
    w.sz_h = round_up((size_t)(M * F) * ea, 256);
    w.p2 = (int)(2 * ((D + 255) / 256));
    w.sz_yb = w.sz_p1 = w.sz_p2 = w.sz_cols = w.sz_wq = w.sz_w1 = w.sz_prep = 0;
    w.sz_lo = w.sz_wt = 0;
    w.tf32 = !w.fast && a.dt == DT_F32 && tf32x3_supported(M, 3 * D, D, D, a.x) && F % 4 == 0 &&
             tf32_requested();
    if (w.tf32) {
        // low parts of the products' A operands: xn, o, yn (M x D, one after another), h (M x F)
        w.sz_lo = round_up((size_t)(M * D) * 4, 256) + round_up((size_t)(M * F) * 4, 256);
        w.sz_wt = a.tf32_wt ? 0 : tf32_weight_bytes(D, F);
    }
    if (w.fused) {
        w.sz_yb = round_up((size_t)(M * D) * 2, 256);
        w.sz_p1 = round_up((size_t)M * 8, 256);
        w.sz_p2 = round_up((size_t)M * 8 * w.p2, 256);
        if (!a.fold_terms) {   // column terms computed in the call
            w.sz_cols = round_up((size_t)(2 * 3 * D + 2 * F) * 4, 256);
            if (a.ln1_g) w.sz_wq = round_up((size_t)(3 * D * D) * 2, 256);
            if (a.ln2_g) w.sz_w1 = round_up((size_t)(D * F) * 2, 256);
            const size_t p1 = fold_prep_scratch_bytes(3 * D, D), p2 = fold_prep_scratch_bytes(F, D);
            w.sz_prep = round_up(p1 > p2 ? p1 : p2, 256);
        }
    }
    w.total = w.sz_buf + w.sz_qkv + w.sz_y + w.sz_h + w.sz_yb + w.sz_p1 + w.sz_p2 + w.sz_cols + w.sz_wq +
              w.sz_w1 + w.sz_prep + w.sz_lo + w.sz_wt;
    return w;
}

// The bf16 path with LayerNorm folded into the GEMMs (prepared weights made with the
// fold, or VIT_LN_FOLD=1; with the CTA-pair GEMM):
//   prep      column terms of both folds (+ gain-scaled weights), unless prepared
//   LN1 stats row (mean, M2) of x
//   QKV GEMM  qkv = rstd (x @ W' - mean colsum) + colbias          (A = x itself)
//   attention o
//   Wo GEMM   y = x + o @ w_o [+ b_o] (fp32), plus a bf16 copy of y and y's row partials
//   W1 GEMM   h = GELU(rstd (yb @ W1' - mean colsum) + colbias)    (colbias holds b1)
//   W2 GEMM   out = y + h @ w_mlp2 [+ b2]
cudaError_t launch_block_fused(const BlockArgs& a, const DeviceInfo& dev, cudaStream_t s,
                               const Workspace& w, void* ws) {
    const int64_t M = a.N * a.T, D = a.D, F = a.F;
    uint8_t* p = static_cast<uint8_t*>(ws);
    void* o = p;                 p += w.sz_buf;
    void* qkv = p;               p += w.sz_qkv;
    void* y = p;                 p += w.sz_y;
    void* h = p;                 p += w.sz_h;
    void* yb = p;                p += w.sz_yb;
    float2* parts1 = reinterpret_cast<float2*>(p);  p += w.sz_p1;
    float2* parts2 = reinterpret_cast<float2*>(p);  p += w.sz_p2;
    float* cols = reinterpret_cast<float*>(p);      p += w.sz_cols;
    __nv_bfloat16* wq_scaled = a.ln1_g ? reinterpret_cast<__nv_bfloat16*>(p) : nullptr;  p += w.sz_wq;
    __nv_bfloat16* w1_scaled = a.ln2_g ? reinterpret_cast<__nv_bfloat16*>(p) : nullptr;  p += w.sz_w1;
    float* prep_scratch = reinterpret_cast<float*>(p);
    const float* colsum1 = cols;
    const float* colbias1 = cols + 3 * D;
    const float* colsum2 = cols + 6 * D;
    const float* colbias2 = cols + 6 * D + F;
    if (a.fold_terms) {
        const FoldTerms& t = *a.fold_terms;
        colsum1 = t.colsum1; colbias1 = t.colbias1; colsum2 = t.colsum2; colbias2 = t.colbias2;
        wq_scaled = static_cast<__nv_bfloat16*>(const_cast<void*>(t.wq_scaled));
        w1_scaled = static_cast<__nv_bfloat16*>(const_cast<void*>(t.w1_scaled));
    }
    cudaError_t e = cudaSuccess;
    auto step = [&](cudaError_t err) {
        if (e == cudaSuccess) e = err;
    };
    const void* wqkv[3] = {a.w_q, a.w_k, a.w_v};
    const void* wqkv_used[3] = {a.w_q, a.w_k, a.w_v};
    if (wq_scaled)
        for (int i = 0; i < 3; ++i) wqkv_used[i] = wq_scaled + (size_t)i * D * D;
    if (!a.fold_terms) step(run(K_FOLD_PREP, s, [&] {
        FoldPrep f1;
        std::memset(&f1, 0, sizeof(f1));
        for (int i = 0; i < 3; ++i) {
            f1.w[i] = wqkv[i];
            f1.w_scaled[i] = wq_scaled ? (void*)(wq_scaled + (size_t)i * D * D) : nullptr;
        }
        f1.n_per_w = D; f1.N = 3 * D; f1.K = D;
        f1.gamma = a.ln1_g; f1.beta = a.ln1_b; f1.bias = nullptr;
        f1.colsum = cols; f1.colbias = cols + 3 * D;
        cudaError_t r = launch_fold_prep(f1, prep_scratch, s);
        if (r != cudaSuccess) return r;
        FoldPrep f2;
        std::memset(&f2, 0, sizeof(f2));
        f2.w[0] = f2.w[1] = f2.w[2] = a.w1;
        f2.w_scaled[0] = f2.w_scaled[1] = f2.w_scaled[2] = w1_scaled;
        f2.n_per_w = F; f2.N = F; f2.K = D;
        f2.gamma = a.ln2_g; f2.beta = a.ln2_b; f2.bias = a.b1;
        f2.colsum = cols + 6 * D; f2.colbias = cols + 6 * D + F;
        return launch_fold_prep(f2, prep_scratch, s);
    }));
    step(run(K_LN1_STATS, s, [&] { return launch_row_parts(a.x, parts1, M, D, s); }));
    TcGemmDesc g;
    std::memset(&g, 0, sizeof(g));
    g.a = a.x; g.lda = D;
    g.w[0] = wqkv_used[0]; g.w[1] = wqkv_used[1]; g.w[2] = wqkv_used[2]; g.n_w = 3; g.n_per_w = D;
    g.M = M; g.N = 3 * D; g.K = D;
    g.epi = TC_EPI_STORE;
    g.out = qkv; g.ldo = 3 * D; g.out_f32 = false;
    g.fold.parts = parts1; g.fold.nparts = 1; g.fold.part_cols = (int)D; g.fold.D = (int)D;
    g.fold.eps = (float)a.eps; g.fold.colsum = colsum1; g.fold.colbias = colbias1;
    step(run(K_QKV, s, [&] { return launch_gemm_tc(g, dev, s); }));
    step(run(K_ATTN, s, [&] {
        if (attention_tc_supported(a.N, a.T, D, a.H, qkv, o)) return launch_attention_tc(qkv, o, a.N, a.T, D, a.H, dev, s);
        if (attention_fast_supported(D, a.H, qkv, o)) return launch_attention_fast(qkv, o, a.N, a.T, D, a.H, s);
        return launch_attention_simt(qkv, DT_BF16, o, a.N, a.T, D, a.H, s);
    }));
    std::memset(&g, 0, sizeof(g));
    g.a = o; g.lda = D; g.w[0] = a.w_o; g.n_w = 1; g.n_per_w = D;
    g.M = M; g.N = D; g.K = D;
    g.epi = TC_EPI_RESID; g.bias = a.b_o; g.residual = a.x; g.ldr = D; g.residual_f32 = false;
    g.out = y; g.ldo = D; g.out_f32 = true;
    g.extra.out_bf16 = yb; g.extra.parts = parts2;
    step(run(K_WO, s, [&] { return launch_gemm_tc(g, dev, s); }));
    std::memset(&g, 0, sizeof(g));
    g.a = yb; g.lda = D; g.w[0] = w1_scaled ? (const void*)w1_scaled : a.w1; g.n_w = 1; g.n_per_w = F;
    g.M = M; g.N = F; g.K = D;
    g.epi = TC_EPI_GELU;
    g.out = h; g.ldo = F; g.out_f32 = false;
    g.fold.parts = parts2; g.fold.nparts = w.p2; g.fold.part_cols = 128; g.fold.D = (int)D;
    g.fold.eps = (float)a.eps; g.fold.colsum = colsum2; g.fold.colbias = colbias2;
    step(run(K_W1, s, [&] { return launch_gemm_tc(g, dev, s); }));
    std::memset(&g, 0, sizeof(g));
    g.a = h; g.lda = F; g.w[0] = a.w2; g.n_w = 1; g.n_per_w = D;
    g.M = M; g.N = D; g.K = F;
    g.epi = TC_EPI_RESID; g.bias = a.b2; g.residual = y; g.ldr = D; g.residual_f32 = true;
    g.out = a.out; g.ldo = D; g.out_f32 = false;
    step(run(K_W2, s, [&] { return launch_gemm_tc(g, dev, s); }));
    return e;
}

// Enqueues the seven steps of the block on `s`, using `ws` (at least w.total bytes)
// as scratch.
cudaError_t launch_block_steps(const BlockArgs& a, const DeviceInfo& dev, cudaStream_t s,
                               const Workspace& w, void* ws) {
    if (w.fused) return launch_block_fused(a, dev, s, w, ws);
    const int64_t M = a.N * a.T, D = a.D, F = a.F;
    const bool fast = w.fast;
    const int acc_dt = w.acc_dt;
    const size_t ea = dt_size(acc_dt);
    const size_t sz_buf = w.sz_buf, sz_qkv = w.sz_qkv, sz_y = w.sz_y;
    cudaError_t e = cudaSuccess;
    uint8_t* base = static_cast<uint8_t*>(ws);
    void* buf = base;
    void* qkv = base + sz_buf;
    void* y = base + sz_buf + sz_qkv;
    void* h = base + sz_buf + sz_qkv + sz_y;

    auto step = [&](cudaError_t err) {
        if (e == cudaSuccess) e = err;
    };
    if (fast) {
        const int xdt = x_dtype(a), odt = out_dtype(a);
        if (has_qkv_bias(a)) step(concat_qkv_bias(a, s));
        step(run(K_LN1, s, [&] {
            return launch_layernorm(a.x, xdt, buf, DT_BF16, a.ln1_g, a.ln1_b, DT_BF16, M, D,
                                    a.eps, s);
        }));
        TcGemmDesc g;
        std::memset(&g, 0, sizeof(g));
        g.a = buf; g.lda = D;
        g.w[0] = a.w_q; g.w[1] = a.w_k; g.w[2] = a.w_v; g.n_w = 3; g.n_per_w = D;
        g.M = M; g.N = 3 * D; g.K = D;
        g.epi = TC_EPI_STORE;
        g.bias = has_qkv_bias(a) ? a.bias_scratch : nullptr;
        g.out = qkv; g.ldo = 3 * D; g.out_f32 = false;
        const bool tc = tc_gemm_supported(g);
        step(run(K_QKV, s, [&] {
            if (tc) return launch_gemm_tc(g, dev, s);
            SimtGemmDesc sd{buf, DT_BF16, D, a.w_q, DT_BF16, D, a.b_q, DT_BF16, nullptr, 0, 0,
                            qkv, DT_BF16, 3 * D, M, D, D, TC_EPI_STORE};
            cudaError_t r = launch_gemm_simt(sd, s);
            sd.w = a.w_k; sd.bias = a.b_k; sd.out = static_cast<__nv_bfloat16*>(qkv) + D;
            if (r == cudaSuccess) r = launch_gemm_simt(sd, s);
            sd.w = a.w_v; sd.bias = a.b_v; sd.out = static_cast<__nv_bfloat16*>(qkv) + 2 * D;
            if (r == cudaSuccess) r = launch_gemm_simt(sd, s);
            return r;
        }));
        step(run(K_ATTN, s, [&] {
            if (attention_tc_supported(a.N, a.T, D, a.H, qkv, buf))
                return launch_attention_tc(qkv, buf, a.N, a.T, D, a.H, dev, s);
            if (attention_fast_supported(D, a.H, qkv, buf))
                return launch_attention_fast(qkv, buf, a.N, a.T, D, a.H, s);
            return launch_attention_simt(qkv, DT_BF16, buf, a.N, a.T, D, a.H, s);
        }));
        g.a = buf; g.w[0] = a.w_o; g.n_w = 1; g.n_per_w = D; g.N = D; g.K = D;
        g.epi = TC_EPI_RESID; g.bias = a.b_o; g.residual = a.x; g.ldr = D; g.residual_f32 = xdt == DT_F32;
        g.out = y; g.ldo = D; g.out_f32 = true;
        step(run(K_WO, s, [&] {
            if (tc_gemm_supported(g)) return launch_gemm_tc(g, dev, s);
            SimtGemmDesc sd{buf, DT_BF16, D, a.w_o, DT_BF16, D, a.b_o, DT_BF16, a.x, xdt, D,
                            y, DT_F32, D, M, D, D, TC_EPI_RESID};
            return launch_gemm_simt(sd, s);
        }));
        step(run(K_LN2, s, [&] {
            return launch_layernorm(y, DT_F32, buf, DT_BF16, a.ln2_g, a.ln2_b, DT_BF16, M, D, a.eps, s);
        }));
        g.a = buf; g.w[0] = a.w1; g.n_w = 1; g.n_per_w = F; g.N = F; g.K = D;
        g.epi = TC_EPI_GELU; g.bias = a.b1; g.residual = nullptr;
        g.out = h; g.ldo = F; g.out_f32 = false;
        step(run(K_W1, s, [&] {
            if (tc_gemm_supported(g)) return launch_gemm_tc(g, dev, s);
            SimtGemmDesc sd{buf, DT_BF16, D, a.w1, DT_BF16, F, a.b1, DT_BF16, nullptr, 0, 0,
                            h, DT_BF16, F, M, F, D, TC_EPI_GELU};
            return launch_gemm_simt(sd, s);
        }));
        g.a = h; g.lda = F; g.w[0] = a.w2; g.n_w = 1; g.n_per_w = D; g.N = D; g.K = F;
        g.epi = TC_EPI_RESID; g.bias = a.b2; g.residual = y; g.ldr = D; g.residual_f32 = true;
        g.out = a.out; g.ldo = D; g.out_f32 = odt == DT_F32;
        step(run(K_W2, s, [&] {
            if (tc_gemm_supported(g)) return launch_gemm_tc(g, dev, s);
            SimtGemmDesc sd{h, DT_BF16, F, a.w2, DT_BF16, D, a.b2, DT_BF16, y, DT_F32, D,
                            a.out, odt, D, M, D, F, TC_EPI_RESID};
            return launch_gemm_simt(sd, s);
        }));
    } else if (w.tf32) {
        // fp32: LayerNorm on the CUDA cores, attention and the products as 3xTF32. Each
        // product's A_lo (the low part of its A operand) is written by the kernel that makes
        // A: the LayerNorms, the attention and the W1 product (a split pass after the
        // CUDA-core attention that other shapes take).
        uint8_t* tail = static_cast<uint8_t*>(h) + w.sz_h;   // the A_lo parts, then the split weights
        float* lo = reinterpret_cast<float*>(tail);                                         // M x D
        float* lo_h = reinterpret_cast<float*>(tail + round_up((size_t)(M * D) * 4, 256));   // M x F
        const Tf32Weights tw = tf32_weight_layout(
            a.tf32_wt ? const_cast<float*>(a.tf32_wt) : reinterpret_cast<float*>(tail + w.sz_lo), D, F);
        float *wqkv_t = tw.wqkv_t, *wqkv_lo = tw.wqkv_lo, *wo_t = tw.wo_t, *wo_lo = tw.wo_lo;
        float *w1_t = tw.w1_t, *w1_lo = tw.w1_lo, *w2_t = tw.w2_t, *w2_lo = tw.w2_lo;
        const float* fx = static_cast<const float*>(a.x);
        float* fbuf = static_cast<float*>(buf);
        float* fqkv = static_cast<float*>(qkv);
        float* fy = static_cast<float*>(y);
        float* fh = static_cast<float*>(h);
        if (!a.tf32_wt) step(run(K_TF32_SPLIT, s, [&] { return tf32_split_weights(a, tw, s); }));
        auto gemm = [&](const float* A, const float* A_lo, int64_t K, const float* bt, const float* btlo, int64_t N,
                        int epi, const void* bias, const float* res, float* out, float* out_lo) {
            Tf32GemmDesc g{A, K, A_lo, bt, btlo, M, N, K, epi, static_cast<const float*>(bias), res, N, out, N, out_lo};
            return launch_gemm_tf32x3(g, dev, s);
        };
        step(run(K_LN1, s, [&] {
            return launch_layernorm_f32_lo(fx, fbuf, lo, a.ln1_g, a.ln1_b, DT_F32, M, D, a.eps, s);
        }));
        if (has_qkv_bias(a)) step(concat_qkv_bias(a, s));
        const void* bqkv = has_qkv_bias(a) ? a.bias_scratch : nullptr;
        step(run(K_QKV, s, [&] {
            return gemm(fbuf, lo, D, wqkv_t, wqkv_lo, 3 * D, TC_EPI_STORE, bqkv, nullptr, fqkv, nullptr);
        }));
        step(run(K_ATTN, s, [&] {
            if (attention_f32_supported(a.N, a.T, D, a.H, qkv, buf))
                return launch_attention_f32(qkv, buf, a.N, a.T, D, a.H, dev, s, lo);
            cudaError_t r = launch_attention_simt(qkv, DT_F32, buf, a.N, a.T, D, a.H, s);
            return r == cudaSuccess ? launch_split_lo(fbuf, M, D, D, lo, s) : r;
        }));
        step(run(K_WO, s, [&] { return gemm(fbuf, lo, D, wo_t, wo_lo, D, TC_EPI_RESID, a.b_o, fx, fy, nullptr); }));
        step(run(K_LN2, s, [&] {
            return launch_layernorm_f32_lo(fy, fbuf, lo, a.ln2_g, a.ln2_b, DT_F32, M, D, a.eps, s);
        }));
        step(run(K_W1, s, [&] { return gemm(fbuf, lo, D, w1_t, w1_lo, F, TC_EPI_GELU, a.b1, nullptr, fh, lo_h); }));
        step(run(K_W2, s, [&] {
            return gemm(fh, lo_h, F, w2_t, w2_lo, D, TC_EPI_RESID, a.b2, fy, static_cast<float*>(a.out), nullptr);
        }));
    } else {
        const int dt = a.dt;
        step(run(K_LN1, s, [&] {
            return launch_layernorm(a.x, x_dtype(a), buf, acc_dt, a.ln1_g, a.ln1_b, dt, M, D, a.eps, s);
        }));
        SimtGemmDesc sd{buf, acc_dt, D, a.w_q, dt, D, a.b_q, dt, nullptr, 0, 0, qkv, acc_dt, 3 * D,
                        M, D, D, TC_EPI_STORE};
        step(run(K_QKV, s, [&] {
            cudaError_t r = launch_gemm_simt(sd, s);
            SimtGemmDesc k2 = sd;
            k2.w = a.w_k;
            k2.bias = a.b_k;
            k2.out = static_cast<uint8_t*>(qkv) + D * ea;
            if (r == cudaSuccess) r = launch_gemm_simt(k2, s);
            k2.w = a.w_v;
            k2.bias = a.b_v;
            k2.out = static_cast<uint8_t*>(qkv) + 2 * D * ea;
            if (r == cudaSuccess) r = launch_gemm_simt(k2, s);
            return r;
        }));
        step(run(K_ATTN, s, [&] {
            if (acc_dt == DT_F32 && attention_f32_supported(a.N, a.T, D, a.H, qkv, buf))
                return launch_attention_f32(qkv, buf, a.N, a.T, D, a.H, dev, s);
            return launch_attention_simt(qkv, acc_dt, buf, a.N, a.T, D, a.H, s);
        }));
        step(run(K_WO, s, [&] {
            SimtGemmDesc w{buf, acc_dt, D, a.w_o, dt, D, a.b_o, dt, a.x, x_dtype(a), D, y, acc_dt, D,
                           M, D, D, TC_EPI_RESID};
            return launch_gemm_simt(w, s);
        }));
        step(run(K_LN2, s, [&] {
            return launch_layernorm(y, acc_dt, buf, acc_dt, a.ln2_g, a.ln2_b, dt, M, D, a.eps, s);
        }));
        step(run(K_W1, s, [&] {
            SimtGemmDesc w{buf, acc_dt, D, a.w1, dt, F, a.b1, dt, nullptr, 0, 0, h, acc_dt, F,
                           M, F, D, TC_EPI_GELU};
            return launch_gemm_simt(w, s);
        }));
        step(run(K_W2, s, [&] {
            SimtGemmDesc w{h, acc_dt, F, a.w2, dt, D, a.b2, dt, y, acc_dt, D, a.out, out_dtype(a), D,
                           M, D, F, TC_EPI_RESID};
            return launch_gemm_simt(w, s);
        }));
    }
    return e;
}

// ---- CLS-only block -------------------------------------------------------------
// Lecture transcript (nipunbatra.github.io), Page 55: when only the CLS token (row 0 of
// each sequence) is read after the last block, that block need only produce row 0. Its
// one query is scored against the keys of all T rows and mixes the value rows of all T
// rows, so LN1 and the key and value projections still cover every row; the query, the
// attention output, the output projection, LN2 and the MLP cover the N CLS rows:
//   1 LN1        x (all rows)          -> xn
//   2 K/V GEMM   xn                    -> kv = xn @ [w_k | w_v] (+ [b_k | b_v])
//   3 Q GEMM     xn rows 0 (stride T D) -> q = xn0 @ w_q (+ b_q)
//   4 attention  q, kv                 -> o (N, D)
//   5 Wo GEMM    o                     -> y = x0 + o @ w_o (+ b_o)
//   6 LN2        y                     -> yn
//   7 W1 GEMM    yn                    -> h = GELU_tanh(yn @ w_mlp1 (+ b1))
//   8 W2 GEMM    h                     -> out (N, D) = y + h @ w_mlp2 (+ b2)
// Scratch: xn (M, D) | kv (M, 2D) | q, o (N, D) | y (N, D) | yn (N, D) | h (N, F), in the
// accumulation type (y fp32 on the bf16 path), plus the 3xTF32 pieces on the fp32 path.
struct ClsWorkspace {
    bool fast, tf32;
    int acc_dt;
    size_t sz_xn, sz_kv, sz_row, sz_y, sz_h, sz_lo, sz_wt;
    size_t sz_split;   // fp32 K-slice sums of the tensor-core GEMMs over few rows
    size_t total;
};

ClsWorkspace cls_workspace_layout(const BlockArgs& a, const DeviceInfo& dev) {
    ClsWorkspace w;
    const int64_t M = a.N * a.T, N = a.N, D = a.D, F = a.F;
    w.fast = fast_path_ok(a);
    w.acc_dt = w.fast ? DT_BF16 : (a.dt == DT_F64 ? DT_F64 : DT_F32);
    const size_t ea = dt_size(w.acc_dt);
    w.sz_xn = round_up((size_t)(M * D) * ea, 256);
    w.sz_kv = round_up((size_t)(M * 2 * D) * ea, 256);
    w.sz_row = round_up((size_t)(N * D) * ea, 256);
    w.sz_y = round_up((size_t)(N * D) * (w.fast ? 4 : ea), 256);
    w.sz_h = round_up((size_t)(N * F) * ea, 256);
    w.tf32 = !w.fast && a.dt == DT_F32 && tf32x3_supported(M, 2 * D, D, D, a.x) && F % 4 == 0 && tf32_requested();
    w.sz_lo = w.sz_wt = 0;
    if (w.tf32) {
        const int64_t lo = M * D > N * F ? M * D : N * F;
        w.sz_lo = round_up((size_t)lo * 4, 256);
        w.sz_wt = tf32_weight_bytes(D, F);
    }
    w.sz_split = 0;
    if (w.fast) {
        const int64_t sizes[5][3] = {{M, 2 * D, D}, {N, D, D}, {N, F, D}, {N, D, F}, {N, D, D}};
        for (const auto& sz : sizes) {
            const size_t b = (size_t)tc_split_ws_bytes(sz[0], sz[1], sz[2], dev);
            if (b > w.sz_split) w.sz_split = b;
        }
        w.sz_split = round_up(w.sz_split, 256);
    }
    w.total = w.sz_xn + w.sz_kv + 3 * w.sz_row + w.sz_y + w.sz_h + w.sz_lo + w.sz_wt + w.sz_split;
    return w;
}

// Enqueues the CLS-only block on `s`; a.out is (N, D) of out_dtype(a).
cudaError_t launch_block_cls_steps(const BlockArgs& a, const DeviceInfo& dev, cudaStream_t s,
                                   const ClsWorkspace& w, void* ws) {
    const int64_t M = a.N * a.T, N = a.N, T = a.T, D = a.D, F = a.F;
    const int acc = w.acc_dt, xdt = x_dtype(a), odt = out_dtype(a);
    const size_t ea = dt_size(acc);
    uint8_t* p = static_cast<uint8_t*>(ws);
    void* xn = p;  p += w.sz_xn;
    void* kv = p;  p += w.sz_kv;
    void* q = p;   p += w.sz_row;
    void* o = p;   p += w.sz_row;
    void* yn = p;  p += w.sz_row;
    void* y = p;   p += w.sz_y;
    void* h = p;   p += w.sz_h;
    float* split = w.sz_split ? reinterpret_cast<float*>(p) : nullptr;
    p += w.sz_split;
    uint8_t* tail = p;
    void* v_of_kv = static_cast<uint8_t*>(kv) + D * ea;
    cudaError_t e = cudaSuccess;
    auto step = [&](cudaError_t err) {
        if (e == cudaSuccess) e = err;
    };
    const bool qkv_bias = has_qkv_bias(a);
    if (qkv_bias) step(concat_qkv_bias(a, s));
    // [b_k | b_v] of the concatenated [b_q | b_k | b_v]
    const void* bkv = qkv_bias ? static_cast<const uint8_t*>(a.bias_scratch) + D * dt_size(a.dt) : nullptr;
    step(run(K_LN1, s, [&] {
        return launch_layernorm(a.x, xdt, xn, acc, a.ln1_g, a.ln1_b, w.fast ? DT_BF16 : a.dt, M, D, a.eps, s);
    }));
    auto attention = [&] {
        return run(K_CLS_ATTN, s, [&] {
            return launch_attention_cls(q, D, kv, v_of_kv, 2 * D, acc, N, T, D, a.H, o, D, s);
        });
    };
    if (w.fast) {
        TcGemmDesc g;
        std::memset(&g, 0, sizeof(g));
        g.a = xn; g.lda = D;
        g.w[0] = a.w_k; g.w[1] = a.w_v; g.n_w = 2; g.n_per_w = D;
        g.M = M; g.N = 2 * D; g.K = D;
        g.epi = TC_EPI_STORE; g.bias = bkv;
        g.out = kv; g.ldo = 2 * D; g.out_f32 = false;
        g.split_ws = split; g.split_ws_bytes = (int64_t)w.sz_split;
        step(run(K_KV, s, [&] {
            if (tc_gemm_supported(g)) return launch_gemm_tc(g, dev, s);
            SimtGemmDesc sd{xn, DT_BF16, D, a.w_k, DT_BF16, D, a.b_k, DT_BF16, nullptr, 0, 0,
                            kv, DT_BF16, 2 * D, M, D, D, TC_EPI_STORE};
            cudaError_t r = launch_gemm_simt(sd, s);
            sd.w = a.w_v; sd.bias = a.b_v; sd.out = v_of_kv;
            if (r == cudaSuccess) r = launch_gemm_simt(sd, s);
            return r;
        }));
        std::memset(&g, 0, sizeof(g));
        g.a = xn; g.lda = T * D; g.w[0] = a.w_q; g.n_w = 1; g.n_per_w = D;
        g.M = N; g.N = D; g.K = D;
        g.epi = TC_EPI_STORE; g.bias = a.b_q;
        g.out = q; g.ldo = D; g.out_f32 = false;
        g.split_ws = split; g.split_ws_bytes = (int64_t)w.sz_split;
        step(run(K_CLS_Q, s, [&] {
            if (tc_gemm_supported(g)) return launch_gemm_tc(g, dev, s);
            SimtGemmDesc sd{xn, DT_BF16, T * D, a.w_q, DT_BF16, D, a.b_q, DT_BF16, nullptr, 0, 0,
                            q, DT_BF16, D, N, D, D, TC_EPI_STORE};
            return launch_gemm_simt(sd, s);
        }));
        step(attention());
        std::memset(&g, 0, sizeof(g));
        g.a = o; g.lda = D; g.w[0] = a.w_o; g.n_w = 1; g.n_per_w = D;
        g.M = N; g.N = D; g.K = D;
        g.epi = TC_EPI_RESID; g.bias = a.b_o; g.residual = a.x; g.ldr = T * D; g.residual_f32 = xdt == DT_F32;
        g.out = y; g.ldo = D; g.out_f32 = true;
        g.split_ws = split; g.split_ws_bytes = (int64_t)w.sz_split;
        step(run(K_CLS_WO, s, [&] {
            if (tc_gemm_supported(g)) return launch_gemm_tc(g, dev, s);
            SimtGemmDesc sd{o, DT_BF16, D, a.w_o, DT_BF16, D, a.b_o, DT_BF16, a.x, xdt, T * D,
                            y, DT_F32, D, N, D, D, TC_EPI_RESID};
            return launch_gemm_simt(sd, s);
        }));
        step(run(K_CLS_LN2, s, [&] {
            return launch_layernorm(y, DT_F32, yn, DT_BF16, a.ln2_g, a.ln2_b, DT_BF16, N, D, a.eps, s);
        }));
        std::memset(&g, 0, sizeof(g));
        g.a = yn; g.lda = D; g.w[0] = a.w1; g.n_w = 1; g.n_per_w = F;
        g.M = N; g.N = F; g.K = D;
        g.epi = TC_EPI_GELU; g.bias = a.b1;
        g.out = h; g.ldo = F; g.out_f32 = false;
        g.split_ws = split; g.split_ws_bytes = (int64_t)w.sz_split;
        step(run(K_CLS_W1, s, [&] {
            if (tc_gemm_supported(g)) return launch_gemm_tc(g, dev, s);
            SimtGemmDesc sd{yn, DT_BF16, D, a.w1, DT_BF16, F, a.b1, DT_BF16, nullptr, 0, 0,
                            h, DT_BF16, F, N, F, D, TC_EPI_GELU};
            return launch_gemm_simt(sd, s);
        }));
        std::memset(&g, 0, sizeof(g));
        g.a = h; g.lda = F; g.w[0] = a.w2; g.n_w = 1; g.n_per_w = D;
        g.M = N; g.N = D; g.K = F;
        g.epi = TC_EPI_RESID; g.bias = a.b2; g.residual = y; g.ldr = D; g.residual_f32 = true;
        g.out = a.out; g.ldo = D; g.out_f32 = odt == DT_F32;
        g.split_ws = split; g.split_ws_bytes = (int64_t)w.sz_split;
        step(run(K_CLS_W2, s, [&] {
            if (tc_gemm_supported(g)) return launch_gemm_tc(g, dev, s);
            SimtGemmDesc sd{h, DT_BF16, F, a.w2, DT_BF16, D, a.b2, DT_BF16, y, DT_F32, D,
                            a.out, odt, D, N, D, F, TC_EPI_RESID};
            return launch_gemm_simt(sd, s);
        }));
    } else if (w.tf32) {
        float* lo = reinterpret_cast<float*>(tail);
        const Tf32Weights tw = tf32_weight_layout(reinterpret_cast<float*>(tail + w.sz_lo), D, F);
        float *wqkv_t = tw.wqkv_t, *wqkv_lo = tw.wqkv_lo, *wo_t = tw.wo_t, *wo_lo = tw.wo_lo;
        float *w1_t = tw.w1_t, *w1_lo = tw.w1_lo, *w2_t = tw.w2_t, *w2_lo = tw.w2_lo;
        step(run(K_TF32_SPLIT, s, [&] { return tf32_split_weights(a, tw, s); }));
        // out (rows, N) = epi(A (rows, K; row stride lda) @ W + bias [+ res (row stride ldr)])
        auto gemm = [&](const void* A, int64_t rows, int64_t K, int64_t lda, const float* bt, const float* btlo,
                        int64_t Nc, int epi, const void* bias, const void* res, int64_t ldr, void* out) {
            cudaError_t r = launch_split_lo(static_cast<const float*>(A), rows, K, lda, lo, s);
            if (r != cudaSuccess) return r;
            Tf32GemmDesc g{static_cast<const float*>(A), lda, lo, bt, btlo, rows, Nc, K, epi,
                           static_cast<const float*>(bias), static_cast<const float*>(res), ldr,
                           static_cast<float*>(out), Nc};
            return launch_gemm_tf32x3(g, dev, s);
        };
        step(run(K_KV, s, [&] {
            return gemm(xn, M, D, D, wqkv_t + D * D, wqkv_lo + D * D, 2 * D, TC_EPI_STORE, bkv, nullptr, 0, kv);
        }));
        step(run(K_CLS_Q, s, [&] {
            return gemm(xn, N, D, T * D, wqkv_t, wqkv_lo, D, TC_EPI_STORE, a.b_q, nullptr, 0, q);
        }));
        step(attention());
        step(run(K_CLS_WO, s, [&] {
            return gemm(o, N, D, D, wo_t, wo_lo, D, TC_EPI_RESID, a.b_o, a.x, T * D, y);
        }));
        step(run(K_CLS_LN2, s, [&] {
            return launch_layernorm(y, DT_F32, yn, DT_F32, a.ln2_g, a.ln2_b, DT_F32, N, D, a.eps, s);
        }));
        step(run(K_CLS_W1, s, [&] { return gemm(yn, N, D, D, w1_t, w1_lo, F, TC_EPI_GELU, a.b1, nullptr, 0, h); }));
        step(run(K_CLS_W2, s, [&] { return gemm(h, N, F, F, w2_t, w2_lo, D, TC_EPI_RESID, a.b2, y, D, a.out); }));
    } else {
        const int dt = a.dt;
        step(run(K_KV, s, [&] {
            SimtGemmDesc sd{xn, acc, D, a.w_k, dt, D, a.b_k, dt, nullptr, 0, 0, kv, acc, 2 * D, M, D, D, TC_EPI_STORE};
            cudaError_t r = launch_gemm_simt(sd, s);
            sd.w = a.w_v; sd.bias = a.b_v; sd.out = v_of_kv;
            if (r == cudaSuccess) r = launch_gemm_simt(sd, s);
            return r;
        }));
        step(run(K_CLS_Q, s, [&] {
            SimtGemmDesc sd{xn, acc, T * D, a.w_q, dt, D, a.b_q, dt, nullptr, 0, 0, q, acc, D, N, D, D, TC_EPI_STORE};
            return launch_gemm_simt(sd, s);
        }));
        step(attention());
        step(run(K_CLS_WO, s, [&] {
            SimtGemmDesc sd{o, acc, D, a.w_o, dt, D, a.b_o, dt, a.x, xdt, T * D, y, acc, D, N, D, D, TC_EPI_RESID};
            return launch_gemm_simt(sd, s);
        }));
        step(run(K_CLS_LN2, s, [&] {
            return launch_layernorm(y, acc, yn, acc, a.ln2_g, a.ln2_b, dt, N, D, a.eps, s);
        }));
        step(run(K_CLS_W1, s, [&] {
            SimtGemmDesc sd{yn, acc, D, a.w1, dt, F, a.b1, dt, nullptr, 0, 0, h, acc, F, N, F, D, TC_EPI_GELU};
            return launch_gemm_simt(sd, s);
        }));
        step(run(K_CLS_W2, s, [&] {
            SimtGemmDesc sd{h, acc, F, a.w2, dt, D, a.b2, dt, y, acc, D, a.out, odt, D, N, D, F, TC_EPI_RESID};
            return launch_gemm_simt(sd, s);
        }));
    }
    return e;
}

// LayerNorm folded into the GEMMs is opt-in (VIT_LN_FOLD=1): it removes the LN2 pass
// and LN1's normalised copy, but the extra epilogue work in the Wo and W1 GEMMs
// currently costs as much as it saves.
bool ln_fold_requested() {
    static const bool on = [] {
        const char* e = std::getenv("VIT_LN_FOLD");
        return e && e[0] == '1';
    }();
    return on;
}

bool fused_ok(const BlockArgs& a, const DeviceInfo& dev) {
    return ln_fold_requested() && tc_pair_enabled(dev) && row_parts_supported(a.D, a.x);
}

// fuse: 1 / 0 runs the LayerNorm-folded / plain bf16 path (the folded one where the
// shapes and pointers allow it); -1 follows VIT_LN_FOLD.
int enqueue_block(const BlockArgs& a, const DeviceInfo& dev, cudaStream_t s, int fuse = -1) {
    const bool f = fuse < 0 ? fused_ok(a, dev)
                            : fuse == 1 && tc_pair_enabled(dev) && row_parts_supported(a.D, a.x);
    const Workspace w = workspace_layout(a, f);
    DeviceState* st = nullptr;
    int rc = current_device(&st);
    if (rc != VIT_OK) return rc;
    void* ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, w.total, st->pool, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return e == cudaErrorMemoryAllocation ? VIT_ERR_NOMEM : VIT_ERR_CUDA;
    }
    e = launch_block_steps(a, dev, s, w, ws);
    cudaError_t fe = cudaFreeAsync(ws, s);
    if (e == cudaSuccess) e = fe;
    if (e != cudaSuccess) {
        cudaGetLastError();
        return status_from(e);
    }
    if (debug_sync()) {
        if (cudaStreamSynchronize(s) != cudaSuccess) return VIT_ERR_CUDA;
        uint32_t w = 0;
        if (cudaMemcpyFromSymbol(&w, g_err_word, sizeof(w)) != cudaSuccess) return VIT_ERR_CUDA;
        if (w) return VIT_ERR_TIMEOUT;
    }
    return VIT_OK;
}

// ---- scratch for vit_block_noalloc ---------------------------------------------
// For callers that cannot allocate device memory, vit_block_noalloc runs the block with
// its scratch in this fixed, library-owned array instead of the stream-ordered pool.
// Every device that loads the library holds it until the process exits. Kernels never
// read a byte of it before writing it, so nothing needs clearing between calls.
constexpr size_t kNoAllocScratchBytes = (size_t)64 << 20;
__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocState {
    bool ready = false;
    DeviceInfo info;
    void* scratch = nullptr;   // device address of g_noalloc_scratch on this device
};
NoAllocState g_noalloc[kMaxDevices];

// Per-device set-up, on the first call with that device current: device attributes and
// the device addresses of the scratch array and the error word (in host code the
// array's name is only a host-side stand-in, so its address must be looked up).
// Nothing here allocates.
int noalloc_device(NoAllocState** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return VIT_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    NoAllocState& st = g_noalloc[dev];
    if (!st.ready) {
        DeviceInfo info;
        info.device = dev;
        if (cudaDeviceGetAttribute(&info.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&info.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&info.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return VIT_ERR_CUDA;
        void* err = nullptr;
        if (cudaGetSymbolAddress(&err, g_err_word) != cudaSuccess) return VIT_ERR_CUDA;
        info.err_word = static_cast<uint32_t*>(err);
        void* scratch = nullptr;
        if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess || !scratch) return VIT_ERR_CUDA;
        st.info = info;
        st.scratch = scratch;
        st.ready = true;
    }
    *out = &st;
    return VIT_OK;
}

// A stack of L blocks (the last one CLS-only when cls_only) and the optional final
// LayerNorm; the entry points vit_encoder, vit_encoder_cls and vit_block_cls.
int encoder_impl(const void* x, const vit_layer* layers, int64_t L, const void* lnf_g, const void* lnf_b,
                 int final_ln, int64_t N, int64_t T, int64_t D, int64_t F, int64_t H, double eps, int dtype,
                 void* out, void* stream, bool cls_only) {
    if (!layers || L < 1 || L > (1 << 20)) return VIT_ERR_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto layer_args = [&](int64_t l, const void* in, void* o) {
        const vit_layer& ly = layers[l];
        BlockArgs a{in, ly.w_q, ly.w_k, ly.w_v, ly.w_o, ly.w_mlp1, ly.w_mlp2, ly.ln1_g, ly.ln1_b, ly.ln2_g,
                    ly.ln2_b, ly.b1, ly.b2, N, T, D, F, H, eps, dtype, o};
        a.b_q = ly.b_q; a.b_k = ly.b_k; a.b_v = ly.b_v; a.b_o = ly.b_o;
        return a;
    };
    // argument checks of every layer against the caller's x and out (as vit_block_ex),
    // plus the projection biases and the final LayerNorm's gain and bias
    // the caller's output: (N, T, D), or (N, D) with a CLS-only last block
    const size_t ob = (size_t)((cls_only ? N : N * T) * D) * dt_size(dtype);
    for (int64_t l = 0; l < L; ++l) {
        int rc = validate(layer_args(l, x, out), ob);
        if (rc != VIT_OK) return rc;
        const size_t xb = ob, db = (size_t)D * dt_size(dtype);
        const vit_layer& ly = layers[l];
        const void* extra[] = {ly.b_q, ly.b_k, ly.b_v, ly.b_o};
        for (const void* p : extra)
            if (overlaps(out, xb, p, db)) return VIT_ERR_ARG;
        if (overlaps(out, xb, lnf_g, db) || overlaps(out, xb, lnf_b, db)) return VIT_ERR_ARG;
    }
    DeviceState* st = nullptr;
    int rc = current_device(&st);
    if (rc != VIT_OK) return rc;
    const DeviceInfo& dev = st->info;
    const int64_t M = N * T;
    const int sdt = dtype == DT_BF16 ? DT_F32 : dtype;   // residual stream between blocks
    const size_t stream_bytes = round_up((size_t)(M * D) * dt_size(sdt), 256);
    const size_t bias_bytes = round_up((size_t)(3 * D) * dt_size(dtype), 256);
    // scratch: the largest block workspace | two residual-stream buffers | qkv bias
    std::vector<Workspace> wl((size_t)L);
    ClsWorkspace wc{};
    size_t block_bytes = 0;
    void* const probe = reinterpret_cast<void*>(256);   // pool memory is 256-byte aligned
    for (int64_t l = 0; l < L; ++l) {
        BlockArgs a = layer_args(l, l == 0 ? x : probe, probe);
        size_t need;
        if (cls_only && l == L - 1) {
            wc = cls_workspace_layout(a, dev);
            if (!attention_cls_supported(N, T, D, H, wc.acc_dt)) return VIT_ERR_UNSUPPORTED;
            need = wc.total;
        } else {
            wl[(size_t)l] = workspace_layout(a, false);
            need = wl[(size_t)l].total;
        }
        block_bytes = need > block_bytes ? need : block_bytes;
    }
    const size_t total = block_bytes + 2 * stream_bytes + bias_bytes;
    void* ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, total, st->pool, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return e == cudaErrorMemoryAllocation ? VIT_ERR_NOMEM : VIT_ERR_CUDA;
    }
    uint8_t* base = static_cast<uint8_t*>(ws);
    void* r[2] = {base + block_bytes, base + block_bytes + stream_bytes};
    void* bias_scratch = base + block_bytes + 2 * stream_bytes;
    const void* cur = x;
    for (int64_t l = 0; l < L && e == cudaSuccess; ++l) {
        const bool last = l == L - 1;
        void* dst = (last && !final_ln) ? out : r[l & 1];
        BlockArgs a = layer_args(l, cur, dst);
        a.x_dt = l == 0 ? dtype : sdt;
        a.out_dt = (last && !final_ln) ? dtype : sdt;
        a.bias_scratch = bias_scratch;
        if (cls_only && last)
            e = launch_block_cls_steps(a, dev, s, wc, ws);
        else
            e = launch_block_steps(a, dev, s, wl[(size_t)l], ws);
        cur = dst;
    }
    if (e == cudaSuccess && final_ln)
        e = run(K_FINAL_LN, s, [&] {
            return launch_layernorm(cur, sdt, out, dtype, lnf_g, lnf_b, dtype, cls_only ? N : M, D, eps, s);
        });
    cudaError_t fe = cudaFreeAsync(ws, s);
    if (e == cudaSuccess) e = fe;
    if (e != cudaSuccess) {
        cudaGetLastError();
        return status_from(e);
    }
    if (debug_sync()) {
        if (cudaStreamSynchronize(s) != cudaSuccess) return VIT_ERR_CUDA;
        uint32_t w = 0;
        if (cudaMemcpyFromSymbol(&w, g_err_word, sizeof(w)) != cudaSuccess) return VIT_ERR_CUDA;
        if (w) return VIT_ERR_TIMEOUT;
    }
    return VIT_OK;
}

// vit_block_host cuts the batch into chunks of whole sequences so that copies in, blocks
// and copies out of successive chunks overlap on three streams. A block on fewer rows
// fills the GPU less well, so the chunks are few and the first and last (whose copies
// cannot be hidden) are the smallest: one chunk per 10,000 tokens, at most 5, with weights
// 1, 1 / 1, 2, 1 / 1, 3, 3, 1 / 1, 2, 2, 2, 1 (1, 2, 2, 2, 1 measured best for 256 ViT-B/16
// sequences, 4 % ahead of 1, 3, 3, 1). VIT_HOST_SPLIT="w1,w2,..." sets the weights ("1": one
// chunk on the caller's stream).
// Compute streams of the host pipeline: 2 (chunks alternate), or 1 with
// VIT_HOST_COMPUTE_STREAMS=1.
int host_compute_streams() {
    static const int n = [] {
        const char* e = std::getenv("VIT_HOST_COMPUTE_STREAMS");
        return e && e[0] == '1' ? 1 : 2;
    }();
    return n;
}

std::vector<int64_t> host_chunks(int64_t N, int64_t T) {
    static const std::vector<double> forced = [] {
        std::vector<double> w;
        const char* e = std::getenv("VIT_HOST_SPLIT");
        while (e && *e) {
            char* end = nullptr;
            const double v = std::strtod(e, &end);
            if (end == e || !(v > 0)) return std::vector<double>();
            w.push_back(v);
            e = *end == ',' ? end + 1 : end;
            if (*end != ',' && *end != 0) return std::vector<double>();
        }
        return w;
    }();
    std::vector<double> w = forced;
    if (w.empty()) {
        int64_t c = (N * T) / 10000;
        if (c > 5) c = 5;
        if (c < 1) c = 1;
        const double mid = c == 5 ? 2.0 : (double)(c - 1);   // 1,2,1 / 1,3,3,1 / 1,2,2,2,1
        for (int64_t i = 0; i < c; ++i) w.push_back(c > 2 && (i == 0 || i == c - 1) ? 1.0 : mid);
    }
    if ((int64_t)w.size() > N) w.resize((size_t)N);
    double tot = 0;
    for (double v : w) tot += v;
    std::vector<int64_t> sizes;
    int64_t used = 0;
    double acc = 0;
    for (size_t i = 0; i < w.size(); ++i) {
        acc += w[i];
        int64_t upto = i + 1 == w.size() ? N : (int64_t)(N * acc / tot + 0.5);
        const int64_t left = (int64_t)(w.size() - i - 1);
        if (upto > N - left) upto = N - left;   // every later chunk keeps a sequence
        if (upto < used + 1) upto = used + 1;
        sizes.push_back(upto - used);
        used = upto;
    }
    return sizes;
}

// The device's three pipeline streams, created on first use (non-blocking).
int pipeline_streams(DeviceState* st) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (st->h2d) return VIT_OK;
    cudaStream_t a = nullptr, b = nullptr, c = nullptr, b2 = nullptr;
    if (cudaStreamCreateWithFlags(&a, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&b, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&b2, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&c, cudaStreamNonBlocking) != cudaSuccess) {
        if (a) cudaStreamDestroy(a);
        if (b) cudaStreamDestroy(b);
        if (b2) cudaStreamDestroy(b2);
        cudaGetLastError();
        return VIT_ERR_CUDA;
    }
    st->comp = b;
    st->comp2 = b2;
    st->d2h = c;
    st->h2d = a;
    return VIT_OK;
}

}  // namespace
}  // namespace vit

using namespace vit;

// One block's weights held on one device (vit_weights_create): the tensors of a vit_layer
// record copied into one allocation, the concatenated [b_q | b_k | b_v], and with the fold
// the column terms and gain-scaled weights of both folded LayerNorms.
struct vit_weights_s {
    int device = -1, dtype = 0;
    int64_t D = 0, F = 0, H = 0;
    bool fold = false;
    void* mem = nullptr;
    size_t bytes = 0;
    vit_layer w{};              // device pointers into mem; absent terms null
    void* qkv_bias = nullptr;   // (3 D) or null
    FoldTerms terms{};
    float* tf32_wt = nullptr;   // fp32: the weights transposed with their low parts, or null
};

namespace vit {
namespace {

// Prepared weights run on the plain path by default: the folded one is barely faster
// and subtracts mean * c after the product, which loses accuracy when a row's mean is
// large against its spread (VIT_PREPARED_FOLD=1 makes the fold the default).
bool prepared_fold_default() {
    static const bool on = [] {
        const char* e = std::getenv("VIT_PREPARED_FOLD");
        return e && e[0] == '1';
    }();
    return on;
}

BlockArgs prepared_args(const vit_weights* w, const void* x, int64_t N, int64_t T, double eps, void* out) {
    const vit_layer& l = w->w;
    BlockArgs a{x, l.w_q, l.w_k, l.w_v, l.w_o, l.w_mlp1, l.w_mlp2, l.ln1_g, l.ln1_b, l.ln2_g, l.ln2_b,
                l.b1, l.b2, N, T, w->D, w->F, w->H, eps, w->dtype, out};
    a.b_q = l.b_q; a.b_k = l.b_k; a.b_v = l.b_v; a.b_o = l.b_o;
    a.bias_scratch = w->qkv_bias;
    a.qkv_bias_ready = w->qkv_bias != nullptr;
    a.fold_terms = w->fold ? &w->terms : nullptr;
    a.tf32_wt = w->tf32_wt;
    return a;
}

// Host-buffer pipeline of vit_block_host and vit_block_w_host. `h` holds host pointers:
// x and out, and the weights and affine terms unless prepared weights `pw` are given, in
// which case only x and out cross the link.
// Host x in, host out. Synchronous: chunks of whole sequences overlap their copies with
// each other's blocks, and `stream` is synchronised before returning. Asynchronous: the
// whole batch is one chunk and nothing waits on the host; the stages of successive calls
// (copy in, block, copy out) queue on the three library streams, so a call's copies run
// beside the blocks of the calls before and after it.
int host_pipeline(const BlockArgs& h, const vit_weights* pw, void* stream, bool async = false) {
    const int64_t N = h.N, T = h.T, D = h.D, F = h.F;
    const int dtype = h.dt;
    DeviceState* st = nullptr;
    int rc = current_device(&st);
    if (rc != VIT_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t es = dt_size(dtype);
    const size_t xb = (size_t)(N * T * D) * es;
    const size_t sizes[14] = {xb, (size_t)(D * D) * es, (size_t)(D * D) * es, (size_t)(D * D) * es,
                              (size_t)(D * D) * es, (size_t)(D * F) * es, (size_t)(D * F) * es,
                              (size_t)D * es, (size_t)D * es, (size_t)D * es, (size_t)D * es,
                              (size_t)F * es, (size_t)D * es, xb};
    const void* src[13] = {h.x, h.w_q, h.w_k, h.w_v, h.w_o, h.w1, h.w2,
                           h.ln1_g, h.ln1_b, h.ln2_g, h.ln2_b, h.b1, h.b2};
    if (pw)
        for (int i = 1; i < 13; ++i) src[i] = nullptr;   // on the device already
    size_t off[14], total = 0;
    for (int i = 0; i < 14; ++i) {
        off[i] = total;
        if (i < 13 && !src[i]) continue;
        total += round_up(sizes[i], 256);
    }
    const std::vector<int64_t> chunk_n = async ? std::vector<int64_t>{N} : host_chunks(N, T);
    const int64_t chunks = (int64_t)chunk_n.size();
    const bool staged = async || chunks > 1;   // on the library streams
    // copy-in, compute (successive chunks alternate between two streams, so that one
    // chunk's kernels can fill the SMs another's leave idle at their ends), copy-out
    cudaStream_t sh = s, sd = s;
    cudaStream_t scs[2] = {s, s};
    if (staged) {
        rc = pipeline_streams(st);
        if (rc != VIT_OK) return rc;
        sh = st->h2d;
        scs[0] = st->comp;
        scs[1] = !async && host_compute_streams() > 1 ? st->comp2 : st->comp;
        sd = st->d2h;
    }
    void* dmem = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&dmem, total, st->pool, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return status_from(e);
    }
    uint8_t* base = static_cast<uint8_t*>(dmem);
    const void* dev_in[13];
    for (int i = 0; i < 13; ++i) dev_in[i] = src[i] ? base + off[i] : nullptr;
    void* dev_out = base + off[13];
    // events: start, then per chunk x copied and block computed, then copies out done
    std::vector<cudaEvent_t> ev;
    auto new_event = [&](cudaEvent_t* out) {
        cudaError_t r = cudaEventCreateWithFlags(out, cudaEventDisableTiming);
        if (r == cudaSuccess) ev.push_back(*out);
        return r;
    };
    cudaEvent_t start = nullptr, end_d2h = nullptr, end_comp[2] = {nullptr, nullptr};
    if (staged) {
        e = new_event(&start);
        if (e == cudaSuccess) e = cudaEventRecord(start, s);   // after the allocation
        if (e == cudaSuccess) e = cudaStreamWaitEvent(sh, start, 0);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(scs[0], start, 0);
        if (e == cudaSuccess && scs[1] != scs[0]) e = cudaStreamWaitEvent(scs[1], start, 0);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(sd, start, 0);
    }
    // weights and affine terms first (none with prepared weights), then x chunk by chunk
    for (int i = 1; i < 13 && e == cudaSuccess; ++i)
        if (src[i]) e = cudaMemcpyAsync(base + off[i], src[i], sizes[i], cudaMemcpyHostToDevice, sh);
    const size_t seq_bytes = (size_t)(T * D) * es;
    int64_t n0 = 0;
    for (int64_t c = 0; c < chunks && e == cudaSuccess && rc == VIT_OK; ++c) {
        const int64_t nc = chunk_n[(size_t)c];
        const size_t o = (size_t)n0 * seq_bytes, nbytes = (size_t)nc * seq_bytes;
        cudaStream_t sc = scs[c & 1];
        e = cudaMemcpyAsync(base + off[0] + o, static_cast<const uint8_t*>(h.x) + o, nbytes,
                            cudaMemcpyHostToDevice, sh);
        cudaEvent_t in_ready = nullptr, done = nullptr;
        if (staged) {
            if (e == cudaSuccess) e = new_event(&in_ready);
            if (e == cudaSuccess) e = cudaEventRecord(in_ready, sh);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(sc, in_ready, 0);
        }
        if (e != cudaSuccess) break;
        void* const out_c = static_cast<uint8_t*>(dev_out) + o;
        if (pw) {
            rc = enqueue_block(prepared_args(pw, base + off[0] + o, nc, T, h.eps, out_c), st->info, sc,
                               pw->fold ? 1 : 0);
        } else {
            BlockArgs d{base + off[0] + o, dev_in[1], dev_in[2], dev_in[3], dev_in[4], dev_in[5], dev_in[6],
                        dev_in[7], dev_in[8], dev_in[9], dev_in[10], dev_in[11], dev_in[12],
                        nc, T, D, F, h.H, h.eps, dtype, out_c};
            rc = enqueue_block(d, st->info, sc);
        }
        if (rc != VIT_OK) break;
        if (staged) {
            e = new_event(&done);
            if (e == cudaSuccess) e = cudaEventRecord(done, sc);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(sd, done, 0);
            end_comp[c & 1] = done;
        }
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<uint8_t*>(h.out) + o, out_c, nbytes, cudaMemcpyDeviceToHost, sd);
        n0 += nc;
    }
    if (staged) {
        // join: the caller's stream waits for the last copy out and the last block (and
        // so for every copy in), then frees the buffers in its own order
        cudaError_t je = new_event(&end_d2h);
        if (je == cudaSuccess) je = cudaEventRecord(end_d2h, sd);
        if (je == cudaSuccess) je = cudaStreamWaitEvent(s, end_d2h, 0);
        for (int i = 0; i < 2; ++i)
            if (je == cudaSuccess && end_comp[i]) je = cudaStreamWaitEvent(s, end_comp[i], 0);
        if (je == cudaSuccess) {
            cudaEvent_t in_done = nullptr;
            je = new_event(&in_done);
            if (je == cudaSuccess) je = cudaEventRecord(in_done, sh);
            if (je == cudaSuccess) je = cudaStreamWaitEvent(s, in_done, 0);
        }
        if (e == cudaSuccess) e = je;
    }
    cudaError_t fe = cudaFreeAsync(dmem, s);
    // an event destroyed before it completes is released once it does
    cudaError_t se = async ? cudaSuccess : cudaStreamSynchronize(s);
    for (cudaEvent_t x : ev) cudaEventDestroy(x);
    if (rc != VIT_OK) return rc;
    if (e == cudaSuccess) e = fe;
    if (e == cudaSuccess) e = se;
    if (e != cudaSuccess) {
        cudaGetLastError();
        return status_from(e);
    }
    return VIT_OK;
}

}  // namespace
}  // namespace vit


extern "C" {

int vit_block_ex(const void* x, const void* w_q, const void* w_k, const void* w_v, const void* w_o,
                 const void* w_mlp1, const void* w_mlp2, const void* ln1_g, const void* ln1_b,
                 const void* ln2_g, const void* ln2_b, const void* b1, const void* b2, int64_t N,
                 int64_t T, int64_t D, int64_t F, int64_t H, double eps, int dtype, void* out,
                 void* stream) {
    BlockArgs a{x, w_q, w_k, w_v, w_o, w_mlp1, w_mlp2, ln1_g, ln1_b, ln2_g, ln2_b, b1, b2,
                N, T, D, F, H, eps, dtype, out};
    int rc = validate(a);
    if (rc != VIT_OK) return rc;
    DeviceState* st = nullptr;
    rc = current_device(&st);
    if (rc != VIT_OK) return rc;
    return enqueue_block(a, st->info, static_cast<cudaStream_t>(stream));
}

int vit_block(const void* x, const void* w_q, const void* w_k, const void* w_v, const void* w_o,
              const void* w_mlp1, const void* w_mlp2, int64_t N, int64_t T, int64_t D, int64_t F,
              int64_t H, double eps, int dtype, void* out, void* stream) {
    return vit_block_ex(x, w_q, w_k, w_v, w_o, w_mlp1, w_mlp2, nullptr, nullptr, nullptr, nullptr,
                        nullptr, nullptr, N, T, D, F, H, eps, dtype, out, stream);
}

int vit_encoder(const void* x, const vit_layer* layers, int64_t L, const void* lnf_g, const void* lnf_b,
                int final_ln, int64_t N, int64_t T, int64_t D, int64_t F, int64_t H, double eps, int dtype,
                void* out, void* stream) {
    return encoder_impl(x, layers, L, lnf_g, lnf_b, final_ln, N, T, D, F, H, eps, dtype, out, stream, false);
}

int vit_encoder_cls(const void* x, const vit_layer* layers, int64_t L, const void* lnf_g, const void* lnf_b,
                    int final_ln, int64_t N, int64_t T, int64_t D, int64_t F, int64_t H, double eps, int dtype,
                    void* out, void* stream) {
    return encoder_impl(x, layers, L, lnf_g, lnf_b, final_ln, N, T, D, F, H, eps, dtype, out, stream, true);
}

int vit_block_cls(const void* x, const vit_layer* layer, int64_t N, int64_t T, int64_t D, int64_t F, int64_t H,
                  double eps, int dtype, void* out, void* stream) {
    return encoder_impl(x, layer, 1, nullptr, nullptr, 0, N, T, D, F, H, eps, dtype, out, stream, true);
}

int vit_patch_embed(const void* images, int64_t N, int64_t C, int64_t Hi, int64_t Wi, int64_t P, int order,
                    const void* w, const void* b, const void* cls, const void* pos, int64_t D, int dtype,
                    void* tokens, void* stream) {
    if (dtype != DT_F32 && dtype != DT_BF16 && dtype != DT_F64) return VIT_ERR_DTYPE;
    if (!images || !w || !tokens) return VIT_ERR_ARG;
    if (N <= 0 || C <= 0 || Hi <= 0 || Wi <= 0 || P <= 0 || D <= 0 || Hi % P != 0 || Wi % P != 0 ||
        (order != 0 && order != 1))
        return VIT_ERR_ARG;
    if (C * P * P > (1 << 22) || D > (1 << 20) || Hi > (1 << 20) || Wi > (1 << 20) || N > ((int64_t)1 << 31))
        return VIT_ERR_ARG;
    const int64_t NP = (Hi / P) * (Wi / P), K = C * P * P, T = NP + (cls ? 1 : 0), M = N * NP;
    const size_t es = dt_size(dtype);
    const size_t tb = (size_t)(N * T * D) * es;
    const void* in[] = {images, w, b, cls, pos};
    const size_t nb[] = {(size_t)(N * C * Hi * Wi) * es, (size_t)(K * D) * es, (size_t)D * es, (size_t)D * es,
                         (size_t)(T * D) * es};
    for (int i = 0; i < 5; ++i)
        if (overlaps(tokens, tb, in[i], nb[i])) return VIT_ERR_ARG;
    DeviceState* st = nullptr;
    int rc = current_device(&st);
    if (rc != VIT_OK) return rc;
    const DeviceInfo& dev = st->info;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int e_dt = dtype == DT_BF16 ? DT_F32 : dtype;
    const bool tf32 = dtype == DT_F32 && tf32_requested() && tf32x3_supported(M, D, K, K, reinterpret_cast<void*>(256)) &&
                      al16(w) && (!b || al16(b));
    // scratch: A (M x K) | E (M x D) | for the fp32 tensor-core product: A_lo | W^T | W^T_lo
    const size_t sa = round_up((size_t)(M * K) * es, 256), se = round_up((size_t)(M * D) * dt_size(e_dt), 256);
    const size_t slo = tf32 ? round_up((size_t)(M * K) * 4, 256) : 0, swt = tf32 ? round_up((size_t)(D * K) * 4, 256) : 0;
    void* ws = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&ws, sa + se + slo + 2 * swt, st->pool, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return e == cudaErrorMemoryAllocation ? VIT_ERR_NOMEM : VIT_ERR_CUDA;
    }
    uint8_t* base = static_cast<uint8_t*>(ws);
    void* A = base;
    void* E = base + sa;
    e = run(K_PATCHIFY, s, [&] { return launch_patchify(images, dtype, N, C, Hi, Wi, P, order, A, s); });
    if (e == cudaSuccess)
        e = run(K_PATCH_GEMM, s, [&] {
            if (dtype == DT_BF16) {
                TcGemmDesc g;
                std::memset(&g, 0, sizeof(g));
                g.a = A; g.lda = K; g.w[0] = w; g.n_w = 1; g.n_per_w = D;
                g.M = M; g.N = D; g.K = K;
                g.epi = TC_EPI_STORE; g.bias = b;
                g.out = E; g.ldo = D; g.out_f32 = true;
                if (tc_gemm_supported(g)) return launch_gemm_tc(g, dev, s);
            }
            if (tf32) {
                float* lo = reinterpret_cast<float*>(base + sa + se);
                float* wt = reinterpret_cast<float*>(base + sa + se + slo);
                float* wt_lo = reinterpret_cast<float*>(base + sa + se + slo + swt);
                const SplitWtJob job{static_cast<const float*>(w), K, D, D, 0, wt, wt_lo};
                cudaError_t r = launch_split_wt(&job, 1, s);
                if (r == cudaSuccess) r = launch_split_lo(static_cast<const float*>(A), M, K, K, lo, s);
                if (r != cudaSuccess) return r;
                Tf32GemmDesc g{static_cast<const float*>(A), K, lo, wt, wt_lo, M, D, K, TC_EPI_STORE,
                               static_cast<const float*>(b), nullptr, 0, static_cast<float*>(E), D};
                return launch_gemm_tf32x3(g, dev, s);
            }
            SimtGemmDesc sd{A, dtype, K, w, dtype, D, b, dtype, nullptr, 0, 0, E, e_dt, D, M, D, K, TC_EPI_STORE};
            return launch_gemm_simt(sd, s);
        });
    if (e == cudaSuccess)
        e = run(K_PATCH_ASSEMBLE, s, [&] {
            return launch_patch_assemble(E, e_dt, cls, pos, dtype, N, NP, D, tokens, s);
        });
    cudaError_t fe = cudaFreeAsync(ws, s);
    if (e == cudaSuccess) e = fe;
    if (e != cudaSuccess) {
        cudaGetLastError();
        return status_from(e);
    }
    if (debug_sync()) {
        if (cudaStreamSynchronize(s) != cudaSuccess) return VIT_ERR_CUDA;
        uint32_t word = 0;
        if (cudaMemcpyFromSymbol(&word, g_err_word, sizeof(word)) != cudaSuccess) return VIT_ERR_CUDA;
        if (word) return VIT_ERR_TIMEOUT;
    }
    return VIT_OK;
}

int vit_block_host(const void* x_host, const void* w_q_host, const void* w_k_host,
                   const void* w_v_host, const void* w_o_host, const void* w_mlp1_host,
                   const void* w_mlp2_host, const void* ln1_g_host, const void* ln1_b_host,
                   const void* ln2_g_host, const void* ln2_b_host, const void* b1_host,
                   const void* b2_host, int64_t N, int64_t T, int64_t D, int64_t F, int64_t H,
                   double eps, int dtype, void* out_host, void* stream) {
    BlockArgs a{x_host, w_q_host, w_k_host, w_v_host, w_o_host, w_mlp1_host, w_mlp2_host,
                ln1_g_host, ln1_b_host, ln2_g_host, ln2_b_host, b1_host, b2_host,
                N, T, D, F, H, eps, dtype, out_host};
    int rc = validate(a);
    if (rc != VIT_OK) return rc;
    return host_pipeline(a, nullptr, stream);
}

int vit_weights_create(const vit_layer* layer, int from_host, int64_t D, int64_t F, int64_t H, int dtype,
                       int fold, vit_weights** out, void* stream) {
    if (!layer || !out) return VIT_ERR_ARG;
    if (dtype != DT_F32 && dtype != DT_BF16 && dtype != DT_F64) return VIT_ERR_DTYPE;
    if (!layer->w_q || !layer->w_k || !layer->w_v || !layer->w_o || !layer->w_mlp1 || !layer->w_mlp2)
        return VIT_ERR_ARG;
    if (D <= 0 || F <= 0 || H <= 0 || D % H != 0 || D > (1 << 20) || F > (1 << 22)) return VIT_ERR_ARG;
    if (fold < -1 || fold > 1 || (from_host != 0 && from_host != 1)) return VIT_ERR_ARG;
    DeviceState* st = nullptr;
    int rc = current_device(&st);
    if (rc != VIT_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the fold runs on the bf16 tensor-core path with the CTA-pair GEMM
    const bool can_fold = dtype == DT_BF16 && tc_pair_enabled(st->info) && D % 64 == 0 && F % 64 == 0 &&
                          D <= 2048 && row_parts_supported(D, reinterpret_cast<void*>(256));
    if (fold == 1 && !can_fold) return VIT_ERR_UNSUPPORTED;
    const bool use_fold = can_fold && (fold == 1 || (fold == -1 && prepared_fold_default()));
    const size_t es = dt_size(dtype);
    const void* src[16] = {layer->w_q, layer->w_k, layer->w_v, layer->w_o, layer->w_mlp1, layer->w_mlp2,
                           layer->ln1_g, layer->ln1_b, layer->ln2_g, layer->ln2_b, layer->b1, layer->b2,
                           layer->b_q, layer->b_k, layer->b_v, layer->b_o};
    const size_t n[16] = {(size_t)(D * D), (size_t)(D * D), (size_t)(D * D), (size_t)(D * D),
                          (size_t)(D * F), (size_t)(D * F), (size_t)D, (size_t)D, (size_t)D, (size_t)D,
                          (size_t)F, (size_t)D, (size_t)D, (size_t)D, (size_t)D, (size_t)D};
    const bool qkv_bias = layer->b_q || layer->b_k || layer->b_v;
    size_t off[16], total = 0;
    for (int i = 0; i < 16; ++i) {
        off[i] = total;
        if (src[i]) total += round_up(n[i] * es, 256);
    }
    const size_t off_bias = total;
    if (qkv_bias) total += round_up((size_t)(3 * D) * es, 256);
    const size_t off_cols = total;
    if (use_fold) total += round_up((size_t)(2 * 3 * D + 2 * F) * 4, 256);
    const size_t off_wq = total;
    if (use_fold && layer->ln1_g) total += round_up((size_t)(3 * D * D) * 2, 256);
    const size_t off_w1 = total;
    if (use_fold && layer->ln2_g) total += round_up((size_t)(D * F) * 2, 256);
    // fp32 on the 3xTF32 tensor-core path: the weights transposed with their low parts
    const bool prep_tf32 = dtype == DT_F32 && tf32_requested() && D % 4 == 0 && F % 4 == 0;
    const size_t off_wt = total;
    if (prep_tf32) total += tf32_weight_bytes(D, F);
    vit_weights* w = new (std::nothrow) vit_weights;
    if (!w) return VIT_ERR_NOMEM;
    w->device = st->info.device;
    w->dtype = dtype;
    w->D = D; w->F = F; w->H = H;
    w->fold = use_fold;
    w->bytes = total;
    if (cudaMalloc(&w->mem, total) != cudaSuccess) {
        cudaGetLastError();
        delete w;
        return VIT_ERR_NOMEM;
    }
    uint8_t* base = static_cast<uint8_t*>(w->mem);
    const void* dst[16];
    for (int i = 0; i < 16; ++i) dst[i] = src[i] ? base + off[i] : nullptr;
    w->w.w_q = dst[0]; w->w.w_k = dst[1]; w->w.w_v = dst[2]; w->w.w_o = dst[3];
    w->w.w_mlp1 = dst[4]; w->w.w_mlp2 = dst[5]; w->w.ln1_g = dst[6]; w->w.ln1_b = dst[7];
    w->w.ln2_g = dst[8]; w->w.ln2_b = dst[9]; w->w.b1 = dst[10]; w->w.b2 = dst[11];
    w->w.b_q = dst[12]; w->w.b_k = dst[13]; w->w.b_v = dst[14]; w->w.b_o = dst[15];
    cudaError_t e = cudaSuccess;
    const cudaMemcpyKind kind = from_host ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice;
    for (int i = 0; i < 16 && e == cudaSuccess; ++i)
        if (src[i]) e = cudaMemcpyAsync(base + off[i], src[i], n[i] * es, kind, s);
    void* prep = nullptr;
    if (e == cudaSuccess && qkv_bias) {
        w->qkv_bias = base + off_bias;
        BlockArgs a{};
        a.D = D; a.dt = dtype;
        a.b_q = w->w.b_q; a.b_k = w->w.b_k; a.b_v = w->w.b_v;
        a.bias_scratch = w->qkv_bias;
        e = concat_qkv_bias(a, s);
    }
    if (e == cudaSuccess && prep_tf32) {
        w->tf32_wt = reinterpret_cast<float*>(base + off_wt);
        BlockArgs a{};
        a.D = D; a.F = F;
        a.w_q = w->w.w_q; a.w_k = w->w.w_k; a.w_v = w->w.w_v;
        a.w_o = w->w.w_o; a.w1 = w->w.w_mlp1; a.w2 = w->w.w_mlp2;
        const Tf32Weights tw = tf32_weight_layout(w->tf32_wt, D, F);
        e = run(K_TF32_SPLIT, s, [&] { return tf32_split_weights(a, tw, s); });
    }
    if (e == cudaSuccess && use_fold) {
        float* cols = reinterpret_cast<float*>(base + off_cols);
        __nv_bfloat16* wq_scaled = layer->ln1_g ? reinterpret_cast<__nv_bfloat16*>(base + off_wq) : nullptr;
        __nv_bfloat16* w1_scaled = layer->ln2_g ? reinterpret_cast<__nv_bfloat16*>(base + off_w1) : nullptr;
        w->terms.colsum1 = cols;
        w->terms.colbias1 = cols + 3 * D;
        w->terms.colsum2 = cols + 6 * D;
        w->terms.colbias2 = cols + 6 * D + F;
        w->terms.wq_scaled = wq_scaled;
        w->terms.w1_scaled = w1_scaled;
        const size_t p1 = fold_prep_scratch_bytes(3 * D, D), p2 = fold_prep_scratch_bytes(F, D);
        e = cudaMallocFromPoolAsync(&prep, p1 > p2 ? p1 : p2, st->pool, s);
        if (e == cudaSuccess) {
            FoldPrep f1;
            std::memset(&f1, 0, sizeof(f1));
            f1.w[0] = w->w.w_q; f1.w[1] = w->w.w_k; f1.w[2] = w->w.w_v;
            for (int i = 0; i < 3; ++i)
                f1.w_scaled[i] = wq_scaled ? (void*)(wq_scaled + (size_t)i * D * D) : nullptr;
            f1.n_per_w = D; f1.N = 3 * D; f1.K = D;
            f1.gamma = w->w.ln1_g; f1.beta = w->w.ln1_b; f1.bias = w->qkv_bias;
            f1.colsum = cols; f1.colbias = cols + 3 * D;
            e = run(K_FOLD_PREP, s, [&] { return launch_fold_prep(f1, static_cast<float*>(prep), s); });
            FoldPrep f2;
            std::memset(&f2, 0, sizeof(f2));
            f2.w[0] = f2.w[1] = f2.w[2] = w->w.w_mlp1;
            f2.w_scaled[0] = f2.w_scaled[1] = f2.w_scaled[2] = w1_scaled;
            f2.n_per_w = F; f2.N = F; f2.K = D;
            f2.gamma = w->w.ln2_g; f2.beta = w->w.ln2_b; f2.bias = w->w.b1;
            f2.colsum = cols + 6 * D; f2.colbias = cols + 6 * D + F;
            if (e == cudaSuccess)
                e = run(K_FOLD_PREP, s, [&] { return launch_fold_prep(f2, static_cast<float*>(prep), s); });
            cudaError_t fe = cudaFreeAsync(prep, s);
            if (e == cudaSuccess) e = fe;
        }
    }
    cudaError_t se = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = se;
    if (e != cudaSuccess) {
        cudaGetLastError();
        cudaFree(w->mem);
        delete w;
        return e == cudaErrorMemoryAllocation ? VIT_ERR_NOMEM : status_from(e);
    }
    *out = w;
    return VIT_OK;
}

int vit_weights_destroy(vit_weights* w) {
    if (!w) return VIT_OK;
    int prev = -1;
    cudaError_t e = cudaGetDevice(&prev);
    if (e == cudaSuccess && prev != w->device) e = cudaSetDevice(w->device);
    if (e == cudaSuccess) e = cudaFree(w->mem);
    if (prev >= 0 && prev != w->device) cudaSetDevice(prev);
    delete w;
    if (e != cudaSuccess) {
        cudaGetLastError();
        return VIT_ERR_CUDA;
    }
    return VIT_OK;
}

int vit_weights_info(const vit_weights* w, int64_t* D, int64_t* F, int64_t* H, int* dtype, int* fold,
                     int* device) {
    if (!w) return VIT_ERR_ARG;
    if (D) *D = w->D;
    if (F) *F = w->F;
    if (H) *H = w->H;
    if (dtype) *dtype = w->dtype;
    if (fold) *fold = w->fold ? 1 : 0;
    if (device) *device = w->device;
    return VIT_OK;
}

int vit_block_w(const void* x, const vit_weights* w, int64_t N, int64_t T, double eps, void* out,
                void* stream) {
    if (!w) return VIT_ERR_ARG;
    const BlockArgs a = prepared_args(w, x, N, T, eps, out);
    int rc = validate(a);
    if (rc != VIT_OK) return rc;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return VIT_ERR_CUDA;
    if (dev != w->device) return VIT_ERR_ARG;
    DeviceState* st = nullptr;
    rc = current_device(&st);
    if (rc != VIT_OK) return rc;
    return enqueue_block(a, st->info, static_cast<cudaStream_t>(stream), w->fold ? 1 : 0);
}

int vit_block_w_host(const void* x_host, const vit_weights* w, int64_t N, int64_t T, double eps,
                     void* out_host, void* stream) {
    if (!w) return VIT_ERR_ARG;
    const BlockArgs a = prepared_args(w, x_host, N, T, eps, out_host);
    int rc = validate(a);
    if (rc != VIT_OK) return rc;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return VIT_ERR_CUDA;
    if (dev != w->device) return VIT_ERR_ARG;
    return host_pipeline(a, w, stream);
}

int vit_block_w_host_async(const void* x_host, const vit_weights* w, int64_t N, int64_t T, double eps,
                           void* out_host, void* stream) {
    if (!w) return VIT_ERR_ARG;
    const BlockArgs a = prepared_args(w, x_host, N, T, eps, out_host);
    int rc = validate(a);
    if (rc != VIT_OK) return rc;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return VIT_ERR_CUDA;
    if (dev != w->device) return VIT_ERR_ARG;
    return host_pipeline(a, w, stream, true);
}

int vit_layernorm(const void* x, int64_t rows, int64_t D, double eps, const void* gamma,
                  const void* beta, int in_dtype, void* out, int out_dtype, void* stream) {
    if (!x || !out || rows <= 0 || D <= 0) return VIT_ERR_ARG;
    const bool ok = (in_dtype == DT_BF16 && out_dtype == DT_BF16) ||
                    (in_dtype == DT_F32 && (out_dtype == DT_BF16 || out_dtype == DT_F32)) ||
                    (in_dtype == DT_F64 && out_dtype == DT_F64);
    if (!ok) return VIT_ERR_DTYPE;
    if (overlaps(out, (size_t)(rows * D) * dt_size(out_dtype), x, (size_t)(rows * D) * dt_size(in_dtype)))
        return VIT_ERR_ARG;
    DeviceState* st = nullptr;
    int rc = current_device(&st);
    if (rc != VIT_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = run(K_LN1, s, [&] {
        return launch_layernorm(x, in_dtype, out, out_dtype, gamma, beta, out_dtype, rows, D, eps, s);
    });
    if (e != cudaSuccess) {
        cudaGetLastError();
        return status_from(e);
    }
    return VIT_OK;
}

int vit_linear(const void* a, const void* w, const void* bias, const void* residual, int64_t M,
               int64_t K, int64_t N, int epilogue, int dtype, int residual_dtype, void* out,
               int out_dtype, void* stream) {
    if (!a || !w || !out || M <= 0 || K <= 0 || N <= 0) return VIT_ERR_ARG;
    if (epilogue < VIT_EPI_STORE || epilogue > VIT_EPI_RESIDUAL) return VIT_ERR_ARG;
    if ((epilogue == VIT_EPI_RESIDUAL) != (residual != nullptr)) return VIT_ERR_ARG;
    if (dtype != DT_F32 && dtype != DT_BF16 && dtype != DT_F64) return VIT_ERR_DTYPE;
    if (dtype == DT_BF16) {
        if (out_dtype != DT_BF16 && out_dtype != DT_F32) return VIT_ERR_DTYPE;
        if (residual && residual_dtype != DT_BF16 && residual_dtype != DT_F32) return VIT_ERR_DTYPE;
    } else {
        if (out_dtype != dtype || (residual && residual_dtype != dtype)) return VIT_ERR_DTYPE;
    }
    const size_t ob = (size_t)(M * N) * dt_size(out_dtype);
    if (overlaps(out, ob, a, (size_t)(M * K) * dt_size(dtype)) ||
        overlaps(out, ob, w, (size_t)(K * N) * dt_size(dtype)) ||
        overlaps(out, ob, bias, (size_t)N * dt_size(dtype)))
        return VIT_ERR_ARG;
    DeviceState* st = nullptr;
    int rc = current_device(&st);
    if (rc != VIT_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int kind = epilogue == VIT_EPI_GELU ? K_W1 : (epilogue == VIT_EPI_RESIDUAL ? K_W2 : K_QKV);
    cudaError_t e = run(kind, s, [&] {
        if (dtype == DT_BF16) {
            TcGemmDesc g;
            std::memset(&g, 0, sizeof(g));
            g.a = a; g.lda = K; g.w[0] = w; g.n_w = 1; g.n_per_w = N; g.M = M; g.N = N; g.K = K;
            g.epi = epilogue; g.bias = bias; g.residual = residual; g.ldr = N;
            g.residual_f32 = residual_dtype == DT_F32; g.out = out; g.ldo = N;
            g.out_f32 = out_dtype == DT_F32;
            if (tc_gemm_supported(g)) return launch_gemm_tc(g, st->info, s);
        }
        SimtGemmDesc sd{a, dtype, K, w, dtype, N, bias, dtype, residual, residual_dtype, N,
                        out, out_dtype, N, M, N, K, epilogue};
        return launch_gemm_simt(sd, s);
    });
    if (e != cudaSuccess) {
        cudaGetLastError();
        return status_from(e);
    }
    return VIT_OK;
}

int vit_attention(const void* qkv, int64_t N, int64_t T, int64_t D, int64_t H, int dtype, void* o,
                  void* stream) {
    if (!qkv || !o || N <= 0 || T <= 0 || D <= 0 || H <= 0 || D % H != 0) return VIT_ERR_ARG;
    if (dtype != DT_F32 && dtype != DT_BF16 && dtype != DT_F64) return VIT_ERR_DTYPE;
    const size_t es = dt_size(dtype);
    if (overlaps(o, (size_t)(N * T * D) * es, qkv, (size_t)(N * T * 3 * D) * es)) return VIT_ERR_ARG;
    DeviceState* st = nullptr;
    int rc = current_device(&st);
    if (rc != VIT_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = run(K_ATTN, s, [&] {
        if (dtype == DT_BF16 && attention_tc_supported(N, T, D, H, qkv, o))
            return launch_attention_tc(qkv, o, N, T, D, H, st->info, s);
        if (dtype == DT_BF16 && attention_fast_supported(D, H, qkv, o) && (D * 2) % 16 == 0)
            return launch_attention_fast(qkv, o, N, T, D, H, s);
        if (dtype == DT_F32 && attention_f32_supported(N, T, D, H, qkv, o))
            return launch_attention_f32(qkv, o, N, T, D, H, st->info, s);
        return launch_attention_simt(qkv, dtype, o, N, T, D, H, s);
    });
    if (e != cudaSuccess) {
        cudaGetLastError();
        return status_from(e);
    }
    return VIT_OK;
}

int vit_block_noalloc(const void* x, const void* w_q, const void* w_k, const void* w_v,
                      const void* w_o, const void* w_mlp1, const void* w_mlp2, const void* ln1_g,
                      const void* ln1_b, const void* ln2_g, const void* ln2_b, const void* b1,
                      const void* b2, int64_t N, int64_t T, int64_t D, int64_t F, int64_t H,
                      double eps, int dtype, void* out, void* stream) {
    BlockArgs a{x, w_q, w_k, w_v, w_o, w_mlp1, w_mlp2, ln1_g, ln1_b, ln2_g, ln2_b, b1, b2,
                N, T, D, F, H, eps, dtype, out};
    int rc = validate(a);
    if (rc != VIT_OK) return rc;
    NoAllocState* st = nullptr;
    rc = noalloc_device(&st);
    if (rc != VIT_OK) return rc;
    const Workspace w = workspace_layout(a, fused_ok(a, st->info));
    if (w.total > kNoAllocScratchBytes) return VIT_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_block_steps(a, st->info, s, w, st->scratch);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return status_from(e);
    }
    if (debug_sync()) {
        if (cudaStreamSynchronize(s) != cudaSuccess) return VIT_ERR_CUDA;
        uint32_t word = 0;
        if (cudaMemcpyFromSymbol(&word, g_err_word, sizeof(word)) != cudaSuccess) return VIT_ERR_CUDA;
        if (word) return VIT_ERR_TIMEOUT;
    }
    return VIT_OK;
}

const char* vit_status_string(int status) {
    switch (status) {
        case VIT_OK: return "success";
        case VIT_ERR_ARG: return "invalid argument (null pointer, size, H not dividing D, or aliasing)";
        case VIT_ERR_DTYPE: return "unsupported dtype";
        case VIT_ERR_CUDA: return "CUDA call or kernel launch failed";
        case VIT_ERR_TIMEOUT: return "a device-side wait timed out";
        case VIT_ERR_NOMEM: return "scratch allocation failed";
        case VIT_ERR_UNSUPPORTED: return "shape or alignment not supported by this entry point";
    }
    return "unknown status";
}

const char* vit_version(void) { return "vit_block 0.1 (sm_103a)"; }

int64_t vit_launch_count(void) { return g_launches.load(); }

int vit_selftest_wait(int abort_first, void* stream) {
    DeviceState* st = nullptr;
    const int rc = current_device(&st);
    if (rc != VIT_OK) return rc;
    if (launch_selftest_wait(abort_first != 0, st->info.err_word, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess) {
        cudaGetLastError();
        return VIT_ERR_CUDA;
    }
    return VIT_OK;
}

int vit_device_error(uint32_t* word) {
    if (cudaDeviceSynchronize() != cudaSuccess) return VIT_ERR_CUDA;
    uint32_t w = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&w, g_err_word, sizeof(w)) != cudaSuccess) return VIT_ERR_CUDA;
    if (cudaMemcpyToSymbol(g_err_word, &zero, sizeof(zero)) != cudaSuccess) return VIT_ERR_CUDA;
    if (word) *word = w;
    return w ? VIT_ERR_TIMEOUT : VIT_OK;
}

int vit_timing_enable(int enable) {
    g_timing.store(enable != 0);
    return VIT_OK;
}

int vit_timing_collect(void) {
    std::vector<Pending> p;
    {
        std::lock_guard<std::mutex> lk(g_tmu);
        p.swap(g_pending);
    }
    int rc = VIT_OK;
    for (const Pending& q : p) {
        float ms = 0.f;
        if (cudaEventSynchronize(q.b) != cudaSuccess || cudaEventElapsedTime(&ms, q.a, q.b) != cudaSuccess)
            rc = VIT_ERR_CUDA;
        else {
            g_total_ms[q.kind] += ms;
            g_count[q.kind] += 1;
        }
        cudaEventDestroy(q.a);
        cudaEventDestroy(q.b);
    }
    return rc;
}

int vit_timing_kernels(void) { return K_COUNT; }

int vit_timing_read(int k, double* total_ms, int64_t* launches, const char** name) {
    if (k < 0 || k >= K_COUNT) return VIT_ERR_ARG;
    if (total_ms) *total_ms = g_total_ms[k];
    if (launches) *launches = g_count[k];
    if (name) *name = kKernNames[k];
    return VIT_OK;
}

int vit_timing_reset(void) {
    for (int k = 0; k < K_COUNT; ++k) {
        g_total_ms[k] = 0;
        g_count[k] = 0;
    }
    return VIT_OK;
}

}  // extern "C"
