/*
 * vit_block.h -- C ABI of the GB300 (sm_103a) ViT encoder block library.
 *
 * The library computes the forward pass of one pre-LayerNorm Vision Transformer
 * encoder block on one GPU, with hand-written CUDA kernels:
 *
 *   xn  = LN1(x)                                  per token, over its D features
 *   Q,K,V = xn @ w_q, xn @ w_k, xn @ w_v          weights stored (in, out)
 *   o   = concat_h softmax(Q_h K_h^T / sqrt(D/H)) V_h     no mask, H heads of D/H
 *   y   = x + o @ w_o
 *   out = y + GELU_tanh(LN2(y) @ w_mlp1 [+ b1]) @ w_mlp2 [+ b2]
 *
 * Definition: "ViT Encoder Block" (crackedaicode), sections "Inputs and output",
 * "Normalize before each stage", "Multi-head attention" and "Feed-forward stage".
 * LN uses population variance (divide by D) and eps is a parameter: that page uses
 * 1e-5, "ViT Encoder Block" (tensortonic.com), "Requirements", uses 1e-6.
 * The optional LN gain/bias pairs and MLP biases are those of "ViT Encoder Block"
 * (ai-engineer-exhaustive), Key Equations, Steps 1, 4 and 5.
 *
 * Conventions shared by every entry point
 *  - Pointers are device pointers unless the name says _host. Arrays are
 *    C-contiguous (row-major) in the stated shapes, all in one element type
 *    `dtype` (a vit_dtype value). The library never writes an input.
 *  - Naming follows the first page: N independent sequences of T tokens of width D;
 *    H heads of width D/H; F the MLP width.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Work is only
 *    enqueued: calls return before the GPU finishes, unless the environment
 *    variable VIT_DEBUG_SYNC=1 is set, in which case each call synchronises the
 *    stream and reports device-side errors in its status.
 *  - Scratch memory is taken from a library-owned, stream-ordered memory pool on the
 *    current device and returned to it on `stream`; the caller owns every pointer it
 *    passes.
 *  - Kernels are launched with programmatic dependent launch: each waits for the
 *    previous kernel in the stream (griddepcontrol.wait) before touching memory and
 *    lets the next one start its set-up early. Stream order is kept for every caller
 *    kernel launched normally. A caller kernel launched after a call with programmatic
 *    stream serialisation must wait on the grid dependency before reading the results,
 *    as CUDA requires of any such launch. VIT_PDL=0 turns it off.
 *  - Every call returns a vit_status (0 = success). No call aborts, traps or throws.
 *  - Results are deterministic: the same inputs give bit-identical outputs.
 */
#ifndef VIT_BLOCK_H
#define VIT_BLOCK_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. VIT_F64 runs on the CUDA-core path only. */
typedef enum { VIT_F32 = 0, VIT_BF16 = 1, VIT_F64 = 2 } vit_dtype;

/* Status codes. */
typedef enum {
    VIT_OK = 0,
    VIT_ERR_ARG = -1,         /* null pointer, non-positive size, H not dividing D, aliasing */
    VIT_ERR_DTYPE = -2,       /* unknown dtype, or a dtype the entry point does not take */
    VIT_ERR_CUDA = -3,        /* a CUDA runtime/driver call or a launch failed */
    VIT_ERR_TIMEOUT = -4,     /* a device-side wait ran out (reported after a sync) */
    VIT_ERR_NOMEM = -5,       /* scratch allocation failed */
    VIT_ERR_UNSUPPORTED = -6  /* a step-level entry point's shape/alignment rule not met */
} vit_status;

/*
 * vit_block -- one encoder block, no LN gain/bias and no biases (the first page).
 *
 *   x        (N, T, D)     input tokens
 *   w_q, w_k, w_v, w_o (D, D)  attention projections, used as  xn @ w
 *   w_mlp1   (D, F), w_mlp2 (F, D)
 *   N, T, D, F, H > 0 with D % H == 0
 *   eps      LN epsilon (> 0 recommended; any finite value is accepted)
 *   dtype    VIT_BF16: bf16 storage, fp32 accumulation; LN statistics, softmax and
 *            GELU in fp32; y kept in fp32; out rounded to bf16 (round-to-nearest-even).
 *            VIT_F32: fp32 storage, LN, softmax and GELU in fp32; the matrix products
 *            as three TF32 tensor-core products per step (hi*hi + hi*lo + lo*hi, about
 *            fp32 accuracy; VIT_FP32_TC=0 selects fp32 CUDA-core products).
 *            VIT_F64: fp64 throughout.
 *   out      (N, T, D), must not overlap any input
 * Errors: VIT_ERR_ARG, VIT_ERR_DTYPE, VIT_ERR_NOMEM, VIT_ERR_CUDA (and VIT_ERR_TIMEOUT
 * under VIT_DEBUG_SYNC=1). On error nothing is guaranteed about `out`.
 */
int vit_block(const void* x, const void* w_q, const void* w_k, const void* w_v,
              const void* w_o, const void* w_mlp1, const void* w_mlp2,
              int64_t N, int64_t T, int64_t D, int64_t F, int64_t H,
              double eps, int dtype, void* out, void* stream);

/*
 * vit_block_ex -- vit_block with the optional affine terms, each nullable:
 *   ln1_g, ln1_b, ln2_g, ln2_b  (D)   LN gain (NULL = 1) and bias (NULL = 0),
 *                                     one pair per LN (the two LNs do not share them)
 *   b1 (F), b2 (D)                    MLP biases (NULL = 0)
 * "ViT Encoder Block" (ai-engineer-exhaustive), Key Equations, Steps 1, 4, 5.
 * Same types, layouts, ownership and errors as vit_block.
 */
int vit_block_ex(const void* x, const void* w_q, const void* w_k, const void* w_v,
                 const void* w_o, const void* w_mlp1, const void* w_mlp2,
                 const void* ln1_g, const void* ln1_b, const void* ln2_g,
                 const void* ln2_b, const void* b1, const void* b2,
                 int64_t N, int64_t T, int64_t D, int64_t F, int64_t H,
                 double eps, int dtype, void* out, void* stream);

/*
 * vit_block_host -- vit_block_ex on HOST arrays: copies the inputs to the device,
 * runs the block and copies `out_host` back, then synchronises `stream` before
 * returning (so out_host is ready on return). Host arrays that are page-locked
 * (cudaHostAlloc / pinned) copy at full link speed; pageable ones work but copy slower.
 * Device buffers come from the library's pool. The optional affine pointers are host
 * pointers or NULL. Errors as vit_block.
 * Large batches (20,000 tokens or more) are cut into up to 5 chunks of whole sequences
 * (sequences are independent: "ViT Encoder Block" (crackedaicode), "Inputs and output");
 * the copy in, the block and the copy out of successive chunks overlap on library-owned
 * streams (one for copies in, two for blocks, one for copies out) that start after, and
 * end before, the work already queued on `stream`. Results are those of one vit_block_ex call on the whole batch, bit for bit.
 */
int vit_block_host(const void* x_host, const void* w_q_host, const void* w_k_host,
                   const void* w_v_host, const void* w_o_host, const void* w_mlp1_host,
                   const void* w_mlp2_host, const void* ln1_g_host, const void* ln1_b_host,
                   const void* ln2_g_host, const void* ln2_b_host, const void* b1_host,
                   const void* b2_host, int64_t N, int64_t T, int64_t D, int64_t F,
                   int64_t H, double eps, int dtype, void* out_host, void* stream);

/*
 * vit_block_noalloc -- vit_block_ex that allocates no device memory.
 *
 * No counterpart on the pages this library follows: it exists for callers that cannot
 * call cudaMalloc or use a memory pool while the block runs -- for example a host
 * application that reserves all device memory up front under a fixed budget, or code
 * running where allocation calls are not allowed. Arguments, layouts, results and
 * errors are those of vit_block_ex; inputs and `out` are still the caller's.
 *
 * Scratch: instead of the stream-ordered pool, the call uses one fixed array of
 * 64 MiB (67,108,864 bytes) that the library keeps in device memory on every GPU that
 * loads it, until the process exits. A call whose scratch would exceed 64 MiB returns
 * VIT_ERR_UNSUPPORTED before launching anything. (Scratch per token: 12 D + 2 F bytes
 * on the bf16 tensor-core path, e.g. 15,360 bytes for D 768 / F 3072, so 4,369
 * tokens; (5 D + F) times the element size on the other paths, plus on the fp32
 * tensor-core path 4 max(D, F) bytes per token and 8 (4 D^2 + 2 D F) bytes for the split
 * weights; more when VIT_LN_FOLD=1 selects the LayerNorm-folded path.) The call makes no
 * cudaMalloc, cudaFree or other allocating call, and nothing in the array needs to be
 * cleared: every scratch byte is written before it is read.
 *
 * The first call on a device looks up the array's device address (a one-time set-up
 * per device, made with that device current); make that first call before any stream
 * capture. All calls share the one array: calls that may overlap on the GPU (on
 * different streams, or from several host threads) race on it and must be ordered by
 * the caller.
 */
int vit_block_noalloc(const void* x, const void* w_q, const void* w_k, const void* w_v,
                      const void* w_o, const void* w_mlp1, const void* w_mlp2,
                      const void* ln1_g, const void* ln1_b, const void* ln2_g,
                      const void* ln2_b, const void* b1, const void* b2,
                      int64_t N, int64_t T, int64_t D, int64_t F, int64_t H,
                      double eps, int dtype, void* out, void* stream);

/* ------------------------------------------------------------------------------
 * Step-level entry points: each runs one stage of the block on its own. They use
 * the same kernels as vit_block and exist for stage-by-stage checking and for
 * callers that compose the stages differently.
 * ------------------------------------------------------------------------------ */

/*
 * vit_encoder -- a stack of L encoder blocks and an optional final LayerNorm.
 *
 * Definition: "ViT Encoder Block" (ai-engineer-exhaustive), introduction (L identical
 * blocks, each with its own weights); lecture transcript (nipunbatra.github.io), Pages
 * 76-77 (block l's whole output is block l+1's input) and Pages 111-112 (the final
 * normalisation of all rows after the stack); the Q, K, V and output-projection biases
 * of Pages 52-53 and 71 (Q = LN(x) W_Q + b_Q, likewise K and V; the joined heads times
 * W_O plus b_O, then the residual). Each block is vit_block_ex plus those biases.
 *
 *   x          (N, T, D) input tokens, `dtype`
 *   layers     HOST array of L vit_layer records (their pointers are device pointers,
 *              `dtype`): the six weights as in vit_block, the other ten nullable
 *              (absent = gain 1, bias 0)
 *   lnf_g, lnf_b  (D) nullable gain and bias of the final LayerNorm
 *   final_ln   1: out = LN(stack output, eps); 0: out = stack output
 *   other arguments as vit_block
 * Between blocks the residual stream is kept in fp32 on the bf16 path (in `dtype`
 * otherwise); only `out` is rounded to `dtype`. Errors as vit_block; VIT_ERR_ARG also for
 * L < 1, a null `layers` or a null weight.
 */
typedef struct {
    const void *w_q, *w_k, *w_v, *w_o, *w_mlp1, *w_mlp2;
    const void *ln1_g, *ln1_b, *ln2_g, *ln2_b;
    const void *b1, *b2;
    const void *b_q, *b_k, *b_v, *b_o;
} vit_layer;

int vit_encoder(const void* x, const vit_layer* layers, int64_t L, const void* lnf_g,
                const void* lnf_b, int final_ln, int64_t N, int64_t T, int64_t D, int64_t F,
                int64_t H, double eps, int dtype, void* out, void* stream);

/* ------------------------------------------------------------------------------
 * Prepared weights: one block's weights held on the device across calls.
 * ------------------------------------------------------------------------------ */

/*
 * vit_weights_create -- copies one block's weights into device memory owned by the
 * library (on the current device) and prepares, once, what depends on the weights alone,
 * so that repeated calls of vit_block_w / vit_block_w_host neither copy nor recompute it:
 *  - the concatenated [b_q | b_k | b_v] of the fused QKV product, when any is given;
 *  - with the LayerNorm fold, the per-column terms of "ViT Encoder Block"
 *    (ai-engineer-exhaustive), Key Equations, Steps 1 and 4 (LayerNorm with gain and bias,
 *    then a linear map): LN(x) @ W = rstd (x @ W' - mean c) + d with W' = diag(gamma) W,
 *    c_j = sum_i W'_ij, d_j = sum_i beta_i W_ij + b_j, mean and rstd = 1/sqrt(var + eps)
 *    of each row of x. Made for LN1 with [w_q | w_k | w_v] (b = [b_q | b_k | b_v]) and
 *    for LN2 with w_mlp1 (b = b1); W' is stored in bf16 and c is summed from the rounded W'.
 *
 *   layer      a vit_layer record (as in vit_encoder): the six weights required, the ten
 *              gains and biases nullable (absent = gain 1, bias 0); all in `dtype`
 *   from_host  1: the record's pointers are host pointers (pinned or pageable);
 *              0: device pointers on the current device
 *   D, F, H, dtype  as vit_block; the handle serves any N, T and eps
 *   fold       1: blocks run with both LayerNorms folded into the QKV and W1 products
 *                 (bf16 with the tensor-core GEMM only; VIT_ERR_UNSUPPORTED otherwise).
 *                 A call whose x is not 16-byte aligned runs the plain path instead.
 *              0: blocks run the plain path: results bit-identical to vit_encoder with
 *                 this one layer and no final LayerNorm (to vit_block_ex when the four
 *                 projection biases are absent)
 *              -1: the library's choice, currently 0 (VIT_PREPARED_FOLD=1 makes it 1
 *                 where available). On a GB300 the folded ViT-B/16 block measured about
 *                 0.5 % faster, too little to make it the default: the fold subtracts
 *                 mean * c after the product, which loses accuracy when a row's mean is
 *                 large against its spread.
 *   out        receives the handle; unchanged on error
 *   stream     the copies and the preparation are enqueued on it, and the call
 *              synchronises it before returning: the caller may then free or change
 *              its arrays
 * Memory: 2 (4 D^2 + 2 D F) bytes of bf16 weights (4 for fp32) plus the gains and biases;
 * with the fold another 8 (3 D + F) bytes and, with LN gains, 2 (3 D^2 + D F) bytes. An
 * fp32 handle (D and F multiples of 4) also holds the weights transposed with their low
 * parts for the 3xTF32 tensor-core products, 8 (4 D^2 + 2 D F) bytes, made once here
 * instead of in every call.
 * Errors: VIT_ERR_ARG (null layer/out/weight, bad sizes, from_host or fold out of range),
 * VIT_ERR_DTYPE, VIT_ERR_NOMEM, VIT_ERR_CUDA, VIT_ERR_UNSUPPORTED.
 */
typedef struct vit_weights_s vit_weights;

int vit_weights_create(const vit_layer* layer, int from_host, int64_t D, int64_t F, int64_t H,
                       int dtype, int fold, vit_weights** out, void* stream);

/* vit_weights_destroy -- frees the handle and its device memory (cudaFree, which waits
 * for work on the device). NULL is accepted. The handle must not be in use. */
int vit_weights_destroy(vit_weights* w);

/* vit_weights_info -- the handle's sizes, dtype, whether it runs the fold (1/0) and its
 * device; each output pointer nullable. VIT_ERR_ARG for a null handle. */
int vit_weights_info(const vit_weights* w, int64_t* D, int64_t* F, int64_t* H, int* dtype,
                     int* fold, int* device);

/*
 * vit_block_w -- one block on prepared weights: vit_block_ex plus the projection biases
 * b_q, b_k, b_v and b_o of the handle's layer (the block of vit_encoder).
 *   x, out    (N, T, D) device arrays in the handle's dtype, on the handle's device (which
 *             must be current); out must not overlap x
 *   eps       LN epsilon, as vit_block
 * Errors as vit_block; VIT_ERR_ARG also for a null handle or another current device.
 */
int vit_block_w(const void* x, const vit_weights* w, int64_t N, int64_t T, double eps,
                void* out, void* stream);

/*
 * vit_block_w_host -- vit_block_w on HOST x and out, with the pipeline of vit_block_host
 * (chunks of whole sequences; copy in, block and copy out overlapped on library streams;
 * `stream` synchronised before returning). Only x and out cross the host link: the
 * weights stay on the device. Results equal vit_block_w's on the same batch, bit for bit.
 */
int vit_block_w_host(const void* x_host, const vit_weights* w, int64_t N, int64_t T, double eps,
                     void* out_host, void* stream);

/*
 * vit_block_w_host_async -- vit_block_w_host without waiting: the copy of x in, the block
 * and the copy of out back are enqueued and the call returns. The work is ordered after
 * everything enqueued on `stream` before the call, and `stream` is ordered after the work
 * (out_host holds the result once `stream` has reached that point: synchronise it or
 * wait on an event recorded on it). Across calls each stage queues on a library stream of
 * its own (one for copies in, one for blocks, one for copies out), so successive calls
 * issued on different streams overlap: the copy in of batch i + 1 and the copy out of
 * batch i - 1 run beside the block of batch i. Calls on one stream run one after another.
 *
 *   x_host, out_host  host arrays as in vit_block_w_host; pinned (page-locked) for the
 *                     copies to run asynchronously (pageable ones work, but a copy out
 *                     to pageable memory returns only when the copy has completed). Both
 *                     stay owned by the caller, must stay valid, and x_host unchanged,
 *                     until `stream` has reached the end of the call's work.
 *   stream            as above; the handle `w` must outlive the enqueued work
 * Returns VIT_OK once everything is enqueued. Argument errors as vit_block_w, with no
 * work enqueued; errors of the enqueued work surface on `stream` and in vit_device_error.
 * Results equal vit_block_w's on the same batch, bit for bit.
 */
int vit_block_w_host_async(const void* x_host, const vit_weights* w, int64_t N, int64_t T, double eps,
                           void* out_host, void* stream);

/*
 * vit_block_cls -- one block computed for the CLS row (row 0 of each sequence) alone.
 *
 * Definition: lecture transcript (nipunbatra.github.io), Page 55 -- when only the CLS
 * token is read after the last block, that block need only produce row 0: its single
 * query is scored against the keys of all T rows and mixes the value rows of all T rows,
 * and the output projection, residual and MLP act on that one row. The result equals row
 * 0 of vit_encoder's single-block output with the same layer.
 *
 *   x      (N, T, D) input tokens, `dtype`, row 0 of each sequence the CLS token
 *   layer  HOST pointer to one vit_layer record (as in vit_encoder)
 *   out    (N, D) `dtype`: the block's output row 0 of each sequence
 * Work and traffic: LN1 and the key and value projections cover all N T rows; the query,
 * attention, output projection, LN2 and MLP cover N rows. Errors as vit_encoder;
 * VIT_ERR_UNSUPPORTED when the T scores of one query do not fit in shared memory
 * (T above about 50,000 in fp32, 25,000 in fp64).
 */
int vit_block_cls(const void* x, const vit_layer* layer, int64_t N, int64_t T, int64_t D,
                  int64_t F, int64_t H, double eps, int dtype, void* out, void* stream);

/*
 * vit_encoder_cls -- vit_encoder whose last block is vit_block_cls: the stack's CLS
 * features. Lecture transcript, Page 55 (CLS-only readout in the final block) and Pages
 * 111-112 (the final normalisation; applied here to the N CLS rows, the only rows read).
 *   out  (N, D) `dtype`: LN(last block's row 0) when final_ln, else that row
 * Other arguments and errors as vit_encoder and vit_block_cls.
 */
int vit_encoder_cls(const void* x, const vit_layer* layers, int64_t L, const void* lnf_g,
                    const void* lnf_b, int final_ln, int64_t N, int64_t T, int64_t D, int64_t F,
                    int64_t H, double eps, int dtype, void* out, void* stream);

/*
 * vit_patch_embed -- the patch-embedding front end: images to tokens.
 *
 * Definition: lecture transcript (nipunbatra.github.io), Pages 96-105 -- non-overlapping
 * P x P patches over the image grid in row-major order, each flattened and projected by
 * one shared linear layer with bias (Pages 96-98, 101), then the CLS row prepended and the
 * positions added (Page 105); "E2E: Tiny Vision Transformer" (mlgrind), forward diagram
 * and patch order.
 *
 *   images   (N, C, Hi, Wi), Hi and Wi multiples of P
 *   order    flatten order inside a patch: 0 = (channel, row, column), the order of
 *            Pages 98 and 101 and of the stride-P convolution; 1 = (row, column, channel),
 *            the E2E page's order
 *   w        (C P P, D) projection, used as  patch_row @ w;  b (D) nullable bias
 *   cls      (D) nullable: prepended as token 0 when given
 *   pos      ((Hi/P)(Wi/P) + [cls], D) nullable: added to every token when given
 *   tokens   (N, T, D) output, T = (Hi/P)(Wi/P) + (cls ? 1 : 0); must not overlap an input
 * dtype as vit_block (bf16: the projection accumulates in fp32 and the position add
 * happens in fp32 before the single rounding). Errors as vit_block; VIT_ERR_ARG also for
 * Hi or Wi not a multiple of P or an unknown order.
 */
int vit_patch_embed(const void* images, int64_t N, int64_t C, int64_t Hi, int64_t Wi, int64_t P,
                    int order, const void* w, const void* b, const void* cls, const void* pos,
                    int64_t D, int dtype, void* tokens, void* stream);

/*
 * vit_layernorm -- out[r, :] = LN(x[r, :]) [* gamma + beta] for r < rows.
 * "ViT Encoder Block" (crackedaicode), "Normalize before each stage".
 *   x     (rows, D) of in_dtype; gamma, beta (D) of out_dtype or NULL
 *   out   (rows, D) of out_dtype
 * Type pairs: (BF16 -> BF16), (F32 -> BF16), (F32 -> F32), (F64 -> F64).
 * Errors: VIT_ERR_ARG, VIT_ERR_DTYPE, VIT_ERR_CUDA.
 */
int vit_layernorm(const void* x, int64_t rows, int64_t D, double eps, const void* gamma,
                  const void* beta, int in_dtype, void* out, int out_dtype, void* stream);

/* Epilogues of vit_linear. */
typedef enum {
    VIT_EPI_STORE = 0,        /* out = a @ w [+ bias]                            */
    VIT_EPI_GELU = 1,         /* out = GELU_tanh(a @ w [+ bias])                 */
    VIT_EPI_RESIDUAL = 2      /* out = residual + a @ w [+ bias]                 */
} vit_epilogue;

/*
 * vit_linear -- out (M, N) = epilogue(a (M, K) @ w (K, N)).
 * "ViT Encoder Block" (crackedaicode): the projections of "Multi-head attention"
 * and the two MLP matrices of "Feed-forward stage"; GELU as defined there.
 *   dtype       element type of a, w, bias
 *   residual    (M, N) of residual_dtype (EPI_RESIDUAL only, else NULL)
 *   out_dtype   element type of out
 * Supported: dtype BF16 with out BF16/F32 and residual BF16/F32 (tensor cores when
 * K % 64 == 0, N % 64 == 0 and every pointer is 16-byte aligned, CUDA cores
 * otherwise); dtype F32 or F64 with out, residual of the same type (CUDA cores).
 * Errors: VIT_ERR_ARG, VIT_ERR_DTYPE, VIT_ERR_CUDA.
 */
int vit_linear(const void* a, const void* w, const void* bias, const void* residual,
               int64_t M, int64_t K, int64_t N, int epilogue, int dtype,
               int residual_dtype, void* out, int out_dtype, void* stream);

/*
 * vit_attention -- unmasked multi-head attention over a fused QKV buffer.
 * "ViT Encoder Block" (crackedaicode), "Multi-head attention"; fused layout
 * [Q | K | V] with head h at columns h*D/H of each block, as in
 * "vision1 reference transcript" (nipunbatra.github.io), Page 106.
 *   qkv  (N, T, 3D) of dtype;  o (N, T, D) of dtype, heads concatenated in order.
 * Errors: VIT_ERR_ARG, VIT_ERR_DTYPE, VIT_ERR_CUDA.
 */
int vit_attention(const void* qkv, int64_t N, int64_t T, int64_t D, int64_t H, int dtype,
                  void* o, void* stream);

/* ------------------------------------------------------------------------------
 * Status, diagnostics and measurement
 * ------------------------------------------------------------------------------ */

/* Static English text for a status code (never NULL). */
const char* vit_status_string(int status);

/*
 * vit_device_error -- synchronise the current device, then read and clear the
 * device error word that kernels set when a bounded wait runs out. Writes the word
 * to *word (0 = no error) and returns VIT_OK, VIT_ERR_TIMEOUT if it was set, or
 * VIT_ERR_CUDA if the synchronisation failed.
 */
int vit_device_error(uint32_t* word);

/*
 * vit_selftest_wait -- exercises the device-side failure detection: one kernel waits
 * on a barrier that nothing completes, with the same bounded wait every kernel of the
 * library uses, and sets a bit (1 << 5) in the device error word when the wait gives up
 * -- after the wait limit (about two seconds of SM clock) or, with abort_first != 0, at
 * once, as when another part of a kernel has already failed. The GPU stays usable.
 * Read the result with vit_device_error. Enqueued on `stream`; returns VIT_ERR_CUDA if
 * the launch fails.
 */
int vit_selftest_wait(int abort_first, void* stream);

/* Number of kernels this library has launched in this process (all devices). */
int64_t vit_launch_count(void);

/*
 * Per-kernel timing. With timing enabled, vit_block records a CUDA event before
 * and after each kernel on the caller's stream. vit_timing_collect synchronises
 * every stream with pending records, adds the elapsed times into per-kernel totals
 * and releases the events. vit_timing_read returns the total milliseconds and the
 * launch count for one kernel index (0 <= k < vit_timing_kernels()) and its name.
 * vit_timing_reset clears the totals. Timing adds two event records per launch.
 */
int vit_timing_enable(int enable);
int vit_timing_collect(void);
int vit_timing_kernels(void);
int vit_timing_read(int k, double* total_ms, int64_t* launches, const char** name);
int vit_timing_reset(void);

/* Library version string. */
const char* vit_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VIT_BLOCK_H */
