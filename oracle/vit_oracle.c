/*
 * vit_oracle.c -- plain float64 CPU oracle of one pre-LayerNorm ViT encoder block.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark may load this code. The product path (the CUDA library) never calls
 * it, shares no code with it, and fails loudly when its own extension is missing.
 *
 * Everything here is the plain definition written out in float64, in the order the
 * pages state it; there is no blocking, fusion or reordering:
 *
 *   "ViT Encoder Block" (crackedaicode), sections "Inputs and output",
 *   "Normalize before each stage", "Multi-head attention", "Feed-forward stage":
 *     xn  = LN(x)                         population variance, eps a parameter
 *     Q,K,V = xn @ w_q, xn @ w_k, xn @ w_v  weights stored (in, out)
 *     per sequence n and head h (columns [h*dh, (h+1)*dh), dh = D/H):
 *       s   = Q_h K_h^T / sqrt(dh);  p = stable softmax over all T keys (no mask)
 *       o_h = p V_h
 *     y   = x + concat_h(o_h) @ w_o
 *     out = y + GELU_tanh(LN(y) @ w_mlp1) @ w_mlp2
 *
 *   "ViT Encoder Block" (ai-engineer-exhaustive), Key Equations, Steps 1, 4 and 5:
 *     optional LN gain/bias (gamma, beta), one pair per LN, and MLP biases b1, b2.
 *     A NULL pointer means "absent": gain 1, bias 0.
 *
 * Every array is C-contiguous float64. Nothing is allocated on the caller's behalf
 * except per-thread scratch, which is freed before return.
 *
 * Pins: tests/test_oracle_pins.py checks every function below against the pages'
 * worked examples, closed forms, invariants and float64 library routines.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* LayerNorm over the last axis of a (rows, D) array.
 * "ViT Encoder Block" (crackedaicode), "Normalize before each stage":
 *   LN(x) = (x - mean) / sqrt(variance + eps), variance divides by D.
 * Gain/bias: "ViT Encoder Block" (ai-engineer-exhaustive), Key Equations, Step 1. */
void oracle_layernorm(const double* x, int64_t rows, int64_t D, double eps,
                      const double* gamma, const double* beta, double* out)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double* xr = x + r * D;
        double* o = out + r * D;
        double mean = 0.0;
        for (int64_t j = 0; j < D; ++j) mean += xr[j];
        mean /= (double)D;
        double var = 0.0;
        for (int64_t j = 0; j < D; ++j) {
            double d = xr[j] - mean;
            var += d * d;
        }
        var /= (double)D;
        double denom = sqrt(var + eps);
        for (int64_t j = 0; j < D; ++j) {
            double v = (xr[j] - mean) / denom;
            if (gamma) v = gamma[j] * v;
            if (beta) v = v + beta[j];
            o[j] = v;
        }
    }
}

/* tanh-approximation GELU.
 * "ViT Encoder Block" (crackedaicode), "Feed-forward stage":
 *   GELU(z) = 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3))). */
double oracle_gelu_tanh(double z)
{
    const double pi = 3.14159265358979323846;
    return 0.5 * z * (1.0 + tanh(sqrt(2.0 / pi) * (z + 0.044715 * z * z * z)));
}

void oracle_gelu_tanh_array(const double* z, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_gelu_tanh(z[i]);
}

/* C (M, N) = A (M, K) @ W (K, N) [+ bias (N)].
 * Each C[m][n] is the sum over k = 0..K-1, in ascending k, of A[m][k] * W[k][n];
 * the bias, when present, is added after the sum. */
void oracle_matmul(const double* A, const double* W, const double* bias,
                   int64_t M, int64_t K, int64_t N, double* C)
{
    for (int64_t m = 0; m < M; ++m) {
        double* c = C + m * N;
        for (int64_t n = 0; n < N; ++n) c[n] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = A[m * K + k];
            const double* w = W + k * N;
            for (int64_t n = 0; n < N; ++n) c[n] += a * w[n];
        }
        if (bias)
            for (int64_t n = 0; n < N; ++n) c[n] += bias[n];
    }
}

/* Stable softmax of each row of a (rows, n) array: subtract the row maximum,
 * exponentiate, divide by the sum. "ViT Encoder Block" (crackedaicode),
 * "Multi-head attention" ("Use stable softmax across key positions"). */
void oracle_softmax_rows(const double* s, int64_t rows, int64_t n, double* p)
{
    for (int64_t r = 0; r < rows; ++r) {
        const double* sr = s + r * n;
        double* pr = p + r * n;
        double m = sr[0];
        for (int64_t u = 1; u < n; ++u)
            if (sr[u] > m) m = sr[u];
        double z = 0.0;
        for (int64_t u = 0; u < n; ++u) {
            pr[u] = exp(sr[u] - m);
            z += pr[u];
        }
        for (int64_t u = 0; u < n; ++u) pr[u] = pr[u] / z;
    }
}

/* Multi-head attention of ONE sequence, no mask.
 * Q, K, V, O are (T, D); head h owns columns [h*dh, (h+1)*dh), dh = D/H.
 * scratch must hold 2*T doubles.
 * "ViT Encoder Block" (crackedaicode), "Multi-head attention":
 *   scores = Q_h K_h^T / sqrt(D/H); weights = softmax(scores, axis=-1);
 *   head_output = weights V_h; heads concatenated in their original order. */
static void attention_one_sequence(const double* Q, const double* K, const double* V,
                                   int64_t T, int64_t D, int64_t H, double* O,
                                   double* scratch)
{
    const int64_t dh = D / H;
    const double scale = sqrt((double)dh);
    double* s = scratch;
    double* p = scratch + T;
    for (int64_t h = 0; h < H; ++h) {
        const int64_t c0 = h * dh;
        for (int64_t t = 0; t < T; ++t) {
            for (int64_t u = 0; u < T; ++u) {
                double dot = 0.0;
                for (int64_t c = 0; c < dh; ++c)
                    dot += Q[t * D + c0 + c] * K[u * D + c0 + c];
                s[u] = dot / scale;
            }
            oracle_softmax_rows(s, 1, T, p);
            for (int64_t c = 0; c < dh; ++c) {
                double acc = 0.0;
                for (int64_t u = 0; u < T; ++u) acc += p[u] * V[u * D + c0 + c];
                O[t * D + c0 + c] = acc;
            }
        }
    }
}

/* Attention over N sequences laid out (N, T, D). */
void oracle_attention(const double* Q, const double* K, const double* V,
                      int64_t N, int64_t T, int64_t D, int64_t H, double* O)
{
    double* scratch = (double*)malloc(sizeof(double) * 2 * (size_t)T);
    for (int64_t n = 0; n < N; ++n)
        attention_one_sequence(Q + n * T * D, K + n * T * D, V + n * T * D, T, D, H,
                               O + n * T * D, scratch);
    free(scratch);
}

/* The whole block over N independent sequences (x is (N, T, D)).
 *
 * Optional stage outputs (each NULL or the stated shape) expose the intermediate
 * values for stage-by-stage comparison:
 *   xn (N,T,D), qkv (N,T,3D) laid out [Q | K | V], o (N,T,D) heads concatenated,
 *   y (N,T,D), yn (N,T,D), g (N,T,F) = GELU output.
 *
 * Returns 0 on success, -1 on invalid sizes (non-positive, or H not dividing D),
 * -2 if scratch allocation fails. nthreads <= 0 uses the OpenMP default. */
/* The block with the optional projection biases of the lecture transcript
 * (nipunbatra.github.io), Pages 52-53 (Q = LN(x) W_Q + b_Q, likewise K and V) and
 * Page 71 (the joined heads times W_O plus b_O, then the residual). NULL biases are
 * absent (zero). */
int oracle_vit_block_full(const double* x, const double* w_q, const double* w_k,
                          const double* w_v, const double* w_o, const double* w_mlp1,
                          const double* w_mlp2, const double* ln1_g, const double* ln1_b,
                          const double* ln2_g, const double* ln2_b, const double* b1,
                          const double* b2, const double* b_q, const double* b_k,
                          const double* b_v, const double* b_o, int64_t N, int64_t T,
                          int64_t D, int64_t F, int64_t H, double eps, double* out,
                          double* st_xn, double* st_qkv, double* st_o, double* st_y,
                          double* st_yn, double* st_g, int nthreads)
{
    if (N <= 0 || T <= 0 || D <= 0 || F <= 0 || H <= 0 || D % H != 0) return -1;
    int failed = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t n = 0; n < N; ++n) {
        const size_t TD = (size_t)(T * D), TF = (size_t)(T * F);
        double* buf = (double*)malloc(sizeof(double) * (8 * TD + 2 * TF + 2 * (size_t)T));
        if (!buf) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
            continue;
        }
        double *xn = buf, *q = xn + TD, *k = q + TD, *v = k + TD, *o = v + TD;
        double *a = o + TD, *y = a + TD, *yn = y + TD, *z = yn + TD, *g = z + TF;
        double* scratch = g + TF;
        const double* xs = x + (size_t)n * TD;
        double* os = out + (size_t)n * TD;

        /* 1. xn = LN1(x) */
        oracle_layernorm(xs, T, D, eps, ln1_g, ln1_b, xn);
        /* 2. Q, K, V = xn @ w_q [+ b_q], xn @ w_k [+ b_k], xn @ w_v [+ b_v] */
        oracle_matmul(xn, w_q, b_q, T, D, D, q);
        oracle_matmul(xn, w_k, b_k, T, D, D, k);
        oracle_matmul(xn, w_v, b_v, T, D, D, v);
        /* 3. per-head unmasked attention, heads concatenated in order */
        attention_one_sequence(q, k, v, T, D, H, o, scratch);
        /* 4. y = x + o @ w_o [+ b_o]  (the residual adds to the un-normalised x) */
        oracle_matmul(o, w_o, b_o, T, D, D, a);
        for (size_t i = 0; i < TD; ++i) y[i] = xs[i] + a[i];
        /* 5. yn = LN2(y)  (LN of y, not of x) */
        oracle_layernorm(y, T, D, eps, ln2_g, ln2_b, yn);
        /* 6. g = GELU_tanh(yn @ w_mlp1 [+ b1]) */
        oracle_matmul(yn, w_mlp1, b1, T, D, F, z);
        oracle_gelu_tanh_array(z, (int64_t)TF, g);
        /* 7. out = y + g @ w_mlp2 [+ b2] */
        oracle_matmul(g, w_mlp2, b2, T, F, D, a);
        for (size_t i = 0; i < TD; ++i) os[i] = y[i] + a[i];

        if (st_xn) memcpy(st_xn + (size_t)n * TD, xn, sizeof(double) * TD);
        if (st_qkv) {
            double* dst = st_qkv + (size_t)n * 3 * TD;
            for (int64_t t = 0; t < T; ++t) {
                memcpy(dst + (size_t)t * 3 * D, q + (size_t)t * D, sizeof(double) * D);
                memcpy(dst + (size_t)t * 3 * D + D, k + (size_t)t * D, sizeof(double) * D);
                memcpy(dst + (size_t)t * 3 * D + 2 * D, v + (size_t)t * D, sizeof(double) * D);
            }
        }
        if (st_o) memcpy(st_o + (size_t)n * TD, o, sizeof(double) * TD);
        if (st_y) memcpy(st_y + (size_t)n * TD, y, sizeof(double) * TD);
        if (st_yn) memcpy(st_yn + (size_t)n * TD, yn, sizeof(double) * TD);
        if (st_g) memcpy(st_g + (size_t)n * TF, g, sizeof(double) * TF);
        free(buf);
    }
    return failed ? -2 : 0;
}

/* The block as the primary statement defines it: no projection biases. */
int oracle_vit_block(const double* x, const double* w_q, const double* w_k,
                     const double* w_v, const double* w_o, const double* w_mlp1,
                     const double* w_mlp2, const double* ln1_g, const double* ln1_b,
                     const double* ln2_g, const double* ln2_b, const double* b1,
                     const double* b2, int64_t N, int64_t T, int64_t D, int64_t F,
                     int64_t H, double eps, double* out, double* st_xn, double* st_qkv,
                     double* st_o, double* st_y, double* st_yn, double* st_g,
                     int nthreads)
{
    return oracle_vit_block_full(x, w_q, w_k, w_v, w_o, w_mlp1, w_mlp2, ln1_g, ln1_b, ln2_g,
                                 ln2_b, b1, b2, NULL, NULL, NULL, NULL, N, T, D, F, H, eps,
                                 out, st_xn, st_qkv, st_o, st_y, st_yn, st_g, nthreads);
}

/* A stack of L blocks and an optional final LayerNorm: "ViT Encoder Block"
 * (ai-engineer-exhaustive), introduction (L identical blocks, each with its own
 * weights); lecture transcript (nipunbatra.github.io), Pages 76-77 (block l's output is
 * block l+1's input) and Pages 111-112 (twelve blocks, then the final normalisation of
 * all rows); "E2E: Tiny Vision Transformer" (mlgrind), forward diagram (final LN).
 * layers: L x 16 pointers per layer, in the order w_q, w_k, w_v, w_o, w_mlp1, w_mlp2,
 * ln1_g, ln1_b, ln2_g, ln2_b, b1, b2, b_q, b_k, b_v, b_o (the last ten may be NULL).
 * final_ln != 0 applies LN(., eps) with the nullable gain lnf_g and bias lnf_b. */
int oracle_vit_encoder(const double* x, const double* const* layers, int64_t L,
                       const double* lnf_g, const double* lnf_b, int final_ln, int64_t N,
                       int64_t T, int64_t D, int64_t F, int64_t H, double eps, double* out,
                       int nthreads)
{
    if (L <= 0 || N <= 0 || T <= 0 || D <= 0) return -1;
    const size_t ND = (size_t)(N * T * D);
    double* r0 = (double*)malloc(sizeof(double) * ND);
    double* r1 = (double*)malloc(sizeof(double) * ND);
    if (!r0 || !r1) {
        free(r0);
        free(r1);
        return -2;
    }
    const double* cur = x;
    int rc = 0;
    for (int64_t l = 0; l < L && rc == 0; ++l) {
        const double* const* w = layers + (size_t)l * 16;
        double* nxt = (l & 1) ? r1 : r0;
        rc = oracle_vit_block_full(cur, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7], w[8],
                                   w[9], w[10], w[11], w[12], w[13], w[14], w[15], N, T, D, F,
                                   H, eps, nxt, NULL, NULL, NULL, NULL, NULL, NULL, nthreads);
        cur = nxt;
    }
    if (rc == 0) {
        if (final_ln)
            oracle_layernorm(cur, N * T, D, eps, lnf_g, lnf_b, out);
        else
            memcpy(out, cur, sizeof(double) * ND);
    }
    free(r0);
    free(r1);
    return rc;
}

/* CLS-only readout of one block: lecture transcript (nipunbatra.github.io), Page 55 --
 * when only the CLS token (row 0 of each sequence) is read after the last block, that
 * block need only produce row 0: its single query is scored against the keys of all T
 * rows and mixes the value rows of all T rows; the rest of the block then acts on that
 * one row. Per sequence:
 *   xn = LN1(x) for all T rows;  K = xn W_K (+ b_K), V = xn W_V (+ b_V) for all T rows;
 *   q = xn[0] W_Q (+ b_Q);  per head h: s_u = q_h . K_h[u] / sqrt(D/H) for u < T,
 *   p = softmax(s), o_h = sum_u p_u V_h[u];
 *   y0 = x[0] + o W_O (+ b_O);  out[n] = y0 + GELU_tanh(LN2(y0) W1 (+ b1)) W2 (+ b2).
 * out is (N, D). Returns as oracle_vit_block_full. */
int oracle_vit_block_cls(const double* x, const double* w_q, const double* w_k,
                         const double* w_v, const double* w_o, const double* w_mlp1,
                         const double* w_mlp2, const double* ln1_g, const double* ln1_b,
                         const double* ln2_g, const double* ln2_b, const double* b1,
                         const double* b2, const double* b_q, const double* b_k,
                         const double* b_v, const double* b_o, int64_t N, int64_t T,
                         int64_t D, int64_t F, int64_t H, double eps, double* out,
                         int nthreads)
{
    if (N <= 0 || T <= 0 || D <= 0 || F <= 0 || H <= 0 || D % H != 0) return -1;
    int failed = 0;
    const int64_t dh = D / H;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t n = 0; n < N; ++n) {
        const size_t TD = (size_t)(T * D);
        double* buf = (double*)malloc(sizeof(double) * (3 * TD + 6 * (size_t)D + 2 * (size_t)F +
                                                         2 * (size_t)T));
        if (!buf) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
            continue;
        }
        double *xn = buf, *keys = xn + TD, *vals = keys + TD, *q0 = vals + TD, *o0 = q0 + D;
        double *a0 = o0 + D, *y0 = a0 + D, *yn0 = y0 + D, *m0 = yn0 + D, *z0 = m0 + D, *g0 = z0 + F;
        double *sc = g0 + F, *pw = sc + T;
        const double* xs = x + (size_t)n * TD;

        /* LN1 and the keys and values of every row */
        oracle_layernorm(xs, T, D, eps, ln1_g, ln1_b, xn);
        oracle_matmul(xn, w_k, b_k, T, D, D, keys);
        oracle_matmul(xn, w_v, b_v, T, D, D, vals);
        /* the query of the CLS row (row 0) alone */
        oracle_matmul(xn, w_q, b_q, 1, D, D, q0);
        /* per head: the T scores of that query, softmax, weighted sum of all T values */
        for (int64_t h = 0; h < H; ++h) {
            const int64_t first = h * dh;
            for (int64_t u = 0; u < T; ++u) {
                double dot = 0.0;
                for (int64_t c = 0; c < dh; ++c) dot += q0[first + c] * keys[u * D + first + c];
                sc[u] = dot / sqrt((double)dh);
            }
            oracle_softmax_rows(sc, 1, T, pw);
            for (int64_t c = 0; c < dh; ++c) {
                double acc = 0.0;
                for (int64_t u = 0; u < T; ++u) acc += pw[u] * vals[u * D + first + c];
                o0[first + c] = acc;
            }
        }
        /* y0 = x[0] + o W_O (+ b_O), then the MLP of the one row with its residual */
        oracle_matmul(o0, w_o, b_o, 1, D, D, a0);
        for (int64_t j = 0; j < D; ++j) y0[j] = xs[j] + a0[j];
        oracle_layernorm(y0, 1, D, eps, ln2_g, ln2_b, yn0);
        oracle_matmul(yn0, w_mlp1, b1, 1, D, F, z0);
        oracle_gelu_tanh_array(z0, F, g0);
        oracle_matmul(g0, w_mlp2, b2, 1, F, D, m0);
        for (int64_t j = 0; j < D; ++j) out[(size_t)n * D + j] = y0[j] + m0[j];
        free(buf);
    }
    return failed ? -2 : 0;
}

/* The stack of oracle_vit_encoder with its last block replaced by the CLS-only readout
 * (oracle_vit_block_cls) and the final LayerNorm applied to the N CLS rows: out is
 * (N, D). The first L - 1 blocks are oracle_vit_encoder without its final LayerNorm. */
int oracle_vit_encoder_cls(const double* x, const double* const* layers, int64_t L,
                           const double* lnf_g, const double* lnf_b, int final_ln, int64_t N,
                           int64_t T, int64_t D, int64_t F, int64_t H, double eps, double* out,
                           int nthreads)
{
    if (L <= 0 || N <= 0 || T <= 0 || D <= 0) return -1;
    double* body = NULL;
    double* c = (double*)malloc(sizeof(double) * (size_t)(N * D));
    if (L > 1) body = (double*)malloc(sizeof(double) * (size_t)(N * T * D));
    if (!c || (L > 1 && !body)) {
        free(body);
        free(c);
        return -2;
    }
    int rc = 0;
    if (L > 1)
        rc = oracle_vit_encoder(x, layers, L - 1, NULL, NULL, 0, N, T, D, F, H, eps, body, nthreads);
    if (rc == 0) {
        const double* const* last = layers + (size_t)(L - 1) * 16;
        rc = oracle_vit_block_cls(L > 1 ? body : x, last[0], last[1], last[2], last[3], last[4],
                                  last[5], last[6], last[7], last[8], last[9], last[10], last[11],
                                  last[12], last[13], last[14], last[15], N, T, D, F, H, eps, c,
                                  nthreads);
    }
    if (rc == 0) {
        if (final_ln)
            oracle_layernorm(c, N, D, eps, lnf_g, lnf_b, out);
        else
            memcpy(out, c, sizeof(double) * (size_t)(N * D));
    }
    free(body);
    free(c);
    return rc;
}

/* Patch embedding front end. Images (N, C, Hi, Wi), non-overlapping P x P patches taken
 * in row-major order over the (Hi/P, Wi/P) grid, each flattened to C P P values and
 * projected: tokens = patches @ w (+ b), w of shape (C P P, D); then, with cls non-NULL,
 * the cls row is prepended; with pos non-NULL, pos (T, D) is added to every row
 * (T = patches + (cls ? 1 : 0)). Flatten order inside a patch:
 *   order 0: (c, p1, p2) -- channel by channel, each row by row: lecture transcript
 *            (nipunbatra.github.io), Pages 98 and 101 (unfold; the same as the stride-P
 *            convolution of Pages 99-100);
 *   order 1: (p1, p2, c) -- "E2E: Tiny Vision Transformer" (mlgrind), "Patch order".
 * CLS prepend and position add: lecture transcript, Page 105; "E2E: Tiny Vision
 * Transformer", forward diagram. */
int oracle_patch_embed(const double* images, int64_t N, int64_t C, int64_t Hi, int64_t Wi,
                       int64_t P, int order, const double* w, const double* b,
                       const double* cls, const double* pos, int64_t D, double* out)
{
    if (N <= 0 || C <= 0 || P <= 0 || D <= 0 || Hi % P != 0 || Wi % P != 0 || (order != 0 && order != 1))
        return -1;
    const int64_t gh = Hi / P, gw = Wi / P, NP = gh * gw, K = C * P * P;
    const int64_t T = NP + (cls ? 1 : 0), off = cls ? 1 : 0;
    double* patch = (double*)malloc(sizeof(double) * (size_t)K);
    if (!patch) return -2;
    for (int64_t n = 0; n < N; ++n) {
        double* o = out + (size_t)n * T * D;
        if (cls)
            for (int64_t d = 0; d < D; ++d) o[d] = cls[d];
        for (int64_t py = 0; py < gh; ++py)
            for (int64_t px = 0; px < gw; ++px) {
                /* flatten this patch */
                for (int64_t c = 0; c < C; ++c)
                    for (int64_t i = 0; i < P; ++i)
                        for (int64_t j = 0; j < P; ++j) {
                            const double v = images[(((size_t)n * C + c) * Hi + py * P + i) * Wi + px * P + j];
                            const int64_t k = order == 0 ? (c * P + i) * P + j : (i * P + j) * C + c;
                            patch[k] = v;
                        }
                /* project: row = patch @ w (+ b) */
                double* row = o + (size_t)(off + py * gw + px) * D;
                for (int64_t d = 0; d < D; ++d) row[d] = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    const double a = patch[k];
                    const double* wk = w + (size_t)k * D;
                    for (int64_t d = 0; d < D; ++d) row[d] += a * wk[d];
                }
                if (b)
                    for (int64_t d = 0; d < D; ++d) row[d] += b[d];
            }
        if (pos)
            for (int64_t t = 0; t < T; ++t)
                for (int64_t d = 0; d < D; ++d) o[(size_t)t * D + d] += pos[(size_t)t * D + d];
    }
    free(patch);
    return 0;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
