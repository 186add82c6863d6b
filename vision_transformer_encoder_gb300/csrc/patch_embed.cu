// patch_embed.cu -- the patch-embedding front end: patchify and token assembly.
//
// Images (N, C, Hi, Wi) are cut into non-overlapping P x P patches in row-major order over
// the (Hi/P, Wi/P) grid; each patch becomes one row of C P P values (the GEMM's A
// operand), flattened
//   order 0: channel by channel, each channel row by row -- lecture transcript
//            (nipunbatra.github.io), Pages 98 and 101 (the stride-P convolution's order);
//   order 1: (row, column, channel) -- "E2E: Tiny Vision Transformer" (mlgrind), patch order.
// After the projection (a GEMM with bias, run by the library's GEMM kernels into an fp32
// or dtype buffer E), the assembly writes tokens (N, T, D): row 0 the CLS vector when
// given, then the patch rows, plus the positions when given (lecture transcript, Page 105),
// summed in the accumulation type and rounded once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace vit {
namespace {

template <typename T>
__device__ __forceinline__ float ld_f(const T* p, int64_t i);
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p, int64_t i) {
    return __bfloat162float(p[i]);
}
template <>
__device__ __forceinline__ float ld_f<float>(const float* p, int64_t i) {
    return p[i];
}

// One thread per element of the patch matrix (N * NP rows of K = C P P), grid-stride.
template <typename T>
__global__ void patchify_kernel(const T* __restrict__ im, int64_t N, int C, int Hi, int Wi, int P, int order,
                                T* __restrict__ A) {
    const int gw = Wi / P, NP = (Hi / P) * gw, K = C * P * P;
    const int64_t total = N * NP * (int64_t)K;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = e / K;
        const int k = (int)(e - row * K);
        const int64_t n = row / NP;
        const int pidx = (int)(row - n * NP);
        const int py = pidx / gw, px = pidx - py * gw;
        int c, i, j;
        if (order == 0) {
            c = k / (P * P);
            const int r = k - c * P * P;
            i = r / P;
            j = r - i * P;
        } else {
            const int ij = k / C;
            c = k - ij * C;
            i = ij / P;
            j = ij - i * P;
        }
        A[e] = im[((n * C + c) * Hi + (int64_t)py * P + i) * Wi + (int64_t)px * P + j];
    }
}

// Order 0 with P and Wi multiples of V (the elements in 16 bytes) and 16-byte aligned
// buffers: each thread moves V consecutive elements of one patch row with one 16-byte
// load and store, 32-bit index arithmetic. grid.y / z = patch row (n, py, px), the
// x-threads cover its K / V vectors.
template <int V>
__global__ void patchify_vec_kernel(const uint4* __restrict__ im, int C, int Hi, int Wi, int P, int NP,
                                    int gw, int64_t rows, uint4* __restrict__ A) {
    const int K8 = C * P * P / V, P8 = P / V;
    const int64_t row64 = blockIdx.y + 65535ll * blockIdx.z;   // n * NP + patch
    if (row64 >= rows) return;
    const unsigned row = (unsigned)row64;
    const unsigned n = row / (unsigned)NP, pidx = row - n * (unsigned)NP;
    const int py = (int)(pidx / (unsigned)gw), px = (int)(pidx - (unsigned)py * gw);
    const int64_t img = (int64_t)n * C * Hi * Wi / V;
    for (int k8 = blockIdx.x * blockDim.x + threadIdx.x; k8 < K8; k8 += gridDim.x * blockDim.x) {
        const int c = k8 / (P * P8), r = k8 - c * P * P8;
        const int i = r / P8, j8 = r - i * P8;
        A[(int64_t)row * K8 + k8] = im[img + (((int64_t)c * Hi + py * P + i) * Wi + px * P) / V + j8];
    }
}

// tokens[n, t] = (t == 0 and cls ? cls : E[n, t - off]) + pos[t]: one CTA per token row
// (grid.x = t, grid.y / z = n), four columns per thread.
template <typename T>
__global__ void assemble_rows_kernel(const float* __restrict__ E, const T* __restrict__ cls,
                                     const T* __restrict__ pos, int64_t N, int NP, int D, T* __restrict__ out) {
    const int off = cls ? 1 : 0, TT = NP + off;
    const int t = blockIdx.x;
    const int64_t n = blockIdx.y + 65535ll * blockIdx.z;
    if (n >= N) return;
    const float* erow = E + ((n * NP) + (t - off)) * (int64_t)D;
    T* orow = out + (n * TT + t) * (int64_t)D;
    for (int d = 4 * threadIdx.x; d < D; d += 4 * blockDim.x) {
        float v[4];
        if (t < off) {
#pragma unroll
            for (int q = 0; q < 4; ++q) v[q] = ld_f(cls, d + q);
        } else {
            const float4 e4 = *reinterpret_cast<const float4*>(erow + d);
            v[0] = e4.x; v[1] = e4.y; v[2] = e4.z; v[3] = e4.w;
        }
        if (pos) {
#pragma unroll
            for (int q = 0; q < 4; ++q) v[q] += ld_f(pos, (int64_t)t * D + d + q);
        }
        if constexpr (sizeof(T) == 2) {
            uint2 w;
            w.x = pack_bf16x2(v[0], v[1]);
            w.y = pack_bf16x2(v[2], v[3]);
            *reinterpret_cast<uint2*>(orow + d) = w;
        } else {
            *reinterpret_cast<float4*>(orow + d) = make_float4(v[0], v[1], v[2], v[3]);
        }
    }
}

// tokens[n, t] = (t == 0 and cls ? cls : E[n, t - off]) + pos[t]; one thread per element.
template <typename T, typename E_T>
__global__ void assemble_kernel(const E_T* __restrict__ E, const T* __restrict__ cls, const T* __restrict__ pos,
                                int64_t N, int NP, int D, T* __restrict__ out) {
    const int off = cls ? 1 : 0, TT = NP + off;
    const int64_t total = N * TT * (int64_t)D;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t nt = e / D;
        const int d = (int)(e - nt * D);
        const int64_t n = nt / TT;
        const int t = (int)(nt - n * TT);
        float v;
        if (t < off)
            v = ld_f(cls, d);
        else
            v = (float)E[((n * NP) + (t - off)) * (int64_t)D + d];
        if (pos) v += ld_f(pos, (int64_t)t * D + d);
        if constexpr (sizeof(T) == 2)
            out[e] = __float2bfloat16_rn(v);
        else
            out[e] = v;
    }
}

// fp64 assembly (E in fp64)
__global__ void assemble_f64_kernel(const double* __restrict__ E, const double* __restrict__ cls,
                                    const double* __restrict__ pos, int64_t N, int NP, int D,
                                    double* __restrict__ out) {
    const int off = cls ? 1 : 0, TT = NP + off;
    const int64_t total = N * TT * (int64_t)D;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t nt = e / D;
        const int d = (int)(e - nt * D);
        const int64_t n = nt / TT;
        const int t = (int)(nt - n * TT);
        double v = t < off ? cls[d] : E[((n * NP) + (t - off)) * (int64_t)D + d];
        if (pos) v += pos[(int64_t)t * D + d];
        out[e] = v;
    }
}

unsigned blocks_for(int64_t total) {
    const int64_t b = (total + 255) / 256;
    return (unsigned)(b < 65536 * 4 ? b : 65536 * 4);
}

}  // namespace

cudaError_t launch_patchify(const void* images, int dt, int64_t N, int64_t C, int64_t Hi, int64_t Wi, int64_t P,
                            int order, void* A, cudaStream_t s) {
    const int64_t total = N * (Hi / P) * (Wi / P) * C * P * P;
    if (total <= 0) return cudaSuccess;
    const int64_t rows = N * (Hi / P) * (Wi / P);
    const int V = dt == DT_BF16 ? 8 : dt == DT_F32 ? 4 : 2;   // elements per 16 bytes
    if (order == 0 && P % V == 0 && Wi % V == 0 && (reinterpret_cast<uintptr_t>(images) & 15) == 0 &&
        (reinterpret_cast<uintptr_t>(A) & 15) == 0 && rows <= 65535ll * 65535ll && rows < (1ll << 32) &&
        N * C * Hi * Wi < (1ll << 40)) {
        const int K8 = (int)(C * P * P / V);
        const int tx = K8 < 128 ? ((K8 + 31) / 32) * 32 : 128;
        const dim3 grid((unsigned)((K8 + tx - 1) / tx), (unsigned)(rows < 65535 ? rows : 65535),
                        (unsigned)((rows + 65534) / 65535));
        const int NP = (int)((Hi / P) * (Wi / P)), gw = (int)(Wi / P);
        const uint4* im = static_cast<const uint4*>(images);
        uint4* a = static_cast<uint4*>(A);
        if (V == 8)
            patchify_vec_kernel<8><<<grid, tx, 0, s>>>(im, (int)C, (int)Hi, (int)Wi, (int)P, NP, gw, rows, a);
        else if (V == 4)
            patchify_vec_kernel<4><<<grid, tx, 0, s>>>(im, (int)C, (int)Hi, (int)Wi, (int)P, NP, gw, rows, a);
        else
            patchify_vec_kernel<2><<<grid, tx, 0, s>>>(im, (int)C, (int)Hi, (int)Wi, (int)P, NP, gw, rows, a);
        return cudaGetLastError();
    }
    if (dt == DT_BF16)
        patchify_kernel<__nv_bfloat16><<<blocks_for(total), 256, 0, s>>>(
            static_cast<const __nv_bfloat16*>(images), N, (int)C, (int)Hi, (int)Wi, (int)P, order,
            static_cast<__nv_bfloat16*>(A));
    else if (dt == DT_F32)
        patchify_kernel<float><<<blocks_for(total), 256, 0, s>>>(static_cast<const float*>(images), N, (int)C,
                                                                 (int)Hi, (int)Wi, (int)P, order,
                                                                 static_cast<float*>(A));
    else
        patchify_kernel<double><<<blocks_for(total), 256, 0, s>>>(static_cast<const double*>(images), N, (int)C,
                                                                  (int)Hi, (int)Wi, (int)P, order,
                                                                  static_cast<double*>(A));
    return cudaGetLastError();
}

cudaError_t launch_patch_assemble(const void* E, int e_dt, const void* cls, const void* pos, int dt, int64_t N,
                                  int64_t NP, int64_t D, void* out, cudaStream_t s) {
    const int64_t total = N * (NP + (cls ? 1 : 0)) * D;
    if (total <= 0) return cudaSuccess;
    if (dt == DT_F64) {
        assemble_f64_kernel<<<blocks_for(total), 256, 0, s>>>(static_cast<const double*>(E),
                                                              static_cast<const double*>(cls),
                                                              static_cast<const double*>(pos), N, (int)NP, (int)D,
                                                              static_cast<double*>(out));
    } else if (D % 4 == 0 && (reinterpret_cast<uintptr_t>(E) & 15) == 0 && N <= 65535ll * 65535ll &&
               NP + 1 <= 0x7fffffff && (reinterpret_cast<uintptr_t>(out) & (dt == DT_BF16 ? 7 : 15)) == 0) {
        if (e_dt != DT_F32) return cudaErrorInvalidValue;
        const dim3 grid((unsigned)(NP + (cls ? 1 : 0)), (unsigned)(N < 65535 ? N : 65535), (unsigned)((N + 65534) / 65535));
        const int tx = D / 4 < 256 ? ((D / 4 + 31) / 32) * 32 : 256;
        if (dt == DT_BF16)
            assemble_rows_kernel<__nv_bfloat16><<<grid, tx, 0, s>>>(
                static_cast<const float*>(E), static_cast<const __nv_bfloat16*>(cls),
                static_cast<const __nv_bfloat16*>(pos), N, (int)NP, (int)D, static_cast<__nv_bfloat16*>(out));
        else
            assemble_rows_kernel<float><<<grid, tx, 0, s>>>(static_cast<const float*>(E), static_cast<const float*>(cls),
                                                            static_cast<const float*>(pos), N, (int)NP, (int)D,
                                                            static_cast<float*>(out));
    } else if (dt == DT_BF16) {
        if (e_dt != DT_F32) return cudaErrorInvalidValue;
        assemble_kernel<__nv_bfloat16, float><<<blocks_for(total), 256, 0, s>>>(
            static_cast<const float*>(E), static_cast<const __nv_bfloat16*>(cls),
            static_cast<const __nv_bfloat16*>(pos), N, (int)NP, (int)D, static_cast<__nv_bfloat16*>(out));
    } else {
        assemble_kernel<float, float><<<blocks_for(total), 256, 0, s>>>(
            static_cast<const float*>(E), static_cast<const float*>(cls), static_cast<const float*>(pos), N,
            (int)NP, (int)D, static_cast<float*>(out));
    }
    return cudaGetLastError();
}

}  // namespace vit
