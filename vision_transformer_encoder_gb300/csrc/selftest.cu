// selftest.cu -- a check of the bounded-wait machinery on the device.
//
// Every device-side wait of the library (ptx::mbar_wait_bounded) gives up after a fixed
// number of SM clock cycles, or at once when the kernel's abort flag is set, and the
// kernel then records a bit in the device error word and unwinds. This kernel makes
// such a wait run out on purpose: one thread waits on an mbarrier that nothing will
// complete, with the library's own wait function, and records ERRBIT_SELFTEST when the
// wait gives up. Nothing faults or hangs: the wait ends by its limit (about two
// seconds), or at once in the abort mode.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace vit {
namespace {

__global__ void selftest_wait_kernel(int abort_first, uint32_t* err) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);   // one arrival completes phase 0; none is made
        abort_flag = abort_first;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        volatile int* af = &abort_flag;
        if (!ptx::mbar_wait_bounded(&bar, 0, af) && err) atomicOr(err, ERRBIT_SELFTEST);
    }
}

}  // namespace

cudaError_t launch_selftest_wait(int abort_first, uint32_t* err, cudaStream_t s) {
    selftest_wait_kernel<<<1, 32, 0, s>>>(abort_first, err);
    return cudaGetLastError();
}

}  // namespace vit
