// launch.cuh -- kernel launches with programmatic dependent launch.
//
// A kernel launched here may start its CTAs while the previous kernel in the stream is
// still running (CUDA's programmatic stream serialisation). Every kernel launched this way
// calls griddep_wait() (common.cuh) in every CTA before its first access to global memory, which
// blocks until the previous grid has completed and its writes are visible; its own setup
// (barrier initialisation, tensor-memory allocation, tensor-map prefetch) runs before that
// and overlaps the previous kernel's last CTAs. Because each such kernel waits for its
// predecessor before it can complete, the ordering is transitive along the stream.
// VIT_PDL=0 launches without the attribute (plain stream order).
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <utility>

namespace vit {

inline bool pdl_enabled() {
    static const bool on = [] {
        const char* e = std::getenv("VIT_PDL");
        return !(e && e[0] == '0');
    }();
    return on;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// A kernel's dynamic shared-memory limit (cudaFuncSetAttribute) is set per device: raise
// it once on each device the kernel runs on. `done` holds one bit per device ordinal below
// 64 (others are set on every call).
template <typename... KArgs>
cudaError_t set_smem_limit_once(void (*kernel)(KArgs...), int bytes, std::atomic<uint64_t>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t)1 << dev : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

}  // namespace vit
