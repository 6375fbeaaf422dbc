// bkv_internal.cuh -- helpers shared by the libbkv.so translation units.
// Host-side status plumbing, launch checks and device queries.  No kernel
// arithmetic lives here.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/bkv.h"

namespace bkv {

// Records the CUDA error text for bkv_last_cuda_error() (thread-local).
void set_cuda_error(cudaError_t e);

// Status after a launch: BKV_ERR_CUDA when the launch itself failed.
inline int launch_status() {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_cuda_error(e);
        return BKV_ERR_CUDA;
    }
    return BKV_OK;
}

// Streaming-multiprocessor count of the current device (cached per device).
int current_sm_count();

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

template <typename T>
__host__ __device__ inline T ceil_div(T a, T b) { return (a + b - 1) / b; }

// Grid size for grid-stride loops: enough blocks to cover n items, capped at
// a few resident waves of the device.
inline unsigned grid_for(int64_t n, int threads, int waves = 8) {
    int64_t blocks = ceil_div<int64_t>(n, threads);
    int64_t cap = (int64_t)current_sm_count() * waves;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return (unsigned)blocks;
}

// Programmatic dependent launch.  Every library kernel starts with
// pdl_wait() before it touches global memory: the wait returns only once the
// preceding kernel in the stream has completed and its writes are visible,
// so launching with the programmatic-serialisation attribute changes no
// result; it lets the launch (and any set-up that needs no global memory)
// overlap the preceding kernel.  pdl_trigger() lets the next such kernel
// launch early; it is always safe for the same reason.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace bkv
