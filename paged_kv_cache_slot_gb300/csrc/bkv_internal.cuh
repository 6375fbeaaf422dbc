// bkv_internal.cuh -- helpers shared by the libbkv.so translation units.
// Host-side status plumbing, launch checks and device queries.  No kernel
// arithmetic lives here.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

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

}  // namespace bkv
