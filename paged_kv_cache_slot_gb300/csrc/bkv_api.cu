// bkv_api.cu -- status strings, version and CUDA error plumbing of libbkv.so.
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "bkv_internal.cuh"

namespace bkv {

static thread_local char g_last_error[256] = "";

void set_cuda_error(cudaError_t e) {
    snprintf(g_last_error, sizeof g_last_error, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
}

int current_sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 152;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace bkv

extern "C" const char *bkv_status_string(int status) {
    switch (status) {
        case BKV_OK: return "ok";
        case BKV_ERR_INVALID_ARG: return "invalid argument";
        case BKV_ERR_UNSUPPORTED: return "unsupported dtype or shape";
        case BKV_ERR_CUDA: return "CUDA launch error";
        default: return "unknown status";
    }
}

extern "C" const char *bkv_last_cuda_error(void) { return bkv::g_last_error; }

extern "C" const char *bkv_version(void) { return "bkv 0.3.0 sm_103a"; }
