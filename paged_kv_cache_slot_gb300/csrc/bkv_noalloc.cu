// bkv_noalloc.cu -- bkv_paged_decode_noalloc: the paged decode with its
// split-KV scratch in a fixed device array owned by the library, for callers
// that cannot allocate device memory (see include/bkv.h for who they are).
//
// The array is a file-scope __device__ variable.  Its name seen from host
// code is only a host-side stand-in, never a device address, so the entry
// point looks the real address up with cudaGetSymbolAddress (the call's
// device current) and hands that pointer to bkv_paged_decode as its
// workspace.  Outside stream capture the lookup is repeated on every call,
// so the address is always the one of the current context (a device reset
// between calls creates a new one); while the call's stream is being
// captured the address found by the last call outside capture on that
// device is used, so that no lookup runs inside the capture.  Nothing here
// allocates.
#include <mutex>

#include "bkv_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[BKV_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void *g_scratch_addr[64] = {};   // last address found outside capture, per device ordinal

// Device address of the scratch array on the current device for a call on
// `stream`, or an error.
int scratch_address(cudaStream_t stream, void **addr) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        bkv::set_cuda_error(e);
        return BKV_ERR_CUDA;
    }
    if (dev < 0 || dev >= 64) return BKV_ERR_UNSUPPORTED;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        (void)cudaGetLastError();   // an illegal query under another thread's capture: treat as capturing
        cs = cudaStreamCaptureStatusActive;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (cs == cudaStreamCaptureStatusNone) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess || !p) {
            bkv::set_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
            return BKV_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    } else if (!g_scratch_addr[dev]) {
        // the first call on this device came under capture: no lookup is made there
        bkv::set_cuda_error(cudaErrorStreamCaptureUnsupported);
        return BKV_ERR_CUDA;
    }
    *addr = g_scratch_addr[dev];
    return BKV_OK;
}

}  // namespace

extern "C" int bkv_paged_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                        const int32_t *block_table, int64_t bt_stride, int32_t bt_cols,
                                        const int32_t *context_lens, int32_t max_context_len, int32_t num_reqs,
                                        int32_t q_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                        int32_t block_size, int64_t total_blocks, float softmax_scale, int mask_mode,
                                        int dtype, void *out, int32_t *err_count, bkv_stream_t stream) {
    const size_t need = bkv_paged_decode_workspace_size(num_reqs, q_len, num_q_heads, num_kv_heads, head_dim,
                                                        block_size, max_context_len);
    if (need == 0) return BKV_ERR_INVALID_ARG;
    if (need > BKV_NOALLOC_SCRATCH_BYTES) return BKV_ERR_UNSUPPORTED;   // larger than the fixed array
    void *scratch = nullptr;
    const int rc = scratch_address((cudaStream_t)stream, &scratch);
    if (rc != BKV_OK) return rc;
    return bkv_paged_decode(q, k_cache, v_cache, block_table, bt_stride, bt_cols, context_lens, max_context_len,
                            num_reqs, q_len, num_q_heads, num_kv_heads, head_dim, block_size, total_blocks,
                            softmax_scale, mask_mode, dtype, out, scratch, BKV_NOALLOC_SCRATCH_BYTES, err_count,
                            stream);
}
