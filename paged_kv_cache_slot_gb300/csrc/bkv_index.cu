// bkv_index.cu -- slot mapping and manager-to-kernel block expansion.
//
// Both are pure integer gathers over small tables: one thread per output
// element, 64-bit index arithmetic, no shared memory.  Their cost is launch
// latency plus a few bytes per token; the block table they read stays in L2.
#include "bkv_internal.cuh"
#include "bkv_slot.cuh"

namespace bkv {

// slot_mapping[i] for i < max_num_tokens: the slot formula of bkv_slot.cuh
// for real tokens, -1 for the padded tail i >= num_tokens ("ブロック表" 設計動機)
// and for padded requests (r < 0; "Padding and Batching with Block KV", Slot
// ID -1: Padding Tokens).
__global__ void __launch_bounds__(256) slot_mapping_kernel(
    const int32_t *__restrict__ block_table, int32_t num_reqs, int64_t bt_stride, int32_t bt_cols,
    const int32_t *__restrict__ req_indices, const int64_t *__restrict__ positions, int64_t num_tokens,
    int64_t max_num_tokens, int32_t block_size, int32_t cp_world, int32_t cp_rank, int32_t cp_inter,
    int64_t *__restrict__ slot_mapping, int32_t *err_count) {
    pdl_wait();
    pdl_trigger();
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < max_num_tokens; i += step) {
        int64_t slot = -1;
        if (i < num_tokens) {
            const int32_t r = req_indices[i];
            if (r >= 0) {
                bool bad;
                slot = slot_of(block_table, num_reqs, bt_stride, bt_cols, r, positions[i], block_size, cp_world,
                               cp_rank, cp_inter, &bad);
                if (bad && err_count) atomicAdd(err_count, 1);
            }
        }
        slot_mapping[i] = slot;
    }
}

// Manager block m -> kernel blocks m * bpk + t ("ブロック表" 設計動機); an id
// the int32 table cannot hold (m * bpk + t > INT32_MAX) names no block: -1.
__global__ void __launch_bounds__(256) kernel_blocks_kernel(
    const int32_t *__restrict__ mgr, int32_t rows, int64_t mgr_stride, int32_t mgr_cols, int32_t bpk,
    int32_t *__restrict__ out, int64_t out_stride) {
    pdl_wait();
    pdl_trigger();
    const int64_t cols = (int64_t)mgr_cols * bpk;
    const int64_t total = (int64_t)rows * cols;
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += step) {
        const int64_t r = e / cols;
        const int64_t c = e - r * cols;
        const int64_t j = c / bpk;
        const int64_t t = c - j * bpk;
        const int64_t m = __ldg(mgr + r * mgr_stride + j);
        const int64_t id = m * bpk + t;
        out[r * out_stride + c] = (m > 0 && id <= INT32_MAX) ? (int32_t)id : -1;
    }
}

}  // namespace bkv

extern "C" int bkv_compute_slot_mapping(const int32_t *block_table, int32_t num_reqs, int64_t bt_stride,
                                        int32_t bt_cols, const int32_t *req_indices, const int64_t *positions,
                                        int64_t num_tokens, int64_t max_num_tokens, int32_t block_size,
                                        int64_t *slot_mapping, int32_t *err_count, bkv_stream_t stream) {
    return bkv_compute_slot_mapping_cp(block_table, num_reqs, bt_stride, bt_cols, req_indices, positions,
                                       num_tokens, max_num_tokens, block_size, 1, 0, 1, slot_mapping, err_count,
                                       stream);
}

extern "C" int bkv_compute_slot_mapping_cp(const int32_t *block_table, int32_t num_reqs, int64_t bt_stride,
                                           int32_t bt_cols, const int32_t *req_indices, const int64_t *positions,
                                           int64_t num_tokens, int64_t max_num_tokens, int32_t block_size,
                                           int32_t cp_world, int32_t cp_rank, int32_t cp_interleave,
                                           int64_t *slot_mapping, int32_t *err_count, bkv_stream_t stream) {
    if (block_size <= 0 || num_tokens < 0 || max_num_tokens < num_tokens || num_reqs < 0 || bt_cols < 0 ||
        bt_stride < bt_cols || cp_world < 1 || cp_rank < 0 || cp_rank >= cp_world || cp_interleave < 1)
        return BKV_ERR_INVALID_ARG;
    if (max_num_tokens == 0) return BKV_OK;
    if (!slot_mapping) return BKV_ERR_INVALID_ARG;
    if (num_tokens > 0 && (!req_indices || !positions)) return BKV_ERR_INVALID_ARG;
    if (num_tokens > 0 && num_reqs > 0 && bt_cols > 0 && !block_table) return BKV_ERR_INVALID_ARG;
    const int threads = 256;
    const cudaError_t e = bkv::launch_pdl(bkv::slot_mapping_kernel, bkv::grid_for(max_num_tokens, threads), threads, 0,
                                          (cudaStream_t)stream, block_table, num_reqs, bt_stride, bt_cols, req_indices,
                                          positions, num_tokens, max_num_tokens, block_size, cp_world, cp_rank,
                                          cp_interleave, slot_mapping, err_count);
    if (e != cudaSuccess) bkv::set_cuda_error(e);
    return bkv::launch_status();
}

extern "C" int bkv_map_to_kernel_blocks(const int32_t *mgr_table, int32_t rows, int64_t mgr_stride,
                                        int32_t mgr_cols, int32_t block_size, int32_t kernel_block_size,
                                        int32_t *kernel_table, int64_t kernel_stride, bkv_stream_t stream) {
    if (block_size <= 0 || kernel_block_size <= 0 || block_size % kernel_block_size != 0 || rows < 0 ||
        mgr_cols < 0 || mgr_stride < mgr_cols)
        return BKV_ERR_INVALID_ARG;
    const int32_t bpk = block_size / kernel_block_size;
    if (kernel_stride < (int64_t)mgr_cols * bpk) return BKV_ERR_INVALID_ARG;
    const int64_t total = (int64_t)rows * mgr_cols * bpk;
    if (total == 0) return BKV_OK;
    if (!mgr_table || !kernel_table) return BKV_ERR_INVALID_ARG;
    const int threads = 256;
    const cudaError_t e = bkv::launch_pdl(bkv::kernel_blocks_kernel, bkv::grid_for(total, threads), threads, 0,
                                          (cudaStream_t)stream, mgr_table, rows, mgr_stride, mgr_cols, bpk,
                                          kernel_table, kernel_stride);
    if (e != cudaSuccess) bkv::set_cuda_error(e);
    return bkv::launch_status();
}
