// bkv_slot.cuh -- the slot formula, shared by the slot-mapping kernel and the
// fused slot-mapping + cache-write kernel so that both give the same slots.
//
// slot = block_table[r][p / bs] * bs + p % bs ("Padding and Batching with
// Block KV", The Core Formula), -1 for a null or sentinel entry (<= 0,
// Special Block and Slot Values).  Under decode context parallelism
// ("ブロック表" 設計動機: a rank writes real slots only for the tokens it
// owns) position p belongs to rank (p / inter) % world and is stored there at
// the local position (p / (inter * world)) * inter + p % inter; world = 1 is
// the plain formula.
#pragma once

#include <stdint.h>

namespace bkv {

// Slot of token (r, p) for a request index r >= 0; sets *bad for the cases
// counted as errors (r past the batch, p < 0, a position past the table
// width), which give -1.
__device__ __forceinline__ int64_t slot_of(const int32_t *__restrict__ block_table, int32_t num_reqs,
                                           int64_t bt_stride, int32_t bt_cols, int32_t r, int64_t p,
                                           int32_t block_size, int32_t cp_world, int32_t cp_rank, int32_t cp_inter,
                                           bool *bad) {
    *bad = (r >= num_reqs) || (p < 0);
    if (*bad) return -1;
    if (cp_world > 1) {
        const int64_t run = p / cp_inter;
        if (run % cp_world != cp_rank) return -1;
        p = run / cp_world * cp_inter + (p - run * cp_inter);   // local position
    }
    const int64_t lb = p / block_size;
    if (lb >= bt_cols) {
        *bad = true;
        return -1;
    }
    const int64_t b = __ldg(block_table + (int64_t)r * bt_stride + lb);
    return b > 0 ? b * block_size + (p - lb * block_size) : -1;
}

}  // namespace bkv
