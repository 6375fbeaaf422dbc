// bkv_ragged.cuh -- shared declarations of the mixed-step (ragged) attention.
#pragma once

#include <cuda.h>

#include "bkv_internal.cuh"

namespace bkv {

// Everything a ragged attention launch needs; passed by value to its kernels.
// Request r's query tokens are rows [qsl[r], qsl[r+1]) of the packed q / out
// ([num_tokens][H_q][D]); token i of r sits at position L_r - q_len_r + i.
struct RaggedArgs {
    const void *q;
    const int32_t *qsl;     // [num_reqs + 1] query_start_loc
    const void *k;
    const void *v;
    const int32_t *bt;
    int64_t bt_stride;
    int32_t bt_cols;
    const int32_t *ctx;
    int32_t max_ctx, max_q;  // host bounds on context_lens and on q_len_r
    int32_t num_reqs;
    int64_t num_tokens;
    int32_t H_q, H_kv, D, bs, G;
    int64_t total_blocks;
    float scale_log2;
    int mask_mode;
    int dtype;
    void *out;
    int32_t *err;
};

// Request r's query tokens [t0, t0 + ql) and cache length L (clamped to the
// host bound); a malformed query_start_loc, or more query tokens than the
// host bound, gives ql = 0 (the request is skipped) and `bad`.
struct RaggedReq {
    int64_t t0;
    int32_t ql, L;
    bool bad;
};

__device__ __forceinline__ RaggedReq ragged_req(const RaggedArgs &a, int r) {
    RaggedReq x;
    const int64_t t0 = __ldg(a.qsl + r), t1 = __ldg(a.qsl + r + 1);
    x.bad = t0 < 0 || t1 < t0 || t1 > a.num_tokens;
    int64_t ql = x.bad ? 0 : t1 - t0;
    if (ql > a.max_q) {
        x.bad = true;
        ql = 0;
    }
    x.t0 = x.bad ? 0 : t0;
    x.ql = (int32_t)ql;
    int32_t L = __ldg(a.ctx + r);
    if (L > a.max_ctx) {
        x.bad = true;
        L = a.max_ctx;
    }
    x.L = L > 0 ? L : 0;
    return x;
}

// tcgen05 / TMA prefill kernel for bf16, head_dim 128 (bkv_ragged_tc.cu).
struct RaggedTc {
    CUtensorMap mk, mv, mq;
    int seg_rows;
    int tok_per_tile;   // query tokens per 128-row tile: 128 / G
};
bool prepare_ragged_tc(const RaggedArgs &a, RaggedTc *t);
int launch_ragged_tc(const RaggedArgs &a, const RaggedTc &t, cudaStream_t stream);

}  // namespace bkv
