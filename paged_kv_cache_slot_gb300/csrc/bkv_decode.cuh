// bkv_decode.cuh -- shared declarations of the paged decode kernels.
#pragma once

#include <cuda.h>

#include "bkv_internal.cuh"

namespace bkv {

// Everything a decode launch needs; passed by value to every kernel.
struct DecodeArgs {
    const void *q;
    const void *k;
    const void *v;
    const int32_t *bt;
    int64_t bt_stride;
    int32_t bt_cols;
    const int32_t *ctx;
    int32_t max_ctx;
    int32_t num_reqs, q_len, H_q, H_kv, D, bs;
    int64_t total_blocks;
    float scale_log2;  // softmax_scale * log2(e): scores are kept in base 2
    int mask_mode;
    int32_t window;    // sliding window W (> 0): query t sees keys j >= L - q_len + t - W + 1; 0: none
    int32_t cp_world, cp_rank, cp_inter;   // decode context parallelism: this rank's share of the keys
    float *lse;        // optional [num_reqs, q_len, H_q] natural-log sum of exp of the scaled scores
    int dtype;         // BKV_BF16 or BKV_F32: q and out (and the caches unless kv_fp8)
    int kv_fp8;        // caches hold E4M3 codes: a key is code * k_scale (folded into scale_log2)
    float v_scale;     // and a value code * v_scale (applied by the merge); 1 otherwise
    uint8_t *q8;       // FP8 tensor-core path: q split into two E4M3 parts [2][num_reqs * q_len][H_q][128]
    float *qexp;       // and the power of two each query row was divided by first [num_reqs * q_len][H_q]
    int32_t chunk;     // tokens per split-KV partition (multiple of the tile and of bs)
    int32_t n_chunks;  // partitions per request at max_ctx
    int32_t G;         // query heads per KV head
    int32_t nq;        // query rows per KV head: q_len * G, row i = t * G + (h % G)
    int32_t parts;     // partials per unit (slots): 1 for the generic kernel, 2 for the tensor-core one
    int32_t stream_k;  // 1: the tensor-core kernel's stream-K partial slots; 0: the generic kernel's
    int32_t sk_grid;   // tensor-core kernel: CTAs of the stream-K split
    float *ws_o;       // [slots][nq][D] unnormalised partial outputs
    float *ws_ml;      // [slots][nq][2]  (running max in base 2, sum of weights)
    void *out;
    int32_t *err;
};

// Split of each request's context into partitions; identical for the
// workspace query and the decode call.  The workspace holds, in order, a
// 256-byte header (unused, kept for alignment) and the partials of whichever
// kernel runs: the generic kernel's (request, KV head, partition) slots or
// the tensor-core kernel's 2 (sk_grid + num_reqs * H_kv) stream-K slots.
// Decode context parallelism ("ブロック表" 設計動機, DCP interleave): with
// world size W, rank k and interleave I, global position p belongs to rank
// (p / I) % W and is its local key (p / (I W)) I + p % I.  cp_local_len is
// how many of a request's L positions rank k holds; cp_global maps its local
// key j back to the global position the masks use.  W = 1: identity.
__host__ __device__ inline int32_t cp_local_len(const DecodeArgs &a, int32_t L) {
    if (a.cp_world <= 1) return L;
    const int64_t cyc = (int64_t)a.cp_inter * a.cp_world;
    const int64_t full = L / cyc;
    int64_t part = (int64_t)L - full * cyc - (int64_t)a.cp_rank * a.cp_inter;
    part = part < 0 ? 0 : (part > a.cp_inter ? a.cp_inter : part);
    return (int32_t)(full * a.cp_inter + part);
}

__host__ __device__ inline int64_t cp_global(const DecodeArgs &a, int64_t j) {
    if (a.cp_world <= 1) return j;
    const int64_t run = j / a.cp_inter;
    return (run * a.cp_world + a.cp_rank) * a.cp_inter + (j - run * a.cp_inter);
}

// The same for a key of a request shorter than 2^31 positions (always: cache
// lengths are int32), in 32-bit arithmetic.
__host__ __device__ inline int32_t cp_global32(const DecodeArgs &a, int32_t j) {
    if (a.cp_world <= 1) return j;
    const int32_t run = j / a.cp_inter;
    return (run * a.cp_world + a.cp_rank) * a.cp_inter + (j - run * a.cp_inter);
}

// First key position any query of a request of cache length L may see (the
// window of its first query token); 0 without a sliding window.
__host__ __device__ inline int32_t window_lo(const DecodeArgs &a, int32_t L) {
    if (a.window <= 0) return 0;
    const int64_t lo = (int64_t)L - a.q_len - a.window + 1;
    return lo > 0 ? (int32_t)lo : 0;
}

// Tiles of a request in the tensor-core kernel's stream-K schedule: its
// keys' 128-position tiles from the one holding the first visible key.  The
// partition kernel lays all streams' tiles end to end in this count, and the
// merge recomputes each stream's slots from it.
constexpr int kDecodeTile = 128;
__host__ __device__ inline int32_t sk_tiles(const DecodeArgs &a, int32_t ctx_len) {
    const int32_t Lg = ctx_len > a.max_ctx ? a.max_ctx : (ctx_len < 0 ? 0 : ctx_len);
    const int32_t L = cp_local_len(a, Lg);
    return (L + kDecodeTile - 1) / kDecodeTile - window_lo(a, Lg) / kDecodeTile;
}

struct DecodePlan {
    int32_t chunk;
    int32_t n_chunks;
    int32_t nq;
    int32_t sk_grid;
    size_t header_bytes;
    size_t q8_offset;  // workspace offset of the FP8 path's split queries (head_dim 128 only)
    size_t ws_bytes;
};

bool make_decode_plan(int32_t num_reqs, int32_t q_len, int32_t num_q_heads, int32_t num_kv_heads,
                      int32_t head_dim, int32_t block_size, int32_t max_context_len, DecodePlan *plan);

// tcgen05 / TMA partition kernel for bf16, head_dim 128 (bkv_decode_tc.cu).
// prepare_decode_tc decides, from the arguments alone, whether it handles
// this call (and encodes its tensor maps); the partition and merge entry
// points take the same decision independently.
struct TcLaunch {
    CUtensorMap mk, mv, mq;
    int seg_rows;
};
bool prepare_decode_tc(const DecodeArgs &a, TcLaunch *t);
int launch_decode_tc(const DecodeArgs &a, const TcLaunch &t, cudaStream_t stream);
// FP8 caches: the split of q into two E4M3 parts the tensor-core kernel reads.
int launch_q_split_e4m3(const DecodeArgs &a, cudaStream_t stream);

}  // namespace bkv
