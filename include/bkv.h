/*
 * bkv.h -- C ABI of libbkv.so, the GB300 (sm_103a) paged (block) KV cache
 * hot path: slot mapping, manager-to-kernel block expansion, the KV cache
 * scatter (bf16 / fp32, or quantised to FP8), GQA paged decode attention
 * with a split-KV merge, mixed-step attention, and the context-parallel
 * slot filter and merge.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer argument is a DEVICE pointer owned by the caller, unless
 *   stated otherwise.  Arrays are dense row-major unless a stride is given
 *   (strides count elements, not bytes).  The library allocates no memory.
 * - Every call is asynchronous: it validates its scalar arguments on the
 *   host, enqueues kernels on `stream` (0 = the legacy default stream) and
 *   returns.  Nothing is read from device memory on the host.
 * - Return value: BKV_OK, or an error status.  BKV_ERR_INVALID_ARG and
 *   BKV_ERR_UNSUPPORTED are decided on the host before anything is enqueued;
 *   BKV_ERR_CUDA means a launch failed (text from bkv_last_cuda_error()).
 * - Bad DATA in device memory (a block id past the cache, a slot past the
 *   cache, a position past the table width, a request index past the batch)
 *   never faults: the token or block is treated as padding (-1) and, when
 *   `err_count` is non-null, *err_count (a device int32) is incremented.
 * - The KV cache layout of record is (total_blocks, block_size,
 *   num_kv_heads, head_dim) for K and for V, separately.
 *
 * Sources: "Padding and Batching with Block KV" (vllm-neuron design notes),
 * "ブロック表" (vLLM v1 BlockTable walkthrough), "KV Caching with vLLM" and
 * "Decode Context-Length Bucketing" (Neuron docs).  Each declaration names the
 * section that defines its operation.
 */
#ifndef BKV_H_
#define BKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *bkv_stream_t; /* same object as cudaStream_t */

enum {
    BKV_OK = 0,
    BKV_ERR_INVALID_ARG = 1, /* a scalar argument or null pointer is invalid */
    BKV_ERR_UNSUPPORTED = 2, /* dtype / head_dim / shape this library does not handle */
    BKV_ERR_CUDA = 3         /* a CUDA launch failed; see bkv_last_cuda_error() */
};

enum { BKV_BF16 = 0, BKV_F32 = 1 };

enum {
    BKV_MASK_CAUSAL = 0, /* query t of a request of cache length L is at L - q_len + t */
    BKV_MASK_ALL = 1     /* every query sees every cached position < L */
};

/* Static text for a status code. */
const char *bkv_status_string(int status);

/* Text of the last CUDA error seen by this library in this thread ("" if none). */
const char *bkv_last_cuda_error(void);

/* Library version, e.g. "bkv 0.3.0 sm_103a". */
const char *bkv_version(void);

/*
 * bkv_compute_slot_mapping
 *   Defined by "Padding and Batching with Block KV", Slot Mapping: From
 *   Position to Cache Location (The Core Formula; Slot Mapping Computation),
 *   Special Block and Slot Values, and "ブロック表" 設計動機 (the padded tail of
 *   the slot buffer written with PAD for CUDA-graph reuse).
 *
 *   For i in [0, max_num_tokens):
 *     slot_mapping[i] = block_table[r * bt_stride + p / block_size] * block_size
 *                       + p % block_size,   r = req_indices[i], p = positions[i]
 *   and slot_mapping[i] = -1 when i >= num_tokens, r < 0 (a padded request),
 *   the table entry is <= 0 (the null block 0 or the sentinel -1), r >=
 *   num_reqs, p < 0, or p / block_size >= bt_cols.  The last three count as
 *   errors in *err_count.  Results are exact 64-bit integers.
 *
 *   block_table  int32 [num_reqs, bt_stride], first bt_cols columns used.
 *   req_indices  int32 [num_tokens]; positions int64 [num_tokens].
 *   slot_mapping int64 [max_num_tokens], written in full.
 *   err_count    int32*, nullable.
 *   INVALID_ARG: block_size <= 0, num_tokens < 0, max_num_tokens <
 *   num_tokens, bt_stride < bt_cols, a needed pointer is null.
 */
int bkv_compute_slot_mapping(const int32_t *block_table, int32_t num_reqs, int64_t bt_stride,
                             int32_t bt_cols, const int32_t *req_indices, const int64_t *positions,
                             int64_t num_tokens, int64_t max_num_tokens, int32_t block_size,
                             int64_t *slot_mapping, int32_t *err_count, bkv_stream_t stream);

/*
 * bkv_map_to_kernel_blocks
 *   Defined by "ブロック表" 設計動機 (a manager block of block_size tokens is
 *   blocks_per_kv_block = block_size / kernel_block_size kernel blocks) and
 *   境界と失敗 (an indivisible pair is an error).
 *
 *   With bpk = block_size / kernel_block_size, for every row r and manager
 *   column j < mgr_cols, t < bpk:
 *     kernel_table[r * kernel_stride + j * bpk + t] = m > 0 ? m * bpk + t : -1,
 *     m = mgr_table[r * mgr_stride + j]
 *   so that the kernel view (total_blocks * bpk, kernel_block_size, H, D) of
 *   a cache is the same memory as the manager view.  Columns at or past
 *   mgr_cols * bpk are not written.  An id m * bpk + t above INT32_MAX
 *   cannot be held by the int32 table and is written as -1 (no block).
 *
 *   INVALID_ARG: kernel_block_size <= 0, block_size % kernel_block_size != 0,
 *   kernel_stride < mgr_cols * bpk, mgr_stride < mgr_cols, null pointers.
 */
int bkv_map_to_kernel_blocks(const int32_t *mgr_table, int32_t rows, int64_t mgr_stride,
                             int32_t mgr_cols, int32_t block_size, int32_t kernel_block_size,
                             int32_t *kernel_table, int64_t kernel_stride, bkv_stream_t stream);

/*
 * bkv_cache_write
 *   Defined by "Padding and Batching with Block KV", Block Structure (cache
 *   layout) and Slot ID -1: Padding Tokens (a -1 slot writes nothing).
 *
 *   For every i < num_tokens with s = slot_mapping[i] >= 0:
 *     k_cache[s / block_size][s % block_size][:][:] = k_new[i][:][:]  (and V)
 *   a bit-for-bit copy of num_kv_heads * head_dim elements.  s >=
 *   total_blocks * block_size is skipped and counted in *err_count.  Two
 *   tokens naming the same slot is invalid input: one of them lands.
 *
 *   k_new, v_new  [num_tokens, new_token_stride] elements of `dtype`; the
 *                 first num_kv_heads * head_dim of each row are copied
 *                 (new_token_stride lets them be slices of a fused buffer).
 *   k_cache, v_cache  [total_blocks, block_size, num_kv_heads, head_dim].
 *   INVALID_ARG: non-positive sizes, new_token_stride < num_kv_heads *
 *   head_dim, null pointers.  UNSUPPORTED: dtype not BKV_BF16 / BKV_F32.
 */
int bkv_cache_write(const void *k_new, const void *v_new, int64_t num_tokens,
                    int64_t new_token_stride, const int64_t *slot_mapping, void *k_cache,
                    void *v_cache, int64_t total_blocks, int32_t block_size, int32_t num_kv_heads,
                    int32_t head_dim, int dtype, int32_t *err_count, bkv_stream_t stream);

/*
 * bkv_slot_mapping_cache_write
 *   bkv_compute_slot_mapping followed by bkv_cache_write, as one kernel
 *   ("Padding and Batching with Block KV", The Core Formula; Slot ID -1:
 *   Padding Tokens; Block Structure): the step's slots are computed and its
 *   new K/V rows scattered to them in one pass.  The results are exactly
 *   those of the two calls in sequence with the same arguments: the same
 *   slot_mapping[0, max_num_tokens) (-1 past num_tokens), the same cache
 *   bytes, and the same *err_count increments (a bad request index,
 *   position or table width, and a slot past total_blocks * block_size,
 *   each counted once).  `block_size` is both the table's and the cache's
 *   block size (use the kernel table of bkv_map_to_kernel_blocks for
 *   hybrid block sizes).
 *
 *   Arguments as bkv_compute_slot_mapping (block_table .. slot_mapping) and
 *   bkv_cache_write (k_new .. dtype); the rows of tokens i < num_tokens are
 *   read.  INVALID_ARG / UNSUPPORTED: the union of the two calls' checks.
 */
int bkv_slot_mapping_cache_write(const int32_t *block_table, int32_t num_reqs, int64_t bt_stride,
                                 int32_t bt_cols, const int32_t *req_indices,
                                 const int64_t *positions, int64_t num_tokens,
                                 int64_t max_num_tokens, int64_t *slot_mapping, const void *k_new,
                                 const void *v_new, int64_t new_token_stride, void *k_cache,
                                 void *v_cache, int64_t total_blocks, int32_t block_size,
                                 int32_t num_kv_heads, int32_t head_dim, int dtype,
                                 int32_t *err_count, bkv_stream_t stream);

/*
 * bkv_paged_decode_workspace_size
 *   Bytes of device workspace bkv_paged_decode needs for these sizes on the
 *   CURRENT device (the split of long contexts into partitions depends on
 *   its SM count).  Returns 0 for invalid sizes.  Call it with the same
 *   arguments, on the same device, as the decode it is for.
 */
size_t bkv_paged_decode_workspace_size(int32_t num_reqs, int32_t q_len, int32_t num_q_heads,
                                       int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                       int32_t max_context_len);

/*
 * bkv_paged_decode
 *   Defined by "Padding and Batching with Block KV", Cache Masking
 *   (mask_cache: positions [0, cache_len) are valid; mask_active: the mask
 *   between this step's query tokens) and Special Block and Slot Values (a
 *   null / -1 block entry contributes nothing); "Decode Context-Length
 *   Bucketing", Problem (read only the blocks a request needs, not the full
 *   max_model_len row).
 *
 *   For request r with L = context_lens[r] (cache length INCLUDING this
 *   step's q_len tokens), query token t < q_len, query head h, G =
 *   num_q_heads / num_kv_heads:
 *     key j is visible iff j < L, j <= L - q_len + t (BKV_MASK_CAUSAL only)
 *     and b = block_table[r * bt_stride + j / block_size] > 0;
 *     out[r][t][h] = softmax_j(softmax_scale * q[r][t][h] . K[b][j % block_size][h / G])
 *                    . V[b][j % block_size][h / G]
 *   and 0 when no key is visible (e.g. L = 0 for a padded NULL row).  Only
 *   the ceil(L / block_size) table entries a request needs are read; cache
 *   memory at masked positions is never used (it may hold NaN).
 *
 *   q, out    [num_reqs, q_len, num_q_heads, head_dim] of `dtype`; out is
 *             rounded to nearest-even from fp32.
 *   k_cache, v_cache  [total_blocks, block_size, num_kv_heads, head_dim].
 *   block_table int32 [num_reqs, bt_stride], bt_cols columns valid.
 *   context_lens int32 [num_reqs].
 *   max_context_len  host-side upper bound on context_lens (sizes the grid);
 *             a larger context_lens[r] is clamped to it and counted once per
 *             such request in *err_count.
 *   softmax_scale    <= 0 selects 1 / sqrt(head_dim).
 *   workspace        device scratch of workspace_bytes >=
 *                    bkv_paged_decode_workspace_size(...); may be null when
 *                    that size is 0.  Used only while the call's kernels run;
 *                    its contents on entry do not matter.
 *   Bad table entries among those a request needs (an id >= total_blocks,
 *   or a block past bt_cols) are masked like null entries and each counts
 *   num_kv_heads times in *err_count (once per KV head that would read it).
 *   INVALID_ARG: num_q_heads % num_kv_heads != 0, non-positive sizes, bad
 *   mask_mode, workspace too small, null pointers.
 *   UNSUPPORTED: dtype not BKV_BF16 / BKV_F32, head_dim > 256 or odd.
 */
int bkv_paged_decode(const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_table, int64_t bt_stride, int32_t bt_cols,
                     const int32_t *context_lens, int32_t max_context_len, int32_t num_reqs,
                     int32_t q_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                     int32_t block_size, int64_t total_blocks, float softmax_scale, int mask_mode,
                     int dtype, void *out, void *workspace, size_t workspace_bytes,
                     int32_t *err_count, bkv_stream_t stream);

/*
 * bkv_paged_decode_swa
 *   bkv_paged_decode for a sliding-window attention layer ("KV Caching with
 *   vLLM", Layer-specific cache specification: an SWA layer keeps only the
 *   recent tokens within the window; "Decode Context-Length Bucketing",
 *   Block-table head-trim vs. SWA tail-trim).  The same arguments with
 *   `sliding_window` inserted after `mask_mode`:
 *     sliding_window W > 0: key j is visible to query t only if also
 *             j >= L - q_len + t - W + 1 (the last W positions up to its
 *             own), and only the blocks that overlap some query's window
 *             are read, so the entries of older blocks may already be null
 *             (-1) and their memory reused.  The table keeps logical block
 *             numbering (entry j covers positions [j * block_size, ...)), so
 *             no position offset is passed.  Bad entries are counted only
 *             among the blocks that are read.
 *     W = 0: exactly bkv_paged_decode.
 *   INVALID_ARG: as bkv_paged_decode, or sliding_window < 0.
 */
int bkv_paged_decode_swa(const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_table, int64_t bt_stride, int32_t bt_cols,
                         const int32_t *context_lens, int32_t max_context_len, int32_t num_reqs,
                         int32_t q_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int64_t total_blocks, float softmax_scale, int mask_mode,
                         int32_t sliding_window, int dtype, void *out, void *workspace,
                         size_t workspace_bytes, int32_t *err_count, bkv_stream_t stream);

/*
 * bkv_paged_decode_partition, bkv_paged_decode_merge
 *   The two phases of bkv_paged_decode_swa (sliding_window 0: of
 *   bkv_paged_decode), with exactly its arguments and checks: the partition
 *   phase reads the cache and writes every split-KV partial (o, max, sum of
 *   weights) into `workspace`; the merge phase, enqueued later with the same
 *   arguments and the same workspace contents, combines them into `out`.
 *   The operation is the one bkv_paged_decode defines ("Padding and Batching
 *   with Block KV", Cache Masking); the pages prescribe no split, so the
 *   split itself and its exact log-sum-exp merge of partial softmaxes belong
 *   to this library (no counterpart on the pages).  bkv_paged_decode_swa is
 *   exactly partition followed by merge, so the two-call form gives
 *   bit-identical results.  Between the calls the caller may run other work
 *   on the stream; the workspace layout is private to this library version,
 *   so it must reach the merge unchanged.
 *   Errors: as bkv_paged_decode_swa; each call validates its arguments again.
 */
int bkv_paged_decode_partition(const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *block_table, int64_t bt_stride, int32_t bt_cols,
                               const int32_t *context_lens, int32_t max_context_len,
                               int32_t num_reqs, int32_t q_len, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int64_t total_blocks, float softmax_scale, int mask_mode,
                               int32_t sliding_window, int dtype, void *out, void *workspace,
                               size_t workspace_bytes, int32_t *err_count, bkv_stream_t stream);
int bkv_paged_decode_merge(const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_table, int64_t bt_stride, int32_t bt_cols,
                           const int32_t *context_lens, int32_t max_context_len, int32_t num_reqs,
                           int32_t q_len, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t head_dim, int32_t block_size, int64_t total_blocks,
                           float softmax_scale, int mask_mode, int32_t sliding_window, int dtype,
                           void *out, void *workspace, size_t workspace_bytes, int32_t *err_count,
                           bkv_stream_t stream);

/*
 * bkv_cache_write_fp8
 *   bkv_cache_write into an FP8 cache.  The pages name a non-FP8 pathway
 *   ("Padding and Batching with Block KV", Block ID 0 vs. Sentinel -1) and
 *   print nothing about the format or its scaling; this library's reading:
 *   cache elements are OCP FP8 E4M3 codes (one byte: sign, 4 exponent bits
 *   of bias 7, 3 mantissa bits; no infinity; 0x7F / 0xFF are NaN; largest
 *   finite 448) with one scale per tensor.  Element x of k_new[i] is stored
 *   as the code nearest to x / k_scale, the quotient taken in IEEE binary32,
 *   ties to the even code, magnitudes above 448 (and infinities) saturated
 *   to +-448, NaN stored as NaN; V likewise with v_scale.  Rows, slots, -1
 *   padding and error counting are bkv_cache_write's.
 *
 *   k_new, v_new  [num_tokens, new_token_stride] of src_dtype (BKV_BF16 /
 *                 BKV_F32), the first num_kv_heads * head_dim of each row.
 *   k_cache, v_cache  uint8 [total_blocks, block_size, num_kv_heads, head_dim].
 *   INVALID_ARG: as bkv_cache_write, or k_scale / v_scale not a positive
 *   finite number.  UNSUPPORTED: src_dtype not BKV_BF16 / BKV_F32.
 */
int bkv_cache_write_fp8(const void *k_new, const void *v_new, int64_t num_tokens,
                        int64_t new_token_stride, const int64_t *slot_mapping, uint8_t *k_cache,
                        uint8_t *v_cache, int64_t total_blocks, int32_t block_size,
                        int32_t num_kv_heads, int32_t head_dim, int src_dtype, float k_scale,
                        float v_scale, int32_t *err_count, bkv_stream_t stream);

/*
 * bkv_slot_mapping_cache_write_fp8
 *   bkv_compute_slot_mapping followed by bkv_cache_write_fp8, as one kernel
 *   (the quantising write of bkv_cache_write_fp8, the slots of
 *   bkv_compute_slot_mapping): the same slot_mapping[0, max_num_tokens), the
 *   same cache bytes and the same *err_count increments as the two calls in
 *   sequence, as bkv_slot_mapping_cache_write is for bf16 / fp32 caches.
 *
 *   Arguments as bkv_slot_mapping_cache_write, with src_dtype the type of
 *   k_new / v_new (BKV_BF16 / BKV_F32), uint8 caches of E4M3 codes, and the
 *   per-tensor k_scale / v_scale of bkv_cache_write_fp8.
 *   INVALID_ARG / UNSUPPORTED: the union of the two calls' checks.
 */
int bkv_slot_mapping_cache_write_fp8(const int32_t *block_table, int32_t num_reqs, int64_t bt_stride,
                                     int32_t bt_cols, const int32_t *req_indices,
                                     const int64_t *positions, int64_t num_tokens,
                                     int64_t max_num_tokens, int64_t *slot_mapping,
                                     const void *k_new, const void *v_new,
                                     int64_t new_token_stride, uint8_t *k_cache, uint8_t *v_cache,
                                     int64_t total_blocks, int32_t block_size, int32_t num_kv_heads,
                                     int32_t head_dim, int src_dtype, float k_scale, float v_scale,
                                     int32_t *err_count, bkv_stream_t stream);

/*
 * bkv_paged_decode_fp8, bkv_paged_decode_fp8_partition, bkv_paged_decode_fp8_merge
 *   bkv_paged_decode_swa (and its two phases) over FP8 caches written by
 *   bkv_cache_write_fp8: a key element with code c stands for the value
 *   e4m3(c) * k_scale and a value element for e4m3(c) * v_scale; the
 *   operation, masks, sliding window, null entries, error counting and
 *   workspace are exactly bkv_paged_decode_swa's ("Padding and Batching with
 *   Block KV", Cache Masking; the FP8 format is the reading stated at
 *   bkv_cache_write_fp8).  `dtype` is the type of q and out (BKV_BF16 /
 *   BKV_F32); k_cache, v_cache are uint8 [total_blocks, block_size,
 *   num_kv_heads, head_dim].  A cache byte at a masked position is never
 *   used (NaN codes there change nothing).  bf16 q with head_dim 128 and at
 *   most 16 query rows per KV head runs the tensor-core kernel: q . k on
 *   E4M3 tensor cores with each query row split into two E4M3 parts (exact
 *   for elements down to 2^-10 of the row's largest, within 2^-17 of it
 *   below), P . v on E4M3 tensor cores with the value codes as stored and
 *   the weights as two E4M3 parts (within 2^-10 of p 2^8); anything else
 *   runs the CUDA-core kernel on the exact code values.  The workspace
 *   (bkv_paged_decode_workspace_size) includes the split queries.
 *   Errors: as bkv_paged_decode_swa, plus INVALID_ARG for a scale that is
 *   not a positive finite number.
 */
int bkv_paged_decode_fp8(const void *q, const uint8_t *k_cache, const uint8_t *v_cache,
                         const int32_t *block_table, int64_t bt_stride, int32_t bt_cols,
                         const int32_t *context_lens, int32_t max_context_len, int32_t num_reqs,
                         int32_t q_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int64_t total_blocks, float softmax_scale, float k_scale,
                         float v_scale, int mask_mode, int32_t sliding_window, int dtype, void *out,
                         void *workspace, size_t workspace_bytes, int32_t *err_count,
                         bkv_stream_t stream);
int bkv_paged_decode_fp8_partition(const void *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                   const int32_t *block_table, int64_t bt_stride, int32_t bt_cols,
                                   const int32_t *context_lens, int32_t max_context_len,
                                   int32_t num_reqs, int32_t q_len, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                   int64_t total_blocks, float softmax_scale, float k_scale,
                                   float v_scale, int mask_mode, int32_t sliding_window, int dtype,
                                   void *out, void *workspace, size_t workspace_bytes,
                                   int32_t *err_count, bkv_stream_t stream);
int bkv_paged_decode_fp8_merge(const void *q, const uint8_t *k_cache, const uint8_t *v_cache,
                               const int32_t *block_table, int64_t bt_stride, int32_t bt_cols,
                               const int32_t *context_lens, int32_t max_context_len, int32_t num_reqs,
                               int32_t q_len, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t head_dim, int32_t block_size, int64_t total_blocks,
                               float softmax_scale, float k_scale, float v_scale, int mask_mode,
                               int32_t sliding_window, int dtype, void *out, void *workspace,
                               size_t workspace_bytes, int32_t *err_count, bkv_stream_t stream);

/*
 * bkv_paged_attention_ragged
 *   Paged attention over a mixed (ragged) step: every request with its own
 *   number of query tokens -- decode tokens, speculative drafts, chunked
 *   prefill -- in one packed batch ("Padding and Batching with Block KV",
 *   Batching with Block KV: a request's new tokens are consecutive
 *   positions ending at its cache length; Cache Masking for mask_active).
 *   Request r's query tokens are rows [query_start_loc[r],
 *   query_start_loc[r+1]) of q and out; with q_len_r their count and L =
 *   context_lens[r] (INCLUDING those tokens), token i sits at position
 *   L - q_len_r + i and sees key j iff j < L, j <= its position
 *   (BKV_MASK_CAUSAL) and its block entry is a real block, exactly as
 *   bkv_paged_decode does for one q_len; out row = softmax-weighted V, 0 if
 *   it sees no key.
 *   q, out    [num_tokens, num_q_heads, head_dim] of `dtype` (token-major).
 *   query_start_loc int32 [num_reqs + 1], non-decreasing, last <= num_tokens.
 *   max_query_len / max_context_len  host bounds on q_len_r / context_lens
 *             (size the grid).  A request with more query tokens than
 *             max_query_len (or a malformed query_start_loc) is skipped, its
 *             rows left as they were, and counted; a longer context is
 *             clamped to max_context_len and counted.
 *   Other arguments as bkv_paged_decode.  No workspace: bf16 with head_dim
 *   128 and at most 128 query heads per KV head runs a tcgen05 kernel with
 *   128-row query tiles; anything else a CUDA-core kernel.
 *   INVALID_ARG: bad sizes or mask_mode, null pointers, grid too large.
 *   UNSUPPORTED: dtype not BKV_BF16 / BKV_F32, head_dim > 256 or odd.
 */
int bkv_paged_attention_ragged(const void *q, const int32_t *query_start_loc, const void *k_cache,
                               const void *v_cache, const int32_t *block_table, int64_t bt_stride,
                               int32_t bt_cols, const int32_t *context_lens, int32_t max_context_len,
                               int32_t max_query_len, int32_t num_reqs, int64_t num_tokens,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t block_size, int64_t total_blocks, float softmax_scale,
                               int mask_mode, int dtype, void *out, int32_t *err_count,
                               bkv_stream_t stream);

/*
 * bkv_compute_slot_mapping_cp
 *   bkv_compute_slot_mapping under decode context parallelism ("ブロック表"
 *   設計動機: with DCP the slot kernel writes the real slot only for the
 *   tokens its own rank holds and PAD for the others; the page names the
 *   world size, rank and interleave size but prints no formula).  Reading
 *   taken: global position p belongs to rank (p / cp_interleave) %
 *   cp_world (runs of cp_interleave consecutive positions dealt round
 *   robin) and is stored on that rank at the local position
 *   p_l = (p / (cp_interleave * cp_world)) * cp_interleave + p % cp_interleave;
 *   `block_table` is this rank's table over local positions, so the slot is
 *   block_table[r][p_l / block_size] * block_size + p_l % block_size.  A
 *   token another rank holds gets -1 and is not an error.  When
 *   cp_interleave divides block_size this is the same as one table shared
 *   by all ranks with blocks of block_size * cp_world global positions.
 *   cp_world = 1 is bkv_compute_slot_mapping exactly.
 *   INVALID_ARG: as bkv_compute_slot_mapping, or cp_world < 1, cp_rank
 *   outside [0, cp_world), cp_interleave < 1.
 */
int bkv_compute_slot_mapping_cp(const int32_t *block_table, int32_t num_reqs, int64_t bt_stride,
                                int32_t bt_cols, const int32_t *req_indices, const int64_t *positions,
                                int64_t num_tokens, int64_t max_num_tokens, int32_t block_size,
                                int32_t cp_world, int32_t cp_rank, int32_t cp_interleave,
                                int64_t *slot_mapping, int32_t *err_count, bkv_stream_t stream);

/*
 * bkv_paged_decode_cp
 *   One rank's part of a context-parallel paged decode: bkv_paged_decode
 *   over the keys this rank holds (the split of bkv_compute_slot_mapping_cp;
 *   k_cache, v_cache and block_table are this rank's, context_lens are the
 *   requests' GLOBAL cache lengths), with the causal mask applied in global
 *   positions.  `out` receives this rank's normalised result and, when `lse`
 *   is not NULL, lse[(r * q_len + t) * num_q_heads + h] receives the natural
 *   log of the sum of exp(softmax_scale * q . k) over this rank's visible
 *   keys (-inf, with out = 0, where it sees none).  Merging the ranks'
 *   (out, lse) with bkv_merge_attn_states gives the attention over all keys
 *   (the exchange between ranks, an all-gather, is the caller's).  The
 *   workspace is the one bkv_paged_decode_workspace_size gives for the
 *   global max_context_len.  cp_world = 1 is bkv_paged_decode plus lse.
 *   Errors: as bkv_paged_decode, plus INVALID_ARG for a bad cp_world /
 *   cp_rank / cp_interleave.
 */
int bkv_paged_decode_cp(const void *q, const void *k_cache, const void *v_cache,
                        const int32_t *block_table, int64_t bt_stride, int32_t bt_cols,
                        const int32_t *context_lens, int32_t max_context_len, int32_t num_reqs,
                        int32_t q_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                        int32_t block_size, int64_t total_blocks, float softmax_scale, int mask_mode,
                        int32_t cp_world, int32_t cp_rank, int32_t cp_interleave, int dtype, void *out,
                        float *lse, void *workspace, size_t workspace_bytes, int32_t *err_count,
                        bkv_stream_t stream);

/*
 * bkv_merge_attn_states
 *   Combines `parts` partial attention results of the same rows, each a
 *   normalised output and its log-sum-exp as bkv_paged_decode_cp writes
 *   them: out = sum_k e^(lse_k - M) outs_k / sum_k e^(lse_k - M) and
 *   lse_out = M + log sum_k e^(lse_k - M), M = max_k lse_k; a row whose parts
 *   are all -inf gives 0 and -inf.  This is the step after the ranks of a
 *   context-parallel decode exchange their results ("ブロック表" 設計動機,
 *   DCP); the pages print no formula for it, and it is the exact split of a
 *   softmax over disjoint key sets.
 *   outs   [parts][rows][head_dim] of `dtype`;  lses  fp32 [parts][rows];
 *   out    [rows][head_dim] of `dtype`;  lse_out fp32 [rows] or NULL.
 *   INVALID_ARG: parts < 1, rows < 0, head_dim < 1, null pointers.
 *   UNSUPPORTED: dtype not BKV_BF16 / BKV_F32.
 */
int bkv_merge_attn_states(const void *outs, const float *lses, int32_t parts, int64_t rows,
                          int32_t head_dim, int dtype, void *out, float *lse_out, bkv_stream_t stream);

/*
 * bkv_paged_decode_noalloc
 *   No counterpart on the pages: this is a convenience of this library.
 *
 *   Same operation, arguments and results as bkv_paged_decode, but with no
 *   workspace argument and no device allocation of any kind.  It is for
 *   callers that cannot call cudaMalloc: code running while a stream is
 *   being captured into a CUDA graph under a mode that forbids allocation,
 *   plugins whose host framework owns all device memory and refuses new
 *   allocations after start-up, or plain C callers that hold only raw
 *   pointers to their inputs and outputs and no allocator.
 *
 *   The split-KV scratch lives in one fixed device array of
 *   BKV_NOALLOC_SCRATCH_BYTES inside this library; every GPU on which the
 *   library is used holds that array until the process exits.  Shapes whose
 *   bkv_paged_decode_workspace_size(...) exceeds it are rejected with
 *   BKV_ERR_UNSUPPORTED before anything is enqueued (use bkv_paged_decode
 *   with your own workspace for those).
 *
 *   The array's device address is looked up (cudaGetSymbolAddress, with
 *   the call's device current) on every call made outside stream capture,
 *   so a device reset between calls does no harm.  A call made while its
 *   stream is being captured uses the address the last call outside
 *   capture found on that device: make one call on each device before
 *   capturing (a first call under capture returns BKV_ERR_CUDA), and do not
 *   reset the device between that call and the replays.  All calls share
 *   the one array and leave the last call's partial results in it (nothing
 *   in it has to start at zero): calls whose kernels overlap on the GPU (on
 *   different streams without ordering between them) race on it and give
 *   undefined results.
 */
#define BKV_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

int bkv_paged_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *block_table, int64_t bt_stride, int32_t bt_cols,
                             const int32_t *context_lens, int32_t max_context_len,
                             int32_t num_reqs, int32_t q_len, int32_t num_q_heads,
                             int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                             int64_t total_blocks, float softmax_scale, int mask_mode, int dtype,
                             void *out, int32_t *err_count, bkv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BKV_H_ */
