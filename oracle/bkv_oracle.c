/*
 * bkv_oracle.c -- plain, slow, obviously-correct CPU oracle for the paged
 * (block) KV cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * helper with the CUDA library; the two only see the same seeded inputs.
 *
 * Every routine is the plain definition written out, one scalar loop at a
 * time, in the order the pages state it.  Floating point is fp64 throughout;
 * bf16 and fp32 inputs are widened exactly (a bf16 value is the top 16 bits
 * of an IEEE binary32 value).
 *
 * Sources (web pages; section names as printed on them):
 *   [P1] "Padding and Batching with Block KV" (vllm-neuron design notes)
 *        - Block KV Cache Architecture / Block Structure, Block Table
 *        - Slot Mapping / The Core Formula, Slot Mapping Computation
 *        - Special Block and Slot Values / Block ID 0 vs. Sentinel -1,
 *          Slot ID -1: Padding Tokens
 *        - Padding with Block KV / Slot Mapping for Padded Tokens
 *        - Cache Masking / mask_cache, mask_active
 *   [P2] "ブロック表" (vLLM v1 BlockTable walkthrough)
 *        - 設計動機 (kernel block_size vs manager block_size; CUDA-graph
 *          padding of the slot-mapping tail)
 *        - 境界と失敗 (block_size % kernel_block_size != 0 is an error)
 *   [P3] "KV Caching with vLLM" (Neuron)
 *        - Layer-specific cache specification (sliding-window layers)
 *   [P4] "Decode Context-Length Bucketing"
 *        - Design / Per-step bucket selection (needed_seq), Block-table
 *          head-trim vs. SWA tail-trim
 *
 * Readings where the pages leave a step open (each is marked R<n> below):
 *   R2  any block-table entry <= 0 (upstream null block 0 or the -1
 *       sentinel) yields slot -1 / is never read.
 *   R3  a token is padding if its index is >= num_tokens or its request
 *       index is negative.
 *   R5  manager block m expands to kernel blocks m*bpk + t, t < bpk;
 *       m <= 0 expands to bpk entries of -1.
 *   R6  attention is scaled dot-product attention; GQA query head h reads
 *       KV head h / (num_q_heads / num_kv_heads).
 *   R7  mask_mode 0: query t of a request with cache length L sits at
 *       position L - q_len + t and sees keys j <= that position; mask_mode 1:
 *       every query sees every key j < L (an all-ones mask_active).
 *   R9  a row with no visible key (context length 0, e.g. a padded batch
 *       row) outputs 0.
 *   R10 a key whose block-table entry is <= 0 is masked out, not read.
 *   R12 a position past the table width gives slot -1 and counts an error.
 *   R15 a mixed (ragged) step: request r has q_len_r = query_start_loc[r+1]
 *       - query_start_loc[r] query tokens, packed token-major in q and out
 *       ([num_tokens][H_q][D]); token i of request r sits at position
 *       L_r - q_len_r + i ([P1 Batching with Block KV]: a request's tokens
 *       are consecutive positions ending at its cache length, as in the
 *       multi-token decode example) and sees keys as R7 with that position;
 *       the decode is the case of one q_len for every request.
 *   R13 sliding window W > 0 ([P4 Block-table head-trim vs. SWA tail-trim;
 *       [P3] Layer-specific cache specification: an SWA layer keeps only
 *       the recent tokens within the window): query t at position p_t =
 *       L - q_len + t sees only keys j >= p_t - W + 1, in both mask modes
 *       (the upper bound is R7's); blocks wholly before every query's window
 *       are never read, so they may be null or hold anything.  W <= 0: no
 *       window.
 *   R14 decode context parallelism ([P2 設計動機]: under DCP the slot
 *       kernel writes real slots only for the tokens its rank owns and
 *       PAD_ID for the rest; the ownership formula is not printed): with
 *       world size Wc, rank k and interleave size I, position p belongs to
 *       rank (p / I) mod Wc (runs of I consecutive positions dealt round
 *       robin); its owner stores it at local position
 *       p_l = (p / (I Wc)) I + p mod I, and the owner's block table indexes
 *       local positions, so slot = table[r][p_l / bs] * bs + p_l mod bs.  A
 *       rank's decode attends over its own keys with the masks in global
 *       positions (local key j stands for (j / I) I Wc + k I + j mod I) and
 *       reports its normalised output and lse = log sum_j exp(s_j) over its
 *       visible keys (-inf if none); merging the ranks' (out, lse) by
 *       out = sum_k exp(lse_k - LSE) out_k, LSE = log sum_k exp(lse_k), is
 *       the attention over all keys.
 *   R16 FP8 KV cache ([P1 Block ID 0 vs. Sentinel -1] names a non-FP8
 *       pathway, so FP8 caches exist; nothing else about them is printed):
 *       cache elements are OCP FP8 E4M3 ("fn": bias 7, no infinities, codes
 *       0x7F / 0xFF are NaN, largest finite 448).  One scale per tensor,
 *       k_scale for K and v_scale for V: a new element x is stored as the
 *       code nearest to the fp32 quotient x / scale (IEEE division in
 *       binary32), ties to the even code, magnitudes above 448 (and
 *       infinities) saturated to 448, NaN to NaN; a stored code c stands for
 *       the value e4m3(c) * scale.  Attention over an FP8 cache is O4 on
 *       those values.
 *   R17 an expanded kernel block id m*bpk + t above INT32_MAX cannot be
 *       held by the int32 kernel table: it is written as -1 (no block),
 *       the same outcome as an entry <= 0 under R2.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_DT_BF16 0
#define ORC_DT_F32 1
#define ORC_DT_E4M3 2   /* cache elements only (R16) */

/* ------------------------------------------------------------------ */
/* element access                                                      */
/* ------------------------------------------------------------------ */

/* Widen one element of a bf16 or fp32 array to double, exactly. */
static double orc_load(const void *base, int64_t idx, int dtype)
{
    if (dtype == ORC_DT_BF16) {
        uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float *)base)[idx];
}

static int orc_elem_bytes(int dtype)
{
    return dtype == ORC_DT_BF16 ? 2 : (dtype == ORC_DT_F32 ? 4 : 0);
}

/* ------------------------------------------------------------------ */
/* FP8 E4M3 (R16)                                                      */
/* ------------------------------------------------------------------ */

/*
 * The value of code c: sign bit 7, exponent field e = bits 6..3 (bias 7),
 * mantissa m = bits 2..0.  e = 0 is subnormal, m/8 * 2^-6; otherwise
 * (1 + m/8) * 2^(e-7).  e = 15 with m = 7 is NaN (there is no infinity).
 */
double orc_e4m3_decode(uint8_t c)
{
    const int sign = c >> 7;
    const int e = (c >> 3) & 15;
    const int m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/*
 * The code of the binary32 value x: NaN -> 0x7F; |x| >= 448 (infinities
 * included) -> the largest finite magnitude, 0x7E, with x's sign;
 * otherwise the finite code whose value is nearest to |x|, the even code on
 * a tie (codes 0x00..0x7E increase with their value, so a binary search
 * finds the two neighbours), with x's sign (so -0 and negative values that
 * round to 0 give 0x80).
 */
uint8_t orc_e4m3_encode(float x)
{
    if (isnan(x))
        return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    /* largest code lo with value(lo) <= a (value(0) = 0 <= a) */
    int lo = 0, hi = 0x7E;
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (orc_e4m3_decode((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid - 1;
    }
    int c = lo;
    if (lo < 0x7E) {
        const double below = a - orc_e4m3_decode((uint8_t)lo);
        const double above = orc_e4m3_decode((uint8_t)(lo + 1)) - a;
        if (above < below || (above == below && ((lo + 1) % 2 == 0)))
            c = lo + 1;
    }
    return (uint8_t)(sign | c);
}

/* Encode n binary32 values (a helper for the tests). */
void orc_e4m3_encode_array(const float *x, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_encode(x[i]);
}

/* One cache element as a double: bf16 / fp32 exactly, an E4M3 code as its
 * value times the tensor's scale (R16; the product is exact in binary64). */
static double orc_load_kv(const void *base, int64_t idx, int dtype, double scale)
{
    if (dtype == ORC_DT_E4M3)
        return orc_e4m3_decode(((const uint8_t *)base)[idx]) * scale;
    return orc_load(base, idx, dtype);
}

/* ------------------------------------------------------------------ */
/* O1: slot mapping                                                    */
/* ------------------------------------------------------------------ */

/*
 * slot = block_table[r][p / bs] * bs + p % bs             [P1 The Core Formula]
 * The table row of request r is looked up at logical block p / bs
 * ([P1 Slot Mapping Computation]); the slot buffer is max_num_tokens long
 * and every entry past num_tokens is the padding id -1 ([P2 設計動機],
 * CUDA-graph tail; [P1 Slot Mapping for Padded Tokens]).
 *
 * Returns the number of tokens flagged as bad input (request index past the
 * batch, negative position, position past the table width), or -1 when the
 * arguments themselves are invalid.
 */
int64_t orc_compute_slot_mapping(const int32_t *block_table, int32_t num_reqs,
                                 int64_t bt_stride, int32_t bt_cols,
                                 const int32_t *req_indices,
                                 const int64_t *positions, int64_t num_tokens,
                                 int64_t max_num_tokens, int32_t block_size,
                                 int64_t *slot_mapping)
{
    if (block_size <= 0 || num_tokens < 0 || max_num_tokens < num_tokens ||
        num_reqs < 0 || bt_cols < 0 || bt_stride < bt_cols)
        return -1;
    int64_t errors = 0;
    for (int64_t i = 0; i < max_num_tokens; ++i) {
        slot_mapping[i] = -1; /* PAD_SLOT_ID */
        if (i >= num_tokens)
            continue; /* tail padding (R3) */
        int32_t r = req_indices[i];
        int64_t p = positions[i];
        if (r < 0)
            continue; /* padded request (R3) */
        if (r >= num_reqs || p < 0) {
            errors += 1;
            continue;
        }
        int64_t logical_block = p / block_size;
        int64_t offset = p % block_size;
        if (logical_block >= bt_cols) { /* R12 */
            errors += 1;
            continue;
        }
        int64_t block_number = block_table[(int64_t)r * bt_stride + logical_block];
        if (block_number <= 0)
            continue; /* null block 0 or sentinel -1 (R2) */
        slot_mapping[i] = block_number * block_size + offset;
    }
    return errors;
}

/*
 * O1 under decode context parallelism (R14): the token's position p is
 * real on rank cp_rank only if (p / cp_interleave) mod cp_world == cp_rank;
 * there the slot follows the core formula at the local position
 * p_l = (p / (cp_interleave * cp_world)) * cp_interleave + p mod cp_interleave.
 * A token another rank owns gets -1 without counting an error.
 * Returns the number of bad indices (as O1), or -1 for invalid arguments.
 */
int64_t orc_compute_slot_mapping_cp(const int32_t *block_table, int32_t num_reqs,
                                    int64_t bt_stride, int32_t bt_cols,
                                    const int32_t *req_indices,
                                    const int64_t *positions, int64_t num_tokens,
                                    int64_t max_num_tokens, int32_t block_size,
                                    int32_t cp_world, int32_t cp_rank,
                                    int32_t cp_interleave, int64_t *slot_mapping)
{
    if (block_size <= 0 || num_tokens < 0 || max_num_tokens < num_tokens ||
        num_reqs < 0 || bt_cols < 0 || bt_stride < bt_cols || cp_world <= 0 ||
        cp_rank < 0 || cp_rank >= cp_world || cp_interleave <= 0)
        return -1;
    int64_t errors = 0;
    for (int64_t i = 0; i < max_num_tokens; ++i) {
        slot_mapping[i] = -1;
        if (i >= num_tokens)
            continue;
        int32_t r = req_indices[i];
        int64_t p = positions[i];
        if (r < 0)
            continue;
        if (r >= num_reqs || p < 0) {
            errors += 1;
            continue;
        }
        int64_t owner = (p / cp_interleave) % cp_world;
        if (owner != cp_rank)
            continue; /* another rank's token: PAD */
        int64_t local = (p / ((int64_t)cp_interleave * cp_world)) * cp_interleave +
                        p % cp_interleave;
        int64_t logical_block = local / block_size;
        if (logical_block >= bt_cols) {
            errors += 1;
            continue;
        }
        int64_t block_number = block_table[(int64_t)r * bt_stride + logical_block];
        if (block_number <= 0)
            continue;
        slot_mapping[i] = block_number * block_size + local % block_size;
    }
    return errors;
}

/* ------------------------------------------------------------------ */
/* O2: manager -> kernel block expansion                               */
/* ------------------------------------------------------------------ */

/*
 * One manager block of block_size tokens is blocks_per_kv_block =
 * block_size / kernel_block_size kernel blocks ([P2 設計動機], e.g. 32 -> 16,
 * two kernel blocks each); an indivisible pair is an error ([P2 境界と失敗]).
 * The layout (R5) is the one under which a kernel block id addresses the
 * same bytes as the manager view: kernel block m*bpk + t holds tokens
 * [t*kbs, (t+1)*kbs) of manager block m.
 *
 * R17: a kernel id m*bpk + t that does not fit in the int32 table names
 * no block; it is written as -1, like an id <= 0 (R2).
 *
 * Returns 0, or 1 for invalid arguments.  Columns of the output past
 * mgr_cols * bpk are left as they were.
 */
int orc_map_to_kernel_blocks(const int32_t *mgr_table, int32_t rows,
                             int64_t mgr_stride, int32_t mgr_cols,
                             int32_t block_size, int32_t kernel_block_size,
                             int32_t *kernel_table, int64_t kernel_stride)
{
    if (block_size <= 0 || kernel_block_size <= 0 ||
        block_size % kernel_block_size != 0 || rows < 0 || mgr_cols < 0 ||
        mgr_stride < mgr_cols)
        return 1;
    int64_t bpk = block_size / kernel_block_size;
    if (kernel_stride < (int64_t)mgr_cols * bpk)
        return 1;
    for (int32_t r = 0; r < rows; ++r) {
        for (int32_t j = 0; j < mgr_cols; ++j) {
            int64_t m = mgr_table[(int64_t)r * mgr_stride + j];
            for (int64_t t = 0; t < bpk; ++t) {
                int64_t out = (m > 0) ? m * bpk + t : -1;
                if (out > INT32_MAX)
                    out = -1;
                kernel_table[(int64_t)r * kernel_stride + j * bpk + t] = (int32_t)out;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* O3: KV cache write (scatter)                                        */
/* ------------------------------------------------------------------ */

/*
 * k_cache[s / bs][s % bs][:][:] = k_new[i], and the same for V, for every
 * token i whose slot s is non-negative ([P1 Block Structure] gives the
 * (total_blocks, block_size, num_kv_heads, head_dim) layout; [P1 Slot ID -1:
 * Padding Tokens] says a -1 slot writes nothing).  A slot past the cache is
 * skipped and counted.  The copy is bit-for-bit.
 *
 * Token i's row starts new_token_stride elements after token i-1's, and
 * holds num_kv_heads * head_dim contiguous elements.
 *
 * Returns the number of out-of-range slots, -1 for invalid arguments, or -2
 * when two tokens name the same slot (such input has no single correct
 * result and is rejected).
 */
int64_t orc_cache_write(const void *k_new, const void *v_new,
                        int64_t num_tokens, int64_t new_token_stride,
                        const int64_t *slot_mapping, void *k_cache,
                        void *v_cache, int64_t total_blocks, int32_t block_size,
                        int32_t num_kv_heads, int32_t head_dim, int dtype)
{
    int eb = orc_elem_bytes(dtype);
    int64_t row = (int64_t)num_kv_heads * head_dim;
    if (eb == 0 || num_tokens < 0 || total_blocks < 0 || block_size <= 0 ||
        num_kv_heads <= 0 || head_dim <= 0 || new_token_stride < row)
        return -1;
    int64_t capacity = total_blocks * block_size;
    unsigned char *seen = (unsigned char *)calloc((size_t)(capacity > 0 ? capacity : 1), 1);
    if (!seen)
        return -1;
    int64_t errors = 0;
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t s = slot_mapping[i];
        if (s < 0)
            continue;
        if (s >= capacity) {
            errors += 1;
            continue;
        }
        if (seen[s]) {
            free(seen);
            return -2;
        }
        seen[s] = 1;
    }
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t s = slot_mapping[i];
        if (s < 0 || s >= capacity)
            continue;
        int64_t block = s / block_size;
        int64_t offset = s % block_size;
        int64_t dst = (block * block_size + offset) * row; /* element index */
        int64_t src = i * new_token_stride;
        memcpy((char *)k_cache + dst * eb, (const char *)k_new + src * eb, (size_t)(row * eb));
        memcpy((char *)v_cache + dst * eb, (const char *)v_new + src * eb, (size_t)(row * eb));
    }
    free(seen);
    return errors;
}

/*
 * O3 for an FP8 cache (R16): the same rows are written, each element of a
 * new K row as orc_e4m3_encode((float)x / k_scale) and of a V row with
 * v_scale, the quotient taken in binary32 (x is bf16 or fp32, widened
 * exactly).  Same return values as orc_cache_write.
 */
int64_t orc_cache_write_fp8(const void *k_new, const void *v_new,
                            int64_t num_tokens, int64_t new_token_stride,
                            const int64_t *slot_mapping, uint8_t *k_cache,
                            uint8_t *v_cache, int64_t total_blocks, int32_t block_size,
                            int32_t num_kv_heads, int32_t head_dim, int src_dtype,
                            float k_scale, float v_scale)
{
    int64_t row = (int64_t)num_kv_heads * head_dim;
    if (orc_elem_bytes(src_dtype) == 0 || num_tokens < 0 || total_blocks < 0 ||
        block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        new_token_stride < row || !(k_scale > 0.0f) || !(v_scale > 0.0f))
        return -1;
    int64_t capacity = total_blocks * block_size;
    unsigned char *seen = (unsigned char *)calloc((size_t)(capacity > 0 ? capacity : 1), 1);
    if (!seen)
        return -1;
    int64_t errors = 0;
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t s = slot_mapping[i];
        if (s < 0)
            continue;
        if (s >= capacity) {
            errors += 1;
            continue;
        }
        if (seen[s]) {
            free(seen);
            return -2;
        }
        seen[s] = 1;
    }
    for (int64_t i = 0; i < num_tokens; ++i) {
        int64_t s = slot_mapping[i];
        if (s < 0 || s >= capacity)
            continue;
        int64_t dst = s * row;   /* block s / bs, offset s % bs */
        int64_t src = i * new_token_stride;
        for (int64_t e = 0; e < row; ++e) {
            float k = (float)orc_load(k_new, src + e, src_dtype);
            float v = (float)orc_load(v_new, src + e, src_dtype);
            float kq = k / k_scale;
            float vq = v / v_scale;
            k_cache[dst + e] = orc_e4m3_encode(kq);
            v_cache[dst + e] = orc_e4m3_encode(vq);
        }
    }
    free(seen);
    return errors;
}

/* ------------------------------------------------------------------ */
/* O4: GQA paged decode attention (one request)                        */
/* ------------------------------------------------------------------ */

/*
 * For request r with cache length L = context_lens[r] ([P1 mask_cache]: the
 * valid positions are [0, L), and L counts this step's tokens) and each of
 * its q_len query tokens t, each query head h:
 *
 *   key position j is visible iff  j < L,  j <= L - q_len + t (mask_mode 0,
 *   R7),  j >= L - q_len + t - W + 1 (sliding window W > 0, R13), and its
 *   table entry b = block_table[r][j / bs] is a real block (b > 0, R10;
 *   b < total_blocks, otherwise counted as an error);
 *   s_j = scale * sum_d q[r,t,h,d] * K[b, j % bs, h / G, d]        (R6)
 *   out[r,t,h,:] = sum_j softmax(s)_j * V[b, j % bs, h / G, :]
 *
 * and 0 when no key is visible (R9).  The softmax subtracts the maximum
 * before exponentiating; that changes no value, only avoids overflow.
 *
 * q and out are (num_reqs, q_len, num_q_heads, head_dim); out is fp64.
 * Returns the number of bad table entries met among the blocks some query
 * may see (positions past the table width or ids past the cache), or -1 for
 * invalid arguments.
 */
/*
 * The general form: the keys are this rank's (R14; cp_world 1 is the plain
 * cache) and, when lse is not NULL, lse[(r * q_len + t) * num_q_heads + h]
 * receives log sum_j exp(s_j) over the visible keys (-inf if none).  Key
 * positions, masks and windows are global; j below is a local key index and
 * g its global position.
 */
/* The decode of one request with the query type dtype and the cache
 * element type kv_dtype (dtype itself, or ORC_DT_E4M3 with the tensors'
 * scales, R16). */
static int64_t orc_decode_core(int32_t r, const void *q, const void *k_cache,
                               const void *v_cache, const int32_t *block_table,
                               int64_t bt_stride, int32_t bt_cols,
                               const int32_t *context_lens, int32_t num_reqs,
                               int32_t q_len, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim,
                               int32_t block_size, int64_t total_blocks,
                               double scale, int mask_mode, int32_t sliding_window,
                               int32_t cp_world, int32_t cp_rank, int32_t cp_interleave,
                               int dtype, int kv_dtype, double k_scale, double v_scale,
                               double *out, double *lse)
{
    if (kv_dtype != dtype && kv_dtype != ORC_DT_E4M3)
        return -1;
    if (orc_elem_bytes(dtype) == 0 || r < 0 || r >= num_reqs || q_len <= 0 ||
        num_q_heads <= 0 || num_kv_heads <= 0 ||
        num_q_heads % num_kv_heads != 0 || head_dim <= 0 || block_size <= 0 ||
        bt_cols < 0 || bt_stride < bt_cols || (mask_mode != 0 && mask_mode != 1) ||
        cp_world <= 0 || cp_rank < 0 || cp_rank >= cp_world || cp_interleave <= 0)
        return -1;
    const int64_t D = head_dim;
    const int64_t G = num_q_heads / num_kv_heads;
    const int64_t L = context_lens[r] > 0 ? context_lens[r] : 0;   /* global cache length */
    const int64_t W = sliding_window > 0 ? sliding_window : 0;
    const int64_t I = cp_interleave, Wc = cp_world;
    /* R14: this rank's keys are the global positions g < L it owns */
    int64_t Lk = 0;
    for (int64_t g = 0; g < L; ++g)
        if ((g / I) % Wc == cp_rank)
            Lk += 1;
    /* R13: no query sees a key before lo (the window of query 0) */
    int64_t lo = 0;
    if (W > 0 && L - q_len - W + 1 > 0)
        lo = L - q_len - W + 1;
    int64_t errors = 0;

    /* Which local keys may be read at all: global position >= lo, a real
     * block (a bad entry counts once per block, at its first key read). */
    unsigned char *readable = (unsigned char *)malloc((size_t)(Lk > 0 ? Lk : 1));
    int64_t *gpos = (int64_t *)malloc(sizeof(int64_t) * (size_t)(Lk > 0 ? Lk : 1));
    double *s = (double *)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
    if (!readable || !gpos || !s) {
        free(readable);
        free(gpos);
        free(s);
        return -1;
    }
    int64_t first_read = -1;
    for (int64_t j = 0; j < Lk; ++j) {
        gpos[j] = (j / I) * I * Wc + cp_rank * I + j % I;
        readable[j] = 0;
        if (gpos[j] < lo)
            continue;
        if (first_read < 0)
            first_read = j;
        const int first = (j == first_read) || (j % block_size == 0);
        int64_t lb = j / block_size;
        if (lb >= bt_cols) {
            if (first)
                errors += 1;
            continue;
        }
        int64_t b = block_table[(int64_t)r * bt_stride + lb];
        if (b <= 0)
            continue;
        if (b >= total_blocks) {
            if (first)
                errors += 1;
            continue;
        }
        readable[j] = 1;
    }

    for (int64_t t = 0; t < q_len; ++t) {
        int64_t last_visible = (mask_mode == 0) ? (L - q_len + t) : (L - 1);
        int64_t first_visible = (W > 0) ? (L - q_len + t - W + 1) : 0;
        for (int64_t h = 0; h < num_q_heads; ++h) {
            int64_t g = h / G;
            const int64_t qoff = (((int64_t)r * q_len + t) * num_q_heads + h) * D;
            double *o = out + qoff;
            for (int64_t d = 0; d < D; ++d)
                o[d] = 0.0;
            if (lse)
                lse[((int64_t)r * q_len + t) * num_q_heads + h] = -INFINITY;

            double m = -INFINITY;
            int any = 0;
            for (int64_t j = 0; j < Lk; ++j) {
                if (!readable[j] || gpos[j] > last_visible || gpos[j] < first_visible)
                    continue;
                int64_t b = block_table[(int64_t)r * bt_stride + j / block_size];
                int64_t krow = ((b * block_size + j % block_size) * num_kv_heads + g) * D;
                double dot = 0.0;
                for (int64_t d = 0; d < D; ++d)
                    dot += orc_load(q, qoff + d, dtype) * orc_load_kv(k_cache, krow + d, kv_dtype, k_scale);
                s[j] = scale * dot;
                if (!any || s[j] > m)
                    m = s[j];
                any = 1;
            }
            if (!any)
                continue; /* R9: nothing visible -> 0 */

            double denom = 0.0;
            for (int64_t j = 0; j < Lk; ++j) {
                if (!readable[j] || gpos[j] > last_visible || gpos[j] < first_visible)
                    continue;
                int64_t b = block_table[(int64_t)r * bt_stride + j / block_size];
                int64_t vrow = ((b * block_size + j % block_size) * num_kv_heads + g) * D;
                double w = exp(s[j] - m);
                denom += w;
                for (int64_t d = 0; d < D; ++d)
                    o[d] += w * orc_load_kv(v_cache, vrow + d, kv_dtype, v_scale);
            }
            for (int64_t d = 0; d < D; ++d)
                o[d] /= denom;
            if (lse)
                lse[((int64_t)r * q_len + t) * num_q_heads + h] = m + log(denom);
        }
    }
    free(readable);
    free(gpos);
    free(s);
    return errors;
}

int64_t orc_paged_decode_cp_request(int32_t r, const void *q, const void *k_cache,
                                    const void *v_cache, const int32_t *block_table,
                                    int64_t bt_stride, int32_t bt_cols,
                                    const int32_t *context_lens, int32_t num_reqs,
                                    int32_t q_len, int32_t num_q_heads,
                                    int32_t num_kv_heads, int32_t head_dim,
                                    int32_t block_size, int64_t total_blocks,
                                    double scale, int mask_mode, int32_t sliding_window,
                                    int32_t cp_world, int32_t cp_rank, int32_t cp_interleave,
                                    int dtype, double *out, double *lse)
{
    return orc_decode_core(r, q, k_cache, v_cache, block_table, bt_stride, bt_cols,
                           context_lens, num_reqs, q_len, num_q_heads, num_kv_heads,
                           head_dim, block_size, total_blocks, scale, mask_mode,
                           sliding_window, cp_world, cp_rank, cp_interleave, dtype,
                           dtype, 1.0, 1.0, out, lse);
}

/*
 * O4 over an FP8 cache (R16), one request: the keys and values are the
 * codes' values times k_scale / v_scale; q and out as orc_paged_decode_request.
 */
int64_t orc_paged_decode_fp8_request(int32_t r, const void *q, const uint8_t *k_cache,
                                     const uint8_t *v_cache, const int32_t *block_table,
                                     int64_t bt_stride, int32_t bt_cols,
                                     const int32_t *context_lens, int32_t num_reqs,
                                     int32_t q_len, int32_t num_q_heads,
                                     int32_t num_kv_heads, int32_t head_dim,
                                     int32_t block_size, int64_t total_blocks,
                                     double scale, double k_scale, double v_scale,
                                     int mask_mode, int32_t sliding_window,
                                     int dtype, double *out)
{
    if (!(k_scale > 0.0) || !(v_scale > 0.0))
        return -1;
    return orc_decode_core(r, q, k_cache, v_cache, block_table, bt_stride, bt_cols,
                           context_lens, num_reqs, q_len, num_q_heads, num_kv_heads,
                           head_dim, block_size, total_blocks, scale, mask_mode,
                           sliding_window, 1, 0, 1, dtype, ORC_DT_E4M3, k_scale,
                           v_scale, out, NULL);
}

/*
 * O4 over a mixed step (R15): every request with its own number of query
 * tokens, packed token-major.  The visible keys, the scores and the softmax
 * are those of O4 for each token at its own position.  Returns the number of
 * bad table entries met (once per request and block), or -1.
 */
int64_t orc_paged_attention_ragged(const void *q, const int32_t *query_start_loc,
                                   const void *k_cache, const void *v_cache,
                                   const int32_t *block_table, int64_t bt_stride,
                                   int32_t bt_cols, const int32_t *context_lens,
                                   int32_t num_reqs, int64_t num_tokens, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                   int64_t total_blocks, double scale, int mask_mode,
                                   int dtype, double *out)
{
    if (orc_elem_bytes(dtype) == 0 || num_reqs < 0 || num_tokens < 0 || num_q_heads <= 0 ||
        num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0 ||
        block_size <= 0 || bt_cols < 0 || bt_stride < bt_cols ||
        (mask_mode != 0 && mask_mode != 1))
        return -1;
    const int64_t D = head_dim;
    const int64_t G = num_q_heads / num_kv_heads;
    for (int64_t i = 0; i < num_tokens * num_q_heads * D; ++i)
        out[i] = 0.0;
    int64_t errors = 0;
    for (int32_t r = 0; r < num_reqs; ++r) {
        const int64_t t0 = query_start_loc[r], t1 = query_start_loc[r + 1];
        if (t0 < 0 || t1 < t0 || t1 > num_tokens)
            return -1;
        const int64_t ql = t1 - t0;
        const int64_t L = context_lens[r] > 0 ? context_lens[r] : 0;
        if (ql == 0 || L == 0)
            continue;
        /* which keys may be read: j < L with a real block */
        unsigned char *readable = (unsigned char *)malloc((size_t)L);
        double *s = (double *)malloc(sizeof(double) * (size_t)L);
        if (!readable || !s) {
            free(readable);
            free(s);
            return -1;
        }
        for (int64_t j = 0; j < L; ++j) {
            readable[j] = 0;
            int64_t lb = j / block_size;
            if (lb >= bt_cols) {
                if (j % block_size == 0)
                    errors += 1;
                continue;
            }
            int64_t b = block_table[(int64_t)r * bt_stride + lb];
            if (b <= 0)
                continue;
            if (b >= total_blocks) {
                if (j % block_size == 0)
                    errors += 1;
                continue;
            }
            readable[j] = 1;
        }
        for (int64_t i = 0; i < ql; ++i) {
            const int64_t p = L - ql + i; /* this token's position */
            const int64_t last_visible = (mask_mode == 0) ? p : L - 1;
            for (int64_t h = 0; h < num_q_heads; ++h) {
                const int64_t g = h / G;
                const int64_t qoff = ((t0 + i) * num_q_heads + h) * D;
                double *o = out + qoff;
                double m = -INFINITY;
                int any = 0;
                for (int64_t j = 0; j < L && j <= last_visible; ++j) {
                    if (!readable[j])
                        continue;
                    int64_t b = block_table[(int64_t)r * bt_stride + j / block_size];
                    int64_t krow = ((b * block_size + j % block_size) * num_kv_heads + g) * D;
                    double dot = 0.0;
                    for (int64_t d = 0; d < D; ++d)
                        dot += orc_load(q, qoff + d, dtype) * orc_load(k_cache, krow + d, dtype);
                    s[j] = scale * dot;
                    if (!any || s[j] > m)
                        m = s[j];
                    any = 1;
                }
                if (!any)
                    continue;
                double denom = 0.0;
                for (int64_t j = 0; j < L && j <= last_visible; ++j) {
                    if (!readable[j])
                        continue;
                    int64_t b = block_table[(int64_t)r * bt_stride + j / block_size];
                    int64_t vrow = ((b * block_size + j % block_size) * num_kv_heads + g) * D;
                    double w = exp(s[j] - m);
                    denom += w;
                    for (int64_t d = 0; d < D; ++d)
                        o[d] += w * orc_load(v_cache, vrow + d, dtype);
                }
                for (int64_t d = 0; d < D; ++d)
                    o[d] /= denom;
            }
        }
        free(readable);
        free(s);
    }
    return errors;
}

/* One request of the plain (single-rank) decode. */
int64_t orc_paged_decode_request(int32_t r, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *block_table,
                                 int64_t bt_stride, int32_t bt_cols,
                                 const int32_t *context_lens, int32_t num_reqs,
                                 int32_t q_len, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim,
                                 int32_t block_size, int64_t total_blocks,
                                 double scale, int mask_mode, int32_t sliding_window,
                                 int dtype, double *out)
{
    return orc_paged_decode_cp_request(r, q, k_cache, v_cache, block_table, bt_stride,
                                       bt_cols, context_lens, num_reqs, q_len,
                                       num_q_heads, num_kv_heads, head_dim, block_size,
                                       total_blocks, scale, mask_mode, sliding_window,
                                       1, 0, 1, dtype, out, NULL);
}

/*
 * Merge of attention states (R14): rows of `parts` partial results, each a
 * normalised output (fp64 [parts][rows][head_dim]) and its lse
 * ([parts][rows]); out = sum_k exp(lse_k - M) out_k / sum_k exp(lse_k - M),
 * lse_out = M + log sum_k exp(lse_k - M), M = max_k lse_k; a row whose parts
 * are all -inf gives 0 and -inf.
 */
int orc_merge_attn_states(const double *outs, const double *lses, int32_t parts,
                          int64_t rows, int32_t head_dim, double *out, double *lse_out)
{
    if (parts <= 0 || rows < 0 || head_dim <= 0)
        return 1;
    for (int64_t i = 0; i < rows; ++i) {
        double M = -INFINITY;
        for (int32_t k = 0; k < parts; ++k)
            if (lses[(int64_t)k * rows + i] > M)
                M = lses[(int64_t)k * rows + i];
        double *o = out + i * head_dim;
        for (int32_t d = 0; d < head_dim; ++d)
            o[d] = 0.0;
        if (M == -INFINITY) {
            lse_out[i] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int32_t k = 0; k < parts; ++k) {
            double w = exp(lses[(int64_t)k * rows + i] - M);
            sum += w;
            const double *ok = outs + ((int64_t)k * rows + i) * head_dim;
            for (int32_t d = 0; d < head_dim; ++d)
                o[d] += w * ok[d];
        }
        for (int32_t d = 0; d < head_dim; ++d)
            o[d] /= sum;
        lse_out[i] = M + log(sum);
    }
    return 0;
}

/* The whole batch: every request in turn. */
int64_t orc_paged_decode(const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_table, int64_t bt_stride,
                         int32_t bt_cols, const int32_t *context_lens,
                         int32_t num_reqs, int32_t q_len, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int64_t total_blocks, double scale,
                         int mask_mode, int32_t sliding_window, int dtype, double *out)
{
    int64_t errors = 0;
    for (int32_t r = 0; r < num_reqs; ++r) {
        int64_t e = orc_paged_decode_request(r, q, k_cache, v_cache, block_table,
                                             bt_stride, bt_cols, context_lens,
                                             num_reqs, q_len, num_q_heads,
                                             num_kv_heads, head_dim, block_size,
                                             total_blocks, scale, mask_mode,
                                             sliding_window, dtype, out);
        if (e < 0)
            return e;
        errors += e;
    }
    return errors;
}

/* ------------------------------------------------------------------ */
/* needed_seq and bucket choice, used only to report bytes             */
/* ------------------------------------------------------------------ */

/*
 * [P4 Design / Per-step bucket selection]: needed_seq = max(num_computed) +
 * 1 + num_speculative_tokens; the bucket is the smallest of buckets U
 * {max_model_len} that is >= needed_seq.  buckets must be ascending.
 * Returns the chosen bucket, or -1 if even max_model_len is too small.
 */
int64_t orc_decode_bucket(const int64_t *num_computed, int64_t n,
                          int64_t num_speculative_tokens, const int64_t *buckets,
                          int64_t num_buckets, int64_t max_model_len)
{
    int64_t mx = 0;
    for (int64_t i = 0; i < n; ++i)
        if (num_computed[i] > mx)
            mx = num_computed[i];
    int64_t needed = mx + 1 + num_speculative_tokens;
    for (int64_t k = 0; k < num_buckets; ++k)
        if (buckets[k] >= needed)
            return buckets[k];
    return max_model_len >= needed ? max_model_len : -1;
}
