/* A plain C caller of the four hot-path calls with the argument lists of the
 * library's boundary statement, declared here by hand (no bkv.h), so that a
 * caller written against that statement alone is what gets tested.
 *
 * Usage: sec8b_caller IN OUT
 * IN  holds 16 int64 sizes, then the arrays (each at an 8-byte aligned
 *     offset): manager block table int32 [R][mcols], request indices int32
 *     [T], positions int64 [T], new K and V rows [T][H_kv][D] of the element
 *     type, queries [R][q_len][H_q][D], context lengths int32 [R].
 * OUT receives the kernel block table int32 [R][mcols * bpk], the slot
 *     mapping int64 [max_tokens], the attention output [R][q_len][H_q][D]
 *     and the int32 error count.
 * The caches start as all-ones bytes (NaN in bf16 and fp32), are filled by
 * the slot mapping + cache write of all T tokens, then decoded.  Exit code 0
 * when every call returned 0 and the files could be read and written. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

int bkv_compute_slot_mapping(const int32_t *block_table, int32_t num_reqs, int64_t bt_stride, int32_t bt_cols,
                             const int32_t *req_indices, const int64_t *positions, int64_t num_tokens,
                             int64_t max_num_tokens, int32_t block_size, int64_t *slot_mapping, int32_t *err_count,
                             cudaStream_t stream);
int bkv_map_to_kernel_blocks(const int32_t *mgr_table, int32_t rows, int64_t mgr_stride, int32_t mgr_cols,
                             int32_t block_size, int32_t kernel_block_size, int32_t *kernel_table,
                             int64_t kernel_stride, cudaStream_t stream);
int bkv_cache_write(const void *k_new, const void *v_new, int64_t num_tokens, int64_t new_token_stride,
                    const int64_t *slot_mapping, void *k_cache, void *v_cache, int64_t total_blocks,
                    int32_t block_size, int32_t num_kv_heads, int32_t head_dim, int dtype, int32_t *err_count,
                    cudaStream_t stream);
size_t bkv_paged_decode_workspace_size(int32_t num_reqs, int32_t q_len, int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t block_size, int32_t max_context_len);
int bkv_paged_decode(const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
                     int64_t bt_stride, int32_t bt_cols, const int32_t *context_lens, int32_t max_context_len,
                     int32_t num_reqs, int32_t q_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                     int32_t block_size, int64_t total_blocks, float softmax_scale, int mask_mode, int dtype,
                     void *out, void *workspace, size_t workspace_bytes, int32_t *err_count, cudaStream_t stream);

static int fail(const char *what, long long code) {
    fprintf(stderr, "FAILED: %s (%lld)\n", what, code);
    return 1;
}

#define CUDA(x)                                                         \
    do {                                                                \
        cudaError_t e_ = (x);                                           \
        if (e_ != cudaSuccess) return fail(#x, (long long)e_);          \
    } while (0)
#define BKV(x)                                                          \
    do {                                                                \
        int s_ = (x);                                                   \
        if (s_ != 0) return fail(#x, (long long)s_);                    \
    } while (0)

static size_t up8(size_t n) { return (n + 7) & ~(size_t)7; }

/* copy n bytes from the input buffer at *off to a new device allocation */
static int upload(const char *buf, size_t *off, size_t n, void **dev) {
    CUDA(cudaMalloc(dev, n > 0 ? n : 16));
    if (n) CUDA(cudaMemcpy(*dev, buf + *off, n, cudaMemcpyHostToDevice));
    *off += up8(n);
    return 0;
}

int main(int argc, char **argv) {
    if (argc != 3) return fail("usage: sec8b_caller IN OUT", 0);
    FILE *f = fopen(argv[1], "rb");
    if (!f) return fail("open IN", 0);
    fseek(f, 0, SEEK_END);
    const long len = ftell(f);
    fseek(f, 0, SEEK_SET);
    char *buf = (char *)malloc((size_t)len);
    if (!buf || fread(buf, 1, (size_t)len, f) != (size_t)len) return fail("read IN", len);
    fclose(f);

    int64_t sz[16];
    memcpy(sz, buf, sizeof sz);
    const int32_t R = (int32_t)sz[0], mcols = (int32_t)sz[1], bs = (int32_t)sz[2], kbs = (int32_t)sz[3];
    const int64_t T = sz[4], max_tokens = sz[5];
    const int32_t H_q = (int32_t)sz[6], H_kv = (int32_t)sz[7], D = (int32_t)sz[8], q_len = (int32_t)sz[9];
    const int64_t total_mgr = sz[10];
    const int dtype = (int)sz[11];
    const int32_t max_ctx = (int32_t)sz[12];
    const int mask_mode = (int)sz[13];
    const size_t e = dtype == 0 ? 2 : 4;
    const int32_t bpk = bs / kbs;
    const int32_t kcols = mcols * bpk;
    const int64_t total_k = total_mgr * bpk;

    size_t off = sizeof sz;
    void *d_mgr, *d_req, *d_pos, *d_k, *d_v, *d_q, *d_ctx;
    if (upload(buf, &off, (size_t)R * mcols * 4, &d_mgr) || upload(buf, &off, (size_t)T * 4, &d_req) ||
        upload(buf, &off, (size_t)T * 8, &d_pos) || upload(buf, &off, (size_t)T * H_kv * D * e, &d_k) ||
        upload(buf, &off, (size_t)T * H_kv * D * e, &d_v) ||
        upload(buf, &off, (size_t)R * q_len * H_q * D * e, &d_q) || upload(buf, &off, (size_t)R * 4, &d_ctx))
        return 1;
    if (off != (size_t)len) return fail("input size", (long long)off);

    const size_t cache_bytes = (size_t)total_k * kbs * H_kv * D * e;
    const size_t out_bytes = (size_t)R * q_len * H_q * D * e;
    void *d_kt, *d_slots, *d_kc, *d_vc, *d_out, *d_err, *d_ws = NULL;
    CUDA(cudaMalloc(&d_kt, (size_t)R * kcols * 4));
    CUDA(cudaMalloc(&d_slots, (size_t)max_tokens * 8));
    CUDA(cudaMalloc(&d_kc, cache_bytes));
    CUDA(cudaMalloc(&d_vc, cache_bytes));
    CUDA(cudaMalloc(&d_out, out_bytes));
    CUDA(cudaMalloc(&d_err, 4));
    CUDA(cudaMemset(d_kc, 0xFF, cache_bytes));
    CUDA(cudaMemset(d_vc, 0xFF, cache_bytes));
    CUDA(cudaMemset(d_err, 0, 4));
    const size_t ws_bytes = bkv_paged_decode_workspace_size(R, q_len, H_q, H_kv, D, kbs, max_ctx);
    if (ws_bytes == 0) return fail("workspace size", 0);
    CUDA(cudaMalloc(&d_ws, ws_bytes));
    cudaStream_t st;
    CUDA(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));

    BKV(bkv_map_to_kernel_blocks((const int32_t *)d_mgr, R, mcols, mcols, bs, kbs, (int32_t *)d_kt, kcols, st));
    BKV(bkv_compute_slot_mapping((const int32_t *)d_kt, R, kcols, kcols, (const int32_t *)d_req,
                                 (const int64_t *)d_pos, T, max_tokens, kbs, (int64_t *)d_slots, (int32_t *)d_err,
                                 st));
    BKV(bkv_cache_write(d_k, d_v, T, (int64_t)H_kv * D, (const int64_t *)d_slots, d_kc, d_vc, total_k, kbs, H_kv, D,
                        dtype, (int32_t *)d_err, st));
    BKV(bkv_paged_decode(d_q, d_kc, d_vc, (const int32_t *)d_kt, kcols, kcols, (const int32_t *)d_ctx, max_ctx, R,
                         q_len, H_q, H_kv, D, kbs, total_k, 0.f, mask_mode, dtype, d_out, d_ws, ws_bytes,
                         (int32_t *)d_err, st));
    CUDA(cudaStreamSynchronize(st));

    const size_t kt_bytes = (size_t)R * kcols * 4, sl_bytes = (size_t)max_tokens * 8;
    char *res = (char *)malloc(kt_bytes + sl_bytes + out_bytes + 4);
    if (!res) return fail("malloc", 0);
    CUDA(cudaMemcpy(res, d_kt, kt_bytes, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(res + kt_bytes, d_slots, sl_bytes, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(res + kt_bytes + sl_bytes, d_out, out_bytes, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(res + kt_bytes + sl_bytes + out_bytes, d_err, 4, cudaMemcpyDeviceToHost));
    FILE *g = fopen(argv[2], "wb");
    if (!g || fwrite(res, 1, kt_bytes + sl_bytes + out_bytes + 4, g) != kt_bytes + sl_bytes + out_bytes + 4)
        return fail("write OUT", 0);
    fclose(g);
    cudaStreamDestroy(st);
    printf("ok\n");
    return 0;
}
