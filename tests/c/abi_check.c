/* A plain C caller of libbkv.so: includes only bkv.h, links only the
 * library, and exercises the calls that are decided on the host (status
 * text, version, argument validation, workspace sizing), so it runs without
 * a GPU.  Prints "ok" and returns 0 when every check holds. */
#include <stdio.h>
#include <string.h>

#include "bkv.h"

static int failures = 0;

static void check(int cond, const char *what) {
    if (!cond) {
        printf("FAILED: %s\n", what);
        ++failures;
    }
}

int main(void) {
    check(strncmp(bkv_version(), "bkv ", 4) == 0, "version string");
    check(strcmp(bkv_status_string(BKV_OK), "ok") == 0, "status text of BKV_OK");
    check(strlen(bkv_status_string(BKV_ERR_INVALID_ARG)) > 0, "status text of BKV_ERR_INVALID_ARG");
    check(strlen(bkv_status_string(12345)) > 0, "status text of an unknown code");

    /* slot mapping: block_size 0, max_num_tokens < num_tokens, nothing to do */
    check(bkv_compute_slot_mapping(NULL, 1, 4, 4, NULL, NULL, 1, 1, 0, NULL, NULL, NULL) == BKV_ERR_INVALID_ARG,
          "slot mapping rejects block_size 0");
    check(bkv_compute_slot_mapping(NULL, 1, 4, 4, NULL, NULL, 5, 4, 16, NULL, NULL, NULL) == BKV_ERR_INVALID_ARG,
          "slot mapping rejects max_num_tokens < num_tokens");
    check(bkv_compute_slot_mapping(NULL, 0, 0, 0, NULL, NULL, 0, 0, 16, NULL, NULL, NULL) == BKV_OK,
          "slot mapping of nothing is ok");

    /* block expansion: indivisible block sizes are an error */
    check(bkv_map_to_kernel_blocks(NULL, 2, 4, 4, 32, 12, NULL, 16, NULL) == BKV_ERR_INVALID_ARG,
          "expansion rejects 32 -> 12");

    /* cache write and the fused write: unsupported dtype, short source stride */
    check(bkv_cache_write(NULL, NULL, 1, 1024, NULL, NULL, NULL, 4, 16, 8, 128, 7, NULL, NULL) == BKV_ERR_UNSUPPORTED,
          "cache write rejects an unknown dtype");
    check(bkv_slot_mapping_cache_write(NULL, 1, 4, 4, NULL, NULL, 1, 1, NULL, NULL, NULL, 1023, NULL, NULL, 4, 16, 8,
                                       128, BKV_BF16, NULL, NULL) == BKV_ERR_INVALID_ARG,
          "fused write rejects a source stride below H_kv * D");

    /* workspace sizing: positive for a valid shape, 0 for an invalid one */
    check(bkv_paged_decode_workspace_size(32, 1, 32, 8, 128, 64, 4097) > 0, "workspace size of the Llama shape");
    check(bkv_paged_decode_workspace_size(32, 1, 30, 8, 128, 64, 4097) == 0, "workspace size with H_q % H_kv != 0");

    /* the decode rejects a too-small workspace before enqueuing anything */
    check(bkv_paged_decode((void *)16, (void *)16, (void *)16, (const int32_t *)16, 4, 4, (const int32_t *)16, 100,
                           2, 1, 8, 2, 128, 16, 10, 0.f, BKV_MASK_CAUSAL, BKV_BF16, (void *)16, (void *)16, 16,
                           NULL, NULL) == BKV_ERR_INVALID_ARG,
          "decode rejects a workspace that is too small");
    check(bkv_paged_decode((void *)16, (void *)16, (void *)16, (const int32_t *)16, 4, 4, (const int32_t *)16, 100,
                           2, 1, 8, 2, 128, 16, 10, 0.f, BKV_MASK_CAUSAL, 7, (void *)16, (void *)16, 1 << 20,
                           NULL, NULL) == BKV_ERR_UNSUPPORTED,
          "decode rejects an unknown dtype");
    /* the sliding-window form: a negative window is invalid */
    check(bkv_paged_decode_swa((void *)16, (void *)16, (void *)16, (const int32_t *)16, 4, 4, (const int32_t *)16,
                               100, 2, 1, 8, 2, 128, 16, 10, 0.f, BKV_MASK_CAUSAL, -1, BKV_BF16, (void *)16,
                               (void *)16, 1 << 20, NULL, NULL) == BKV_ERR_INVALID_ARG,
          "windowed decode rejects a negative window");

    if (failures) return 1;
    printf("ok\n");
    return 0;
}
