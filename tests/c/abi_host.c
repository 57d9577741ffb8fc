/* Uses the library's C ABI from plain C, with no Python and no GPU: sizes, the host twin of
 * the planner, status strings, and host-side argument checks.  Exit code 0 when every
 * check holds; the failing check's line otherwise. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "mla_decode.h"

#define CHECK(c)                                                  \
    do {                                                          \
        if (!(c)) {                                               \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #c); \
            return __LINE__;                                      \
        }                                                         \
    } while (0)

int main(void) {
    const int B = 64, H = 128, sms = 152;
    int32_t seq_lens[64];
    for (int b = 0; b < B; ++b) seq_lens[b] = 1024 + 97 * b;
    const size_t ws = mla_decode_workspace_size(B, H, sms);
    CHECK(ws > 0);
    CHECK(mla_decode_workspace_size(0, H, sms) == 0);
    void *buf = calloc(1, ws);
    CHECK(buf != NULL);
    CHECK(mla_decode_plan_host(seq_lens, B, H, 0, MLA_KV_BF16, sms, buf, ws) == MLA_OK);
    CHECK(mla_decode_plan_host(seq_lens, B, H, 0, MLA_KV_FP8_E4M3, sms, buf, ws) == MLA_OK);
    CHECK(mla_decode_plan_host(seq_lens, B, H, 0, MLA_KV_BF16, sms, buf, 16) == MLA_ERR_WORKSPACE);
    CHECK(mla_decode_plan_host(NULL, B, H, 0, MLA_KV_BF16, sms, buf, ws) == MLA_ERR_INVALID_ARG);
    CHECK(strcmp(mla_status_string(MLA_OK), "unknown status") != 0);
    CHECK(strcmp(mla_status_string((mla_status)99), "unknown status") == 0);
    /* host-side rejections happen before any device work */
    CHECK(mla_absorb_query(NULL, NULL, B, H, NULL, NULL, NULL) == MLA_ERR_INVALID_ARG);
    CHECK(mla_topk_select(NULL, 64, 64, NULL, B, 8, NULL, NULL, NULL) == MLA_ERR_INVALID_ARG);
    CHECK(mla_prefill_attention(NULL, NULL, NULL, NULL, NULL, 16, H, 0.07f, NULL, NULL, NULL, NULL) ==
          MLA_ERR_INVALID_ARG);
    CHECK(mla_decode_set_wait_limit(-1) == MLA_ERR_INVALID_ARG);
    CHECK(mla_decode_set_wait_limit(0) == MLA_OK); /* the default */
    free(buf);
    printf("c abi ok: workspace %zu bytes\n", ws);
    return 0;
}
