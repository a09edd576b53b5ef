/* Calls the h3attn C ABI from plain C (C99, gcc): the header must compile as C
 * and the library must link and answer without a GPU -- version, status
 * strings, build flags, and argument checks that refuse a call before any
 * CUDA work.  Exit status 0 = every check passed. */
#include <stdio.h>
#include <string.h>

#include "h3attn.h"

static int failures = 0;
#define CHECK(cond)                                                        \
    do {                                                                   \
        if (!(cond)) {                                                     \
            fprintf(stderr, "check failed: %s (line %d)\n", #cond, __LINE__); \
            ++failures;                                                    \
        }                                                                  \
    } while (0)

int main(void) {
    void *fake = (void *)0x10000; /* aligned, never dereferenced: refused first */
    void *fake2 = (void *)0x20000000;
    int32_t kv_bad[1] = {0};
    CHECK(h3attn_version() == H3ATTN_VERSION);
    CHECK(strcmp(h3attn_strerror(H3ATTN_OK), "ok") == 0);
    CHECK(strstr(h3attn_strerror(H3ATTN_ERR_DEVICE_TIMEOUT), "timeout") != NULL);
    CHECK(h3attn_build_flags() == 0);
    CHECK(h3attn_last_cuda_error() == 0);
    /* null q */
    CHECK(h3attn_forward(NULL, fake, fake, fake2, 1, 256, 4, 64, 0, 4, NULL, 0.0f, NULL) == H3ATTN_ERR_ARG);
    /* head_dim 96 is not supported */
    CHECK(h3attn_forward(fake, fake, fake, fake2, 1, 256, 4, 96, 0, 4, NULL, 0.0f, NULL) == H3ATTN_ERR_SHAPE);
    /* kv_len outside [1, S] */
    CHECK(h3attn_forward(fake, fake, fake, fake2, 1, 256, 4, 64, 0, 4, kv_bad, 0.0f, NULL) == H3ATTN_ERR_SHAPE);
    /* H % P != 0 for the exchange */
    CHECK(h3attn_seq2head(fake, fake2, 64, 56, 128, 3, NULL) == H3ATTN_ERR_SHAPE);
    /* d_t + d_h + d_w != D */
    CHECK(h3attn_qk_norm_rope(fake, fake2, fake2, fake2, NULL, fake, fake, fake, 1, 16, 4, 64, 16, 24, 22, 1e-6f,
                              1e4f, NULL) == H3ATTN_ERR_SHAPE);
    CHECK(h3attn_selftest_wait_timeout(0, NULL) == H3ATTN_ERR_ARG);
    if (failures == 0) printf("abi_from_c ok\n");
    return failures == 0 ? 0 : 1;
}
