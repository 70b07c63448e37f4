/* Plain C99 use of the C ABI: both headers compile as C, the library links from
 * C, and the host-side checks answer without a GPU (no call here reaches a
 * kernel: each passes an argument the entry point rejects before any CUDA
 * call).  Exit status 0 on success. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "dspark.h"
#include "dspark_debug.h"

static int check(const char* what, int got, int want) {
    if (got != want) {
        fprintf(stderr, "%s: got %d, want %d\n", what, got, want);
        return 1;
    }
    return 0;
}

int main(void) {
    int bad = 0;
    void* fake = (void*)(uintptr_t)0x1000;
    bad |= strcmp(dspark_status_string(DSPARK_OK), "DSPARK_OK") != 0;
    bad |= check("draft B = 0",
                 dspark_draft_block(0, 7, 64, 8, 16, DSPARK_BF16, fake, fake, fake, fake, fake, 0.0f,
                                    (const int32_t*)fake, 0.7f, 1, (int32_t*)fake, (float*)fake, (float*)fake,
                                    (float*)fake, (float*)fake, fake, (size_t)1 << 30, NULL),
                 DSPARK_ERR_INVALID_ARGUMENT);
    bad |= check("schedule gamma = 33",
                 dspark_schedule_prefix(4, 33, (const float*)fake, (const double*)fake, (int32_t*)fake,
                                        (int32_t*)fake, (double*)fake, fake, 256, NULL),
                 DSPARK_ERR_INVALID_ARGUMENT);
    bad |= check("verify bad dtype",
                 dspark_verify(4, 7, 64, 16, (dspark_dtype_t)7, fake, fake, fake, fake, (const int32_t*)fake,
                               (const int32_t*)fake, (const float*)fake, (const float*)fake,
                               (const int32_t*)fake, 0.7f, 1, (int32_t*)fake, (int32_t*)fake, fake,
                               (size_t)1 << 30, NULL),
                 DSPARK_ERR_INVALID_ARGUMENT);
    bad |= check("tv rows < 0",
                 dspark_accept_rate_tv(-1, 64, DSPARK_BF16, fake, fake, (float*)fake, fake, 256, NULL),
                 DSPARK_ERR_INVALID_ARGUMENT);
    bad |= check("workspace sizes are nonzero",
                 dspark_draft_block_workspace_size(64, 7, 151936, 256) > 0 &&
                     dspark_verify_workspace_size(64, 7, 151936, 256) > 0 &&
                     dspark_schedule_prefix_workspace_size(64, 7) > 0,
                 1);
    return bad;
}
