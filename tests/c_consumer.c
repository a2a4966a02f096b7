/* A C99 program using the library through include/gemm.h only, as a C caller
 * would.  It exercises what needs no GPU: status strings, argument checks that
 * return before any device work, no-op sizes, the per-thread stream and the
 * launch counter.  Prints "ok" and exits 0, or names the failed check and
 * exits 1. */
#include <stdio.h>
#include <string.h>

#include "gemm.h"

static int failures = 0;

#define CHECK(cond)                                                  \
    do {                                                             \
        if (!(cond)) {                                               \
            fprintf(stderr, "check failed: %s (line %d)\n", #cond, __LINE__); \
            ++failures;                                              \
        }                                                            \
    } while (0)

int main(void)
{
    static float fbuf[4096];
    static uint16_t hbuf[4096];
    const unsigned long long launches = gemm_kernel_launches();

    CHECK(strcmp(gemm_status_string(GEMM_OK), "GEMM_OK") == 0);
    CHECK(strcmp(gemm_status_string(GEMM_ERR_ALIAS), "GEMM_ERR_ALIAS") == 0);
    CHECK(strcmp(gemm_status_string((gemm_status_t)99), "GEMM_ERR_UNKNOWN") == 0);

    /* negative sizes are rejected on the host */
    CHECK(gemm_f32_rm(fbuf, fbuf + 1024, fbuf + 2048, -1, 4, 4) == GEMM_ERR_INVALID_VALUE);
    CHECK(gemm_f16_cm(hbuf, hbuf + 1024, hbuf + 2048, 4, -4, 4) == GEMM_ERR_INVALID_VALUE);
    CHECK(gemm_bf16_rm(hbuf, hbuf + 1024, hbuf + 2048, 4, 4, -4) == GEMM_ERR_INVALID_VALUE);
    CHECK(gemm_last_error() != NULL);

    /* the general form's enums and leading dimensions */
    CHECK(gemm_ex((gemm_dtype_t)3, GEMM_ROW_MAJOR, GEMM_OP_N, GEMM_OP_N, 4, 4, 4, 1.0f, fbuf, 4, 0,
                  fbuf + 1024, 4, 0, 0.0f, fbuf + 2048, 4, 16, 1) == GEMM_ERR_INVALID_VALUE);
    CHECK(gemm_ex(GEMM_F32, GEMM_ROW_MAJOR, GEMM_OP_N, GEMM_OP_N, 4, 4, 4, 1.0f, fbuf, 3, 0,
                  fbuf + 1024, 4, 0, 0.0f, fbuf + 2048, 4, 16, 1) == GEMM_ERR_INVALID_VALUE);
    CHECK(gemm_ex(GEMM_F32, GEMM_ROW_MAJOR, GEMM_OP_N, GEMM_OP_N, 4, 4, 4, 1.0f, fbuf, 4, 0,
                  fbuf + 1024, 4, 0, 0.0f, fbuf + 2, 4, 16, 1) == GEMM_ERR_ALIAS);

    /* M = 0 is a no-op that succeeds without a device */
    CHECK(gemm_ex(GEMM_BF16, GEMM_COL_MAJOR, GEMM_OP_T, GEMM_OP_N, 0, 4, 4, 1.0f, hbuf, 4, 0,
                  hbuf + 1024, 4, 0, 0.0f, hbuf + 2048, 4, 16, 1) == GEMM_OK);
    CHECK(strcmp(gemm_last_kernel(), "noop") == 0);

    /* an unknown kernel family is refused; clearing the choice is not */
    CHECK(gemm_force_kernel("cpu") == GEMM_ERR_INVALID_VALUE);
    CHECK(gemm_force_kernel(NULL) == GEMM_OK);

    /* the calling thread's stream round-trips */
    CHECK(gemm_set_stream(NULL) == GEMM_OK);
    CHECK(gemm_get_stream() == NULL);

    /* nothing above launched a kernel */
    CHECK(gemm_kernel_launches() == launches);

    if (failures) return 1;
    printf("ok\n");
    return 0;
}
