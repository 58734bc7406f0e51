/*
 * Plain-C client of liblowbit: compiled and linked against include/lowbit.h and
 * the built shared library, it calls the entry points that need no GPU (sizes,
 * status strings, path selection, argument validation) and exits non-zero on
 * the first mismatch.  Run by tests/test_abi_host.py.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "lowbit.h"

#define CHECK(cond)                                                   \
    do {                                                              \
        if (!(cond)) {                                                \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
            return 1;                                                 \
        }                                                             \
    } while (0)

int main(void)
{
    /* K codes of b bits per row, N rows: N*K*b/8 bytes. */
    CHECK(lowbit_packed_bytes(4096, 14336, 3) == (size_t)4096 * 14336 * 3 / 8);
    CHECK(lowbit_packed_bytes(1, 8, 7) == 7);
    CHECK(lowbit_packed_bytes(1, 4, 3) == 0);          /* row not a whole number of bytes */
    CHECK(lowbit_packed_bytes(1, 64, 8) == 0);         /* bit width out of range */

    CHECK(strcmp(lowbit_status_string(LOWBIT_OK), "ok") == 0);
    CHECK(lowbit_status_string((lowbit_status)99) != NULL);

    CHECK(lowbit_select_path(1, 4096, 4096, 4, 64) == LOWBIT_PATH_QMV);
    CHECK(lowbit_select_path(128, 4096, 4096, 4, 128) == LOWBIT_PATH_QMM);
    CHECK(lowbit_select_path(128, 96, 64, 4, 32) == LOWBIT_PATH_QMV);     /* K % 128 != 0 */
    CHECK(lowbit_select_path(1, 4096, 4096, 9, 64) == LOWBIT_PATH_AUTO);  /* rejected */

    /* Argument validation happens before any CUDA call. */
    uint16_t *fake = (uint16_t *)(uintptr_t)0x1000;
    CHECK(lowbit_linear(fake, (const uint8_t *)fake, fake, fake, NULL, fake, 1, 64, 8, 0, 32, NULL)
          == LOWBIT_EINVAL);
    CHECK(lowbit_linear(fake, (const uint8_t *)fake, fake, fake, NULL, fake, 1, 80, 8, 4, 32, NULL)
          == LOWBIT_EINVAL);
    CHECK(lowbit_linear(fake, (const uint8_t *)fake, fake, fake, NULL, fake, 0, 64, 8, 4, 32, NULL)
          == LOWBIT_OK);                               /* empty call */
    CHECK(lowbit_linear_swiglu(fake, (const uint8_t *)fake, fake, fake, NULL, fake, 1, 64, -1, 4, 32, NULL)
          == LOWBIT_EINVAL);
    CHECK(lowbit_pack_weights(NULL, NULL, 4, 8, 0, NULL) == LOWBIT_EINVAL);
    CHECK(lowbit_wait_timeouts(NULL, 0) == LOWBIT_EINVAL);
    printf("c abi ok\n");
    return 0;
}
