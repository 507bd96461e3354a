/* A plain C99 client of include/w4a8.h: the header compiles as C, the library links, and the
 * calls that need no GPU (version, status strings, size queries, argument rejection) answer
 * as the header documents.  Prints "ok" and returns 0, or names the first failed check. */
#include <stdio.h>
#include <string.h>

#include "w4a8.h"

#define CHECK(cond)                                          \
    do {                                                     \
        if (!(cond)) {                                       \
            printf("failed: %s (line %d)\n", #cond, __LINE__); \
            return 1;                                        \
        }                                                    \
    } while (0)

int main(void) {
    static float x[4 * 64];
    static unsigned char wq[8 * 32];
    static uint16_t sw[8];
    static float y[4 * 8];
    const size_t bad = (size_t)-1;

    CHECK(w4a8_abi_version() > 0);
    CHECK(strcmp(w4a8_status_string(W4A8_OK), "ok") == 0);
    CHECK(strlen(w4a8_status_string(W4A8_ERR_SHAPE)) > 0);

    /* size queries: empty problems need nothing, a K that is not a multiple of 64 is invalid */
    CHECK(w4a8_prefill_workspace_bytes(0, 8, 64) == 0);
    CHECK(w4a8_linear_workspace_bytes(4, 8, 100) == bad);
    CHECK(w4a8_prefill_host_workspace_bytes(512, 3072, 1024) >= (size_t)512 * (1024 + 3072) * 4);
    CHECK(w4a8_prepared_weights_bytes(8, 64) >= 8 * 64);

    /* argument rejection before any device work */
    CHECK(w4a8_prefill_linear(x, wq, sw, sw, NULL, y, 4, 8, 100, NULL, 0, NULL) == W4A8_ERR_SHAPE);
    CHECK(w4a8_prefill_linear(x, wq, sw, sw, NULL, y, -1, 8, 64, NULL, 0, NULL) == W4A8_ERR_ARG);
    CHECK(w4a8_prefill_linear(NULL, NULL, NULL, NULL, NULL, NULL, 0, 8, 64, NULL, 0, NULL) == W4A8_OK);
    CHECK(w4a8_quant_pack(x, 4, 96, NULL, NULL, NULL, NULL) == W4A8_ERR_SHAPE);
    CHECK(w4a8_prefill_linear_ex(x, wq, sw, sw, NULL, y, 7, -1.0f, 1.0f, 4, 8, 64, NULL, 0, NULL) ==
          W4A8_ERR_ARG);
    CHECK(w4a8_prefill_linear_host(NULL, wq, sw, sw, NULL, y, 4, 8, 64, y, 1024, NULL) == W4A8_ERR_ARG);
    CHECK(w4a8_tape_begin(NULL) == W4A8_ERR_ARG);
    w4a8_tape_free(NULL);

    printf("ok\n");
    return 0;
}
