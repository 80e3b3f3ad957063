/* A plain C consumer of the library: no C++, no Python, no torch. It includes
 * the public header, links libw4a16.so and exercises the calls that need no
 * device work: status strings, set-up (W4_OK with a GPU, W4_ERR_NO_DEVICE
 * without one) and argument validation, which runs before any launch. */
#include <stdio.h>
#include <string.h>

#include "w4a16.h"

int main(void)
{
    if (strcmp(w4_status_string(W4_OK), "W4_OK") != 0 ||
        strcmp(w4_status_string(W4_ERR_MISALIGNED), "W4_ERR_MISALIGNED") != 0) {
        fprintf(stderr, "status strings\n");
        return 1;
    }
    const int init = w4_init();
    if (init != W4_OK && init != W4_ERR_NO_DEVICE) {
        fprintf(stderr, "w4_init: %d (%s)\n", init, w4_status_string(init));
        return 2;
    }
    /* NULL output: rejected by validation, no device touched. */
    if (w4a16_gemv(NULL, NULL, NULL, NULL, 1, 16, 64, 32, NULL) != W4_ERR_INVALID_ARG) {
        fprintf(stderr, "validation\n");
        return 3;
    }
    /* An unsupported group size. */
    char buf[64] __attribute__((aligned(16)));
    if (w4a16_gemv((float *)buf, (const uint16_t *)buf, (const uint32_t *)buf, (const uint16_t *)buf, 1, 16,
                   96, 48, NULL) != W4_ERR_UNSUPPORTED) {
        fprintf(stderr, "group check\n");
        return 4;
    }
    printf("c consumer ok (w4_init = %s)\n", w4_status_string(init));
    return 0;
}
