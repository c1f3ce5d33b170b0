/*
 * abi_check.c -- a plain C99 consumer of include/linrec.h, linked against
 * liblinrec.so.  It needs no GPU: it runs only calls that return before any
 * CUDA call (version, status strings, the dispatcher, argument checks) and
 * prints "abi_check: ok", or the first mismatch and exits 1.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "linrec.h"

static int failures = 0;

#define EXPECT(cond)                                                        \
    do {                                                                    \
        if (!(cond)) {                                                      \
            fprintf(stderr, "abi_check: %s:%d: %s\n", __FILE__, __LINE__, #cond); \
            ++failures;                                                     \
        }                                                                   \
    } while (0)

int main(void) {
    EXPECT(linrec_version() >= 100);
    EXPECT(linrec_debug_checks() == 0);
    for (int s = LINREC_OK; s <= LINREC_ERR_TMA_TIMEOUT; ++s) {
        const char *name = linrec_status_string((linrec_status_t)s);
        EXPECT(name != NULL && strlen(name) > 0);
    }

    /* the dispatcher, on the (32, 4096, 256) shape of the pages: slice-owner chunked tiles of 64 channels */
    linrec_options_t opt;
    memset(&opt, 0, sizeof(opt));
    linrec_plan_t plan;
    memset(&plan, 0, sizeof(plan));
    EXPECT(linrec_plan_f32(32, 4096, 256, 152, 16, 0, &opt, &plan) == LINREC_OK);
    EXPECT(plan.path == LINREC_PATH_CHUNKED && plan.lookback == 0 && plan.twopass == 0 && plan.blocks == 0);
    EXPECT(plan.tile_d == 64 && plan.chunks * plan.tile_t >= 4096 && plan.grid == 128);
    EXPECT(plan.chain == 0 && plan.speculative == 0);
    EXPECT(plan.n_tiles == (int64_t)32 * (256 / plan.tile_d) * plan.chunks);
    /* one long sequence: the speculative mode, 128 segments of 8192 steps */
    EXPECT(linrec_plan_f32(1, (int64_t)1 << 20, 64, 152, 16, 0, &opt, &plan) == LINREC_OK);
    EXPECT(plan.speculative == 128 && plan.twopass == 0 && plan.chunks == 64 && plan.grid == 256);
    /* an option no input can take is refused */
    opt.chunk_mode = 9;
    EXPECT(linrec_plan_f32(32, 4096, 256, 152, 16, 0, &opt, &plan) == LINREC_ERR_INVALID_VALUE);

    /* argument checks: fake, never-dereferenced addresses */
    const float *a = (const float *)(uintptr_t)((uint64_t)1 << 36);
    const float *b = a + (1 << 20);
    float *h = (float *)(uintptr_t)((uint64_t)1 << 37);
    EXPECT(linrec_scan_f32(a, b, h, -1, 4, 4, NULL) == LINREC_ERR_INVALID_VALUE);
    EXPECT(linrec_scan_f32(NULL, NULL, NULL, 0, 4, 4, NULL) == LINREC_OK);
    EXPECT(linrec_scan_f32(a, NULL, h, 1, 4, 4, NULL) == LINREC_ERR_INVALID_VALUE);
    EXPECT(linrec_scan_f32(a, b, (float *)(uintptr_t)(a + 2), 1, 4, 4, NULL) == LINREC_ERR_ALIAS);
    EXPECT(linrec_scan_f32((const float *)(uintptr_t)16, b, h, (int64_t)1 << 20, (int64_t)1 << 20,
                           (int64_t)1 << 22, NULL) == LINREC_ERR_INVALID_VALUE);
    EXPECT(linrec_workspace_bytes(-1, 4, 4) == 0);

    if (failures) return 1;
    printf("abi_check: ok\n");
    return 0;
}
