/* A plain C99 consumer of the C ABI in include/ddp_reducer.h: bucket
 * assignment, locators and the readiness state machine (dry run, so no GPU
 * is needed), driven through the exported symbols only.
 *
 * Model: 6 fp32 tensors of 100 .. 600 elements, cap 2000 bytes.  The reverse
 * walk closes a bucket once its bytes reach the cap: {5} (2400 B), {4} (2000
 * B), {3, 2} (2800 B), and the remainder {1, 0}.  Reporting the variables in
 * forward order parks buckets 3, 2 and 1 until bucket 0 completes; the last
 * event then releases all four, in index order, in one run.
 * Prints "c abi ok" and exits 0 when every check holds. */

#include <stdint.h>
#include <stdio.h>

#include "ddp_reducer.h"

static int failures = 0;

#define CHECK(cond)                                                   \
    do {                                                              \
        if (!(cond)) {                                                \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
            ++failures;                                               \
        }                                                             \
    } while (0)

int main(void) {
    const int64_t numel[6] = {100, 200, 300, 400, 500, 600};
    ddp_ctx* ctx = NULL;
    CHECK(ddp_build_buckets(numel, 6, DDP_F32, 2000, &ctx) == DDP_OK);
    if (!ctx) return 1;

    int32_t B = 0;
    int64_t offs[5] = {0};
    CHECK(ddp_get_bucket_info(ctx, &B, offs) == DDP_OK);
    CHECK(B == 4);
    const int64_t want_offs[5] = {0, 600, 1100, 1800, 2100};
    for (int b = 0; b <= 4; ++b) CHECK(offs[b] == want_offs[b]);

    ddp_locator loc[6];
    CHECK(ddp_get_locators(ctx, loc) == DDP_OK);
    /* variable: bucket, push position, offset in the bucket, length */
    const int64_t want[6][4] = {{3, 1, 200, 100}, {3, 0, 0, 200}, {2, 1, 400, 300},
                                {2, 0, 0, 400},   {1, 0, 0, 500}, {0, 0, 0, 600}};
    for (int v = 0; v < 6; ++v) {
        CHECK(loc[v].bucket == want[v][0]);
        CHECK(loc[v].intra == want[v][1]);
        CHECK(loc[v].offset == want[v][2]);
        CHECK(loc[v].length == want[v][3]);
    }

    /* dry run: the state machine runs, nothing is launched, the pointers are
     * only recorded (stand-in addresses, 16-byte aligned arena) */
    CHECK(ddp_set_option(ctx, DDP_OPT_DRY_RUN, 1) == DDP_OK);
    const void* grads[2 * 6];
    for (int i = 0; i < 12; ++i) grads[i] = (const void*)(uintptr_t)(0x100000u + 0x10000u * (unsigned)i);
    CHECK(ddp_bind(ctx, 2, grads, (float*)(uintptr_t)0x4000000u, NULL, 0) == DDP_OK);

    int32_t launched[4];
    int32_t n = -1;
    CHECK(ddp_begin_iteration(ctx) == DDP_OK);
    for (int32_t v = 0; v < 5; ++v) {
        CHECK(ddp_mark_ready(ctx, v, launched, &n, NULL) == DDP_OK);
        CHECK(n == 0);                          /* buckets 3, 2, 1 park */
    }
    int32_t next = -1, parked[4], n_parked = -1;
    CHECK(ddp_get_progress(ctx, &next, parked, &n_parked) == DDP_OK);
    CHECK(next == 0 && n_parked == 3 && parked[0] == 1 && parked[1] == 2 && parked[2] == 3);
    CHECK(ddp_mark_ready(ctx, 0, launched, &n, NULL) == DDP_ERR_ALREADY_READY);
    CHECK(ddp_mark_ready(ctx, 5, launched, &n, NULL) == DDP_OK);
    CHECK(n == 4);
    for (int b = 0; b < 4 && n == 4; ++b) CHECK(launched[b] == b);
    /* the iteration finished, so the next one may begin */
    CHECK(ddp_begin_iteration(ctx) == DDP_OK);
    CHECK(ddp_status_string(DDP_ERR_ALREADY_READY) != NULL);

    /* launch options of the batched call and of built-in hooks */
    int64_t value = -1;
    CHECK(ddp_get_option(ctx, DDP_OPT_COALESCE_ELEMS, &value) == DDP_OK && value == (int64_t)1 << 21);
    CHECK(ddp_set_option(ctx, DDP_OPT_COALESCE_ELEMS, -1) == DDP_ERR_INVALID_ARG);
    CHECK(ddp_get_option(ctx, DDP_OPT_HOOK_FUSED, &value) == DDP_OK && value == 1);

    /* ownership plan of the all-reduce across ranks: 100 elements over 3
     * ranks -> chunks of 40 (ceil(100 / 3) = 34, rounded up to 8) */
    int64_t chunk = 0, lo = -1, hi = -1, at = 0;
    for (int32_t g = 0; g < 3; ++g) {
        CHECK(ddp_shard_range(100, 3, g, &chunk, &lo, &hi) == DDP_OK);
        CHECK(chunk == 40 && lo == at);
        at = hi;
    }
    CHECK(at == 100 && lo == 80);
    CHECK(ddp_shard_range(100, 3, 3, &chunk, &lo, &hi) == DDP_ERR_INVALID_ARG);

    ddp_destroy(ctx);
    if (failures) return 1;
    printf("c abi ok\n");
    return 0;
}
