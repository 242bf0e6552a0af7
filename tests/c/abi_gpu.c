/* A plain C consumer of the C ABI on the GPU, without Python or PyTorch:
 * device memory from cudaMalloc, one iteration through the readiness state
 * machine, results copied back and checked.
 *
 * W = 4 replicas of 5 fp32 tensors (sizes 1000, 3, 70001, 0, 64; cap 64 KiB).
 * Replica r holds (i mod 7) + r at element i of its flat buffer, so every sum
 * is an exact small integer and the mean is exactly (4 (i mod 7) + 6) / 4.
 * Prints "c abi gpu ok" and exits 0 when every element of every copy-back and
 * of the bucket arena holds that value. */

#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "ddp_reducer.h"

#define P 5
#define W 4

static int fail(const char* what) {
    fprintf(stderr, "failed: %s\n", what);
    return 1;
}

int main(void) {
    const int64_t numel[P] = {1000, 3, 70001, 0, 64};
    int64_t off[P], total = 0;
    for (int v = 0; v < P; ++v) {
        off[v] = total;
        total += (numel[v] + 63) / 64 * 64;          /* 256-byte starts, as separate allocations */
    }
    ddp_ctx* ctx = NULL;
    if (ddp_build_buckets(numel, P, DDP_F32, 64 << 10, &ctx) != DDP_OK) return fail("build");
    int32_t B = 0;
    if (ddp_get_bucket_info(ctx, &B, NULL) != DDP_OK || B < 1) return fail("bucket info");
    int64_t* boff = (int64_t*)malloc(sizeof(int64_t) * (size_t)(B + 1));
    ddp_get_bucket_info(ctx, &B, boff);
    const int64_t arena_n = boff[B];

    float* host = (float*)malloc(sizeof(float) * (size_t)total);
    float* grad_dev[W];
    for (int r = 0; r < W; ++r) {
        for (int64_t i = 0; i < total; ++i) host[i] = (float)(i % 7 + r);
        if (cudaMalloc((void**)&grad_dev[r], sizeof(float) * (size_t)total) != cudaSuccess) return fail("malloc grads");
        cudaMemcpy(grad_dev[r], host, sizeof(float) * (size_t)total, cudaMemcpyHostToDevice);
    }
    float *arena = NULL, *out = NULL;
    if (cudaMalloc((void**)&arena, sizeof(float) * (size_t)arena_n) != cudaSuccess) return fail("malloc arena");
    if (cudaMalloc((void**)&out, sizeof(float) * (size_t)total) != cudaSuccess) return fail("malloc out");
    cudaMemset(out, 0xFF, sizeof(float) * (size_t)total);

    const void* grads[W * P];
    float* outs[P];
    for (int r = 0; r < W; ++r)
        for (int v = 0; v < P; ++v) grads[r * P + v] = grad_dev[r] + off[v];
    for (int v = 0; v < P; ++v) outs[v] = out + off[v];
    if (ddp_bind(ctx, W, grads, arena, outs, 1) != DDP_OK) return fail(ddp_last_error(ctx));

    int32_t order[P], done = 0;
    for (int v = 0; v < P; ++v) order[v] = P - 1 - v;
    if (ddp_begin_iteration(ctx) != DDP_OK) return fail("begin");
    if (ddp_mark_ready_many(ctx, order, P, &done, NULL) != DDP_OK || done != P) return fail(ddp_last_error(ctx));
    if (cudaDeviceSynchronize() != cudaSuccess) return fail("synchronize");
    int32_t status = -1;
    if (ddp_get_device_status(ctx, &status) != DDP_OK || status != 0) return fail("device status");

    float* back = (float*)malloc(sizeof(float) * (size_t)total);
    cudaMemcpy(back, out, sizeof(float) * (size_t)total, cudaMemcpyDeviceToHost);
    for (int v = 0; v < P; ++v)
        for (int64_t j = 0; j < numel[v]; ++j) {
            const int64_t i = off[v] + j;
            const float want = (float)(4 * (i % 7) + 6) / 4.0f;
            if (back[i] != want) {
                fprintf(stderr, "variable %d element %lld: %g, want %g\n", v, (long long)j, back[i], want);
                return 1;
            }
        }
    /* the bucket arena holds the same means at each variable's locator */
    ddp_locator loc[P];
    ddp_get_locators(ctx, loc);
    float* ar = (float*)malloc(sizeof(float) * (size_t)(arena_n > 0 ? arena_n : 1));
    cudaMemcpy(ar, arena, sizeof(float) * (size_t)arena_n, cudaMemcpyDeviceToHost);
    for (int v = 0; v < P; ++v)
        for (int64_t j = 0; j < numel[v]; ++j) {
            const int64_t i = off[v] + j;
            if (ar[boff[loc[v].bucket] + loc[v].offset + j] != (float)(4 * (i % 7) + 6) / 4.0f) return fail("arena");
        }

    ddp_destroy(ctx);
    for (int r = 0; r < W; ++r) cudaFree(grad_dev[r]);
    cudaFree(arena);
    cudaFree(out);
    free(host);
    free(back);
    free(ar);
    free(boff);
    printf("c abi gpu ok\n");
    return 0;
}
