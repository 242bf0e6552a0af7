// The bucket all-reduce split across ranks that each hold some of the
// replicas: the ownership plan and the owner's reduction.
//
// "PyTorch Distributed Training Internals", section "3. The All-Reduce
// Itself", describes the all-reduce of a bucket as a reduce-scatter followed
// by an all-gather: every one of G ranks owns one contiguous 1/G chunk of the
// bucket's flat range, ends up with the reduced values of that chunk, and
// then every rank collects every chunk (2(G-1)/G of the bucket's bytes move
// per rank).  "NCCL 专家课程 30", section "Bucket 必须按序发起", fixes the
// order: every rank issues its buckets' collectives in bucket-index order.
//
// Exactness: the reduce-scatter here moves the replicas' raw values
// (all-to-alls of chunks) and the owner sums them itself, replica 0 .. W-1 in
// the one-GPU order, then scales by fl32(1/W) -- the single-GPU pass's
// definition -- so the sharded result equals the one-GPU emulation bit for
// bit.  A ring reduce-scatter would add partial sums in another order.

#include "ddp_reducer.h"

#include <cuda_runtime.h>

#include <cstdint>

#include "ddp_kernels.h"

namespace {

constexpr int64_t kChunkAlign = 8;   // elements: 16 bytes of bf16, 32 of fp32

}  // namespace

extern "C" {

int ddp_shard_range(int64_t n, int32_t G, int32_t g, int64_t* chunk, int64_t* lo, int64_t* hi) {
    if (n < 0 || G < 1 || g < 0 || g >= G) return DDP_ERR_INVALID_ARG;
    // equal chunks of ceil(n / G) elements rounded up to the alignment; the
    // last non-empty chunk takes the remainder, ranks past it own nothing
    const int64_t c = ((n + G - 1) / G + kChunkAlign - 1) / kChunkAlign * kChunkAlign;
    const int64_t a = static_cast<int64_t>(g) * c < n ? static_cast<int64_t>(g) * c : n;
    const int64_t b = static_cast<int64_t>(g + 1) * c < n ? static_cast<int64_t>(g + 1) * c : n;
    if (chunk) *chunk = c;
    if (lo) *lo = a;
    if (hi) *hi = b;
    return DDP_OK;
}

int ddp_shard_mean(int32_t G, ddp_dtype dtype, const void* const* chunks, float* out, int64_t n, void* stream) {
    if (G < 1 || G > ddpk::kMaxHookReplicas || n < 0 || (dtype != DDP_F32 && dtype != DDP_BF16))
        return DDP_ERR_INVALID_ARG;
    if (n == 0) return DDP_OK;
    if (!chunks || !out) return DDP_ERR_INVALID_ARG;
    for (int32_t c = 0; c < G; ++c)
        if (!chunks[c]) return DDP_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DDP_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DDP_ERR_CUDA;
    const ddpk::InType in = dtype == DDP_F32 ? ddpk::IN_F32 : ddpk::IN_BF16;
    const cudaError_t e = ddpk::launch_flat_mean(in, G, chunks, out, n, 1.0f / static_cast<float>(G), 0, sms,
                                                 static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DDP_OK : DDP_ERR_CUDA;
}

}  // extern "C"
