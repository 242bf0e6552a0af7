// ddp_reduce_all_noalloc: the fused bucket pass over every bucket with no
// device allocation at all.
//
// Some callers cannot call cudaMalloc: a framework whose caching allocator
// already owns the whole device memory budget, and real-time loops where an
// allocation (and the device synchronisation it implies) is not allowed.
// This entry point serves them: the caller passes the gradients and the
// outputs, and the segment table that the ordinary path keeps in a
// cudaMalloc'd block (made by ddp_bind) lives instead in a fixed array in the
// library's static device memory, sized once for every process.  The launch
// shape is fixed (the context's options are not read), and the status word
// of the kernel's bounded waits is not reported to the caller.

#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>

#include "ddp_kernels.h"
#include "ddp_layout.h"
#include "ddp_reducer.h"

namespace {

constexpr size_t kScratchBytes = DDP_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The device-side table: every GPU that loads the library holds this array
// until the process exits.  Host code must never pass its name to a kernel
// (on the host it is only a stand-in); it uses the address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Host staging copy of the table, and the per-device scratch addresses.
alignas(256) unsigned char g_host_table[kScratchBytes];
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_mutex;

size_t up16(size_t x) { return (x + 15) / 16 * 16; }

int fail(ddp_ctx* c, int status, const std::string& msg) {
    ddp_internal::set_error(c, msg);
    return status;
}

int cuda_fail(ddp_ctx* c, cudaError_t e, const char* where) {
    return fail(c, DDP_ERR_CUDA, std::string(where) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

}  // namespace

extern "C" int ddp_reduce_all_noalloc(ddp_ctx* ctx, int32_t W, const void* const* grads, float* bucket_arena,
                                      float* const* grad_out, int32_t n_out, void* stream) {
    if (!ctx) return DDP_ERR_INVALID_ARG;
    const ddp_internal::Layout L = ddp_internal::layout(ctx);
    if (W < 1) return fail(ctx, DDP_ERR_INVALID_ARG, "W must be >= 1");
    if (n_out != 0 && n_out != 1 && n_out != W) return fail(ctx, DDP_ERR_INVALID_ARG, "n_out must be 0, 1 or W");
    if (L.P > 0 && !grads) return fail(ctx, DDP_ERR_INVALID_ARG, "grads is NULL");
    if (n_out > 0 && L.P > 0 && !grad_out) return fail(ctx, DDP_ERR_INVALID_ARG, "grad_out is NULL with n_out > 0");
    const int64_t total = L.bucket_off[L.B];
    if (total > 0 && !bucket_arena) return fail(ctx, DDP_ERR_INVALID_ARG, "bucket_arena is NULL");
    if (reinterpret_cast<uintptr_t>(bucket_arena) & 15u)
        return fail(ctx, DDP_ERR_INVALID_ARG, "bucket_arena must be 16-byte aligned");

    // One segment per non-empty variable, buckets in index order, members in
    // push order: exactly the arena layout.
    size_t S = 0;
    for (int32_t v = 0; v < L.P; ++v)
        if (L.numel[v] > 0) ++S;
    const size_t b_status = 16;
    const size_t b_off = up16((S + 1) * sizeof(int64_t));
    const size_t b_src = up16(S * W * sizeof(void*));
    const size_t b_dst = up16(S * n_out * sizeof(float*));
    const size_t b_vec = up16((S > 0 ? S : 1) * sizeof(int32_t));
    const size_t bytes = b_status + b_off + b_src + b_dst + b_vec;
    if (bytes > kScratchBytes)
        return fail(ctx, DDP_ERR_INVALID_ARG,
                    "segment table needs " + std::to_string(bytes) + " bytes; the static scratch holds " +
                        std::to_string(kScratchBytes) + " (use ddp_bind + ddp_reduce_all for this size)");
    if (total == 0 || S == 0) return DDP_OK;

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(ctx, DDP_ERR_INVALID_ARG, "device index out of range");
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaDeviceGetAttribute");

    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {   // once per device, with that device current
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaGetSymbolAddress(static scratch)");
        g_scratch_addr[dev] = p;
    }

    unsigned char* h = g_host_table;
    std::memset(h, 0, bytes);   // status word and padding start at zero
    auto* off = reinterpret_cast<int64_t*>(h + b_status);
    auto* src = reinterpret_cast<const void**>(h + b_status + b_off);
    auto* dst = reinterpret_cast<float**>(h + b_status + b_off + b_src);
    auto* vec = reinterpret_cast<int32_t*>(h + b_status + b_off + b_src + b_dst);
    size_t s = 0;
    for (int32_t b = 0; b < L.B; ++b) {
        for (int32_t v : (*L.members)[b]) {
            const int64_t n = L.numel[v];
            if (n == 0) continue;
            const int64_t a0 = L.bucket_off[b] + L.loc[v].offset;
            bool ok16 = true;
            for (int r = 0; r < W; ++r) {
                const void* g = grads[static_cast<int64_t>(r) * L.P + v];
                if (!g) return fail(ctx, DDP_ERR_INVALID_ARG, "NULL gradient for replica " + std::to_string(r));
                src[s * W + r] = g;
                ok16 = ok16 && ((reinterpret_cast<uintptr_t>(g) - static_cast<uintptr_t>(a0 * L.elem)) & 15u) == 0;
            }
            for (int o = 0; o < n_out; ++o) {
                float* d = grad_out[static_cast<int64_t>(o) * L.P + v];
                if (!d) return fail(ctx, DDP_ERR_INVALID_ARG, "NULL output for copy " + std::to_string(o));
                dst[s * n_out + o] = d;
                ok16 = ok16 && ((reinterpret_cast<uintptr_t>(d) - static_cast<uintptr_t>(a0 * 4)) & 15u) == 0;
            }
            off[s] = a0;
            vec[s] = ok16 ? 1 : 0;
            ++s;
        }
    }
    off[S] = total;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned char* base = static_cast<unsigned char*>(g_scratch_addr[dev]);
    e = cudaMemcpyAsync(base, h, bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "cudaMemcpyAsync(static scratch)");

    ddpk::SegTable t;
    t.add = 0;   // W source streams per segment: the call's own gradients
    t.status = reinterpret_cast<int*>(base);
    t.seg_off = reinterpret_cast<const long long*>(base + b_status);
    t.seg_src = reinterpret_cast<const void* const*>(base + b_status + b_off);
    t.seg_dst = reinterpret_cast<float* const*>(base + b_status + b_off + b_src);
    t.seg_vec = reinterpret_cast<const int*>(base + b_status + b_off + b_src + b_dst);
    ddpk::LaunchCfg cfg{};
    cfg.sms = sms;
    cfg.block = 256;
    cfg.ctas_per_sm = 1;
    cfg.pdl = true;
    cfg.kernel = ddpk::KERNEL_TMA;
    cfg.stages = 3;
    cfg.stage_bytes = 32 * 1024;
    cfg.tma_ctas_per_sm = 1;
    const ddpk::InType in = L.bf16 ? ddpk::IN_BF16 : ddpk::IN_F32;
    e = ddpk::launch_reduce_tma(t, in, W, n_out, bucket_arena, 0, total, 0, static_cast<int>(S),
                                1.0f / static_cast<float>(W), cfg, st, nullptr);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "bucket reduce launch (no-alloc)");
    return DDP_OK;
}
