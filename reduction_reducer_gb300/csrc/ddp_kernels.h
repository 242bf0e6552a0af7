// Internal interface between the host core (ddp_host.cpp) and the device
// kernels (ddp_kernels.cu, ddp_kernels_tma.cu).  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ddpk {

// Device copy of the bind-time segment table.  A segment is a run of
// variables of one bucket that is contiguous in the arena, in every replica's
// gradients and in every copy-back output, so one pointer per stream covers
// it.  seg_off[s] is the arena element index where segment s starts
// (strictly increasing; seg_off[S] = arena length); seg_src[s*W + r] points
// at replica r's first element of the segment; seg_dst[s*n_out + o] at output
// copy o's first element; seg_vec[s] != 0 when every pointer has the same
// 16-byte phase as the arena, so 128-bit accesses (and bulk copies) line up.
// status is a device word the kernels set when a bounded wait gives up.
// add != 0 (fused last micro-step of a no_sync block, fp32 only): each
// segment has 2W source pointers, seg_src[s*2W + r] replica r's accumulated
// gradient and seg_src[s*2W + W + r] its last-step gradient; replica r then
// contributes fl32(acc_r + g_r).
struct SegTable {
    const long long* seg_off;
    const void* const* seg_src;
    float* const* seg_dst;
    const int* seg_vec;
    int* status;
    int add;
};

// KERNEL_AUTO is resolved per context by the host core (median bucket size).
enum KernelKind { KERNEL_LDG = 0, KERNEL_TMA = 1, KERNEL_AUTO = 2 };

struct LaunchCfg {
    int sms;           // multiprocessors on the device
    int block;         // threads per CTA (register-streaming kernel)
    int ctas_per_sm;   // CTAs per SM of the register-streaming bucket kernel (resident waves x occupancy)
    bool pdl;          // programmatic dependent launch
    int kernel;        // KernelKind
    int stages;        // bulk-copy kernel: ring depth
    int stage_bytes;   // bulk-copy kernel: bytes of all replicas' tiles per stage
    int tma_ctas_per_sm;        // bulk-copy kernels: CTAs per SM; 0 = tma_waves resident waves
    int tma_waves;              // resident waves of a bulk-copy launch when tma_ctas_per_sm is 0 (0 = 2)
    int chain;                  // per launch: see pdl_enter in ddp_device.cuh
    int last;                   // per launch: the iteration's final launch (nothing follows to overlap its tail)
    int compress;               // bucket reduce: each replica value rounded to bf16 first (fp32 inputs,
                                // no mask, no fused last step): the bf16-compression hook in the pass
    int* status;                // device status word of the binding (bulk-copy kernels)
};

enum InType { IN_F32 = 0, IN_BF16 = 1 };

// Local-use masks of one launch with unused parameters (one parameter per
// segment): bit r of bits[s - s0] set = replica r has a gradient for segment
// s.  Passed by value in the kernel's parameter block.
constexpr int kMaxMaskSegs = 3840;   // 8 B each: the block stays < 32 KiB

struct SegMask {
    int n;
    unsigned long long bits[kMaxMaskSegs];
};

struct NoMask {
    int unused;
};

// Fused bucket pass over arena range [lo, hi) = segments [s0, s1):
// gather W replicas, fp32 sum in rank order, x inv_w, write arena and copies.
// mask: nullptr for launches without unused parameters; otherwise the masks of
// segments [s0, s1) (s1 - s0 <= kMaxMaskSegs).
cudaError_t launch_reduce(const SegTable& t, InType in, int W, int n_out, float* arena,
                          long long lo, long long hi, int s0, int s1, float inv_w,
                          const LaunchCfg& cfg, cudaStream_t stream, long long* launches,
                          const SegMask* mask = nullptr);

// Largest number of resident CTAs per SM of the register-streaming kernel
// (add: the fused last-step variant).
int reduce_max_ctas_per_sm(InType in, int W, int block, bool add = false);

// One accumulation pair: acc = g (assign) or acc = fl32(acc + g) over len elements.
struct AccPair {
    const float* g;
    float* acc;
    long long len;
    int assign;
};

// Every pair; the bulk-copy variant when cfg.kernel is KERNEL_TMA.
cudaError_t launch_accumulate(const AccPair* pairs, int n, const LaunchCfg& cfg,
                              cudaStream_t stream, long long* launches);

int accumulate_max_ctas_per_sm(int block);

// ------------------------------------------------------------------ hook path

// Gather (mode 0): for segments [s0, s1) copy every replica's gradients into
// its bucket buffer at the arena offsets (rb[r] + a, grad element size).
// Copy-back (mode 1): copy the arena into every output copy's views.
constexpr int kMaxHookReplicas = 64;
cudaError_t launch_seg_copy(const SegTable& t, int mode, int elem, int W, int n_out, const float* arena,
                            void* const* rb, long long lo, long long hi, int s0, int s1,
                            const LaunchCfg& cfg, cudaStream_t stream, long long* launches);

// out[i] = fp32 rank-order mean of widen(in_r[i]) x inv_w (compress = 1: each
// fp32 value first rounded to bf16, round to nearest even).
cudaError_t launch_flat_mean(InType in, int W, const void* const* src, float* out, long long n, float inv_w,
                             int compress, int sms, cudaStream_t stream);

// Bulk-copy (TMA) pipelined variant of launch_accumulate, in ddp_kernels_tma.cu.
cudaError_t launch_accumulate_tma(const AccPair* pairs, int n, const LaunchCfg& cfg,
                                  cudaStream_t stream, long long* launches);

// One CTA that waits on an mbarrier nothing completes, for limit_cycles; the
// bounded wait writes its timeout code into *status (ddp_kernels_tma.cu).
cudaError_t launch_wait_selftest(long long limit_cycles, int* status, cudaStream_t stream);

// The launch trace of a -DDDP_TRACE build (see ddp_read_launch_trace);
// *seq = -1 in other builds.
cudaError_t read_launch_trace(unsigned long long* out, int* grid, long long* seq);

// Bulk-copy (TMA) pipelined variant of launch_reduce, in ddp_kernels_tma.cu.
cudaError_t launch_reduce_tma(const SegTable& t, InType in, int W, int n_out, float* arena,
                              long long lo, long long hi, int s0, int s1, float inv_w,
                              const LaunchCfg& cfg, cudaStream_t stream, long long* launches,
                              const SegMask* mask = nullptr);

}  // namespace ddpk
