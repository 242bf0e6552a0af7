// Device-side helpers shared by the bucket-reduce kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "ddp_kernels.h"

namespace ddpk {
namespace dev {

// ------------------------------------------------------------------ PTX helpers

// Programmatic dependent launch: let the next launch in the stream start its
// CTAs now; and wait until every earlier grid has finished and its memory is
// visible.  Both are no-ops without the launch attribute.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// 128-bit loads through the non-coherent path, no L1 allocation (the data
// is read exactly once).
__device__ __forceinline__ float4 ld_stream(const float4* p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Evict-first 128-bit store: outputs are not re-read by this pass.
__device__ __forceinline__ void st_stream(float* p, float4 v) {
    __stcs(reinterpret_cast<float4*>(p), v);
}

// ------------------------------------------------------------------ debug checks

// Debug builds (-DDDP_DEBUG) check every range a kernel walks and every bulk
// copy it issues.  The first failed check records its code in word 1 of the
// binding's 16-byte status block and the offending element index in words
// 2..3, and the access is skipped (no trap: the context stays usable).
// Release builds compile the checks away.
enum DebugCode {
    kDbgSegRange = 101,    // a segment range outside its segment or the launch
    kDbgChunkRange = 102,  // a staged chunk outside its segment, slice or stage
    kDbgCopyAlign = 103,   // a bulk copy not 16-byte aligned or sized
    kDbgPairRange = 104,   // an accumulate range outside its pair
};

#ifdef DDP_DEBUG
constexpr bool kDebug = true;
static __device__ __noinline__ void debug_record(int* status, int code, long long index) {
    if (status && atomicCAS(status + 1, 0, code) == 0)
        atomicExch(reinterpret_cast<unsigned long long*>(status + 2), static_cast<unsigned long long>(index));
}
#else
constexpr bool kDebug = false;
__device__ __forceinline__ void debug_record(int*, int, long long) {}
#endif

// `ok`, recording a failure in debug builds; always true in release builds.
__device__ __forceinline__ bool debug_ok(int* status, bool ok, int code, long long index) {
    if constexpr (kDebug) {
        if (!ok) debug_record(status, code, index);
        return ok;
    } else {
        return true;
    }
}

// ------------------------------------------------------------------ element types

// bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits.
__device__ __forceinline__ float widen1(float x) { return x; }
__device__ __forceinline__ float widen1(uint16_t x) {
    return __uint_as_float(static_cast<uint32_t>(x) << 16);
}

template <typename Tin> struct Vec;

template <> struct Vec<float> {
    static constexpr int N = 4;          // elements per 16-byte access
    using Raw = float4;
    __device__ __forceinline__ static void unpack(const Raw& r, float (&f)[N]) {
        f[0] = r.x; f[1] = r.y; f[2] = r.z; f[3] = r.w;
    }
};

template <> struct Vec<uint16_t> {
    static constexpr int N = 8;
    using Raw = uint4;
    __device__ __forceinline__ static void unpack(const Raw& r, float (&f)[N]) {
        f[0] = __uint_as_float(r.x << 16); f[1] = __uint_as_float(r.x & 0xffff0000u);
        f[2] = __uint_as_float(r.y << 16); f[3] = __uint_as_float(r.y & 0xffff0000u);
        f[4] = __uint_as_float(r.z << 16); f[5] = __uint_as_float(r.z & 0xffff0000u);
        f[6] = __uint_as_float(r.w << 16); f[7] = __uint_as_float(r.w & 0xffff0000u);
    }
};

// ------------------------------------------------------------------ segment search

// Largest s in [s0, s1) with off[s] <= x, given off[s0] <= x < off[s1].
// 32-ary search: each round every lane tests one of 32 evenly spaced
// candidates and a ballot picks the last one not above x.  Call with the
// whole warp converged.
__device__ __forceinline__ int find_segment(const long long* __restrict__ off, int s0, int s1,
                                            long long x) {
    const int lane = threadIdx.x & 31;
    int lo = s0;
    int n = s1 - s0;
    while (n > 32) {
        const int stride = (n + 31) >> 5;
        const int idx = lo + lane * stride;
        const bool le = idx < s1 && __ldg(off + idx) <= x;
        const unsigned m = __ballot_sync(0xffffffffu, le);
        lo += (31 - __clz(m)) * stride;
        n = min(stride, s1 - lo);
    }
    const int idx = lo + lane;
    const bool le = lane < n && __ldg(off + idx) <= x;
    const unsigned m = __ballot_sync(0xffffffffu, le);
    return lo + 31 - __clz(m);
}

// ------------------------------------------------------------------ launch parameters

struct ReduceParams {
    const long long* seg_off;
    const void* const* seg_src;
    float* const* seg_dst;
    const int* seg_vec;
    float* arena;
    int* status;        // device status word (0 = ok)
    long long base;     // start of slice 0 (lo rounded down to the vector width)
    long long lo, hi;   // arena range of this launch
    long long piece;    // elements per CTA, multiple of the vector width
    int s0, s1;         // segment range of this launch
    int W;
    int n_out;
    float inv_w;
    int stages;         // pipelined kernel: ring depth
    int tile;           // pipelined kernel: elements per replica per stage
    int chain;          // 1: follows a launch of the same iteration (see pdl_enter)
    int first_wave;     // pipelined kernel: CTAs resident at once (the first wave of the grid)
    int trace_slot;     // trace builds (-DDDP_TRACE): the launch's row of the launch trace
};

// Entry/exit ordering with the previous launch in the stream.
//   chain == 0: wait for every earlier grid, then let the successor start;
//   chain == 1: the previous launch is this iteration's own bucket kernel on
//               the same stream (disjoint data) and the caller guarantees that
//               nothing else runs on the stream during the iteration: start at
//               once, and wait for the predecessor only before exiting, so
//               this grid still completes after everything before it.
// A grid completes when its last CTA exits, so one waiting CTA (block 0, which
// always has work) is enough for that ordering; the others can retire as soon
// as their slice is done and hand their SM slots to the launches behind them.
// That pays when slices are short (per-gradient and small buckets); with long
// slices it lets the fastest SMs run ahead into later launches and leaves a
// tail of late-started slices at the end of the iteration, so there every CTA
// waits (hold_all).
__device__ __forceinline__ void pdl_enter(int chain) {
    if (!chain) pdl_wait();
    pdl_trigger();
}

__device__ __forceinline__ void pdl_exit(int chain, bool hold_all) {
    if (chain && (hold_all || blockIdx.x == 0)) pdl_wait();
}

// Bucket-reduce slices (elements per CTA) from which every CTA of a chained
// launch waits for its predecessor.  GB300, GPT-2-medium bf16 W=8: early
// release gains 3.2 % at cap 0 and 2.5 % at cap 1, holding every CTA is 5 %
// faster at cap 100 (slices of ~4e5 elements); BERT-large W=4 ties.  The
// accumulate kernels always release early (CTA 0 alone waits): their chained
// launches are equal blocks of (acc, g) pairs, and ResNet-50 W=16 micro-steps
// measured 1.3 % faster that way.
constexpr long long kHoldAllPiece = 1LL << 17;

// ------------------------------------------------------------------ replica masks

// Local-use masks of a launch with unused parameters: bit r of bits[s - s0]
// is set when replica r has a gradient for segment s (one parameter per
// segment in this mode).  A clear bit makes the replica contribute +0.0 (its
// zero-filled bucket slice) without loading anything; a segment with no bit
// set is unused on every replica and its copy-back is not written.
__device__ __forceinline__ unsigned long long seg_mask(const NoMask&, int) { return ~0ull; }
__device__ __forceinline__ unsigned long long seg_mask(const SegMask& m, int rel) { return m.bits[rel]; }

__device__ __forceinline__ bool has_replica(unsigned long long mk, int r) { return (mk >> r) & 1ull; }

// Any replica uses the segment (W <= 64 in masked launches; ~0 otherwise).
__device__ __forceinline__ bool any_replica(unsigned long long mk, int W) {
    return W >= 64 ? mk != 0ull : (mk & ((1ull << W) - 1ull)) != 0ull;
}

// fp32 -> bf16 with round to nearest even, widened back to fp32: the
// hardware conversion (cvt.rn.bf16.f32; values past the largest bf16 round to
// infinity, subnormals are kept, a NaN becomes a quiet NaN), its 16 bits
// placed as the high half of the fp32 pattern.  GB300, the compression hook
// inside the fused pass on BERT-large W=4: 7,123 GB/s against 7,009 for the
// same rounding done with integer operations on the bit pattern.
__device__ __forceinline__ float round_bf16(float x) {
    uint32_t h;
    asm("{\n\t.reg .b16 t;\n\tcvt.rn.bf16.f32 t, %1;\n\tmov.b32 %0, {0, t};\n\t}" : "=r"(h) : "f"(x));
    return __uint_as_float(h);
}

// Replica r's input at segment element j: its gradient, or with ADD (fused
// last micro-step) fl32(accumulated + last-step gradient), whose pointers
// are src[r] and src[W + r]; with CMP (the bf16-compression hook fused into
// the pass) the fp32 value rounded to bf16 first.
template <bool ADD, bool CMP = false, typename Tin>
__device__ __forceinline__ float replica_in(const Tin* const* src, int W, int r, long long j) {
    if constexpr (ADD) return __fadd_rn(widen1(src[r][j]), widen1(src[W + r][j]));
    else if constexpr (CMP) return round_bf16(widen1(src[r][j]));
    else return widen1(src[r][j]);
}

// Rank-order fp32 mean of one element, scalar path (heads, tails, segments
// whose pointers do not share the arena's 16-byte phase).
template <typename Tin, bool ADD = false, bool CMP = false>
__device__ __forceinline__ void reduce_scalar(const ReduceParams& p, const Tin* const* src,
                                              float* const* dst, long long a0, long long x,
                                              long long e, int W, int tid, int nthr,
                                              unsigned long long mk = ~0ull) {
    const bool write_dst = any_replica(mk, W);
    for (long long a = x + tid; a < e; a += nthr) {
        const long long j = a - a0;
        float acc = has_replica(mk, 0) ? replica_in<ADD, CMP>(src, W, 0, j) : 0.0f;
        for (int r = 1; r < W; ++r)
            acc = __fadd_rn(acc, has_replica(mk, r) ? replica_in<ADD, CMP>(src, W, r, j) : 0.0f);
        const float m = __fmul_rn(acc, p.inv_w);
        p.arena[a] = m;
        if (write_dst)
            for (int o = 0; o < p.n_out; ++o) dst[o][j] = m;
    }
}

template <int N>
__device__ __forceinline__ void store_vec(const ReduceParams& p, float* const* dst, long long a,
                                          long long j, const float (&m)[N], bool write_dst = true) {
#pragma unroll
    for (int q = 0; q < N; q += 4)
        st_stream(p.arena + a + q, make_float4(m[q], m[q + 1], m[q + 2], m[q + 3]));
    if (!write_dst) return;
    for (int o = 0; o < p.n_out; ++o) {
        float* d = dst[o] + j;
#pragma unroll
        for (int q = 0; q < N; q += 4)
            st_stream(d + q, make_float4(m[q], m[q + 1], m[q + 2], m[q + 3]));
    }
}

// ------------------------------------------------------------------ accumulate parameters

// The (acc, g) pairs of one accumulate launch travel in the kernel's
// parameter block (40 B each; the block stays under 32 KiB).
constexpr int kMaxAccPairs = 800;

struct AccPairDev {
    const float* g;
    float* acc;
    long long off;   // start in the launch's flat space (multiple of 4)
    long long len;
    int assign;      // 1: acc = g (the gradient field was empty); 0: acc = fl32(acc + g)
    int pad;
};

struct AccParams {
    long long total;   // flat extent (last pair's padded end)
    long long piece;   // elements per CTA, multiple of 4
    int npairs;
    int chain;         // 1: follows this call's previous accumulate launch
    int stages;        // bulk-copy variant: ring depth
    int tile;          // bulk-copy variant: elements per operand per stage (multiple of 4)
    int* status;       // device status block (bulk-copy waits, debug checks)
    AccPairDev pair[kMaxAccPairs];
};

// Largest i with pair[i].off <= x (pair[0].off = 0 <= x); 32-ary warp-ballot
// search over the pairs' flat offsets.  Call with the whole warp converged.
__device__ __forceinline__ int find_pair(const AccParams& p, long long x) {
    const int lane = threadIdx.x & 31;
    int lo = 0;
    int n = p.npairs;
    while (n > 32) {
        const int stride = (n + 31) >> 5;
        const int idx = lo + lane * stride;
        const bool le = idx < p.npairs && p.pair[idx].off <= x;
        const unsigned m = __ballot_sync(0xffffffffu, le);
        lo += (31 - __clz(m)) * stride;
        n = min(stride, p.npairs - lo);
    }
    const int idx = lo + lane;
    const bool le = lane < n && p.pair[idx].off <= x;
    const unsigned m = __ballot_sync(0xffffffffu, le);
    return lo + 31 - __clz(m);
}

}  // namespace dev
}  // namespace ddpk
