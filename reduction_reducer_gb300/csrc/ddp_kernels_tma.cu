// Bulk-copy (TMA) pipelined variant of the fused bucket pass, sm_103a.
//
// Same arithmetic and outputs as bucket_reduce_kernel in ddp_kernels.cu
// (gather of the W replicas' per-parameter gradients, fp32 rank-order sum,
// x fl32(1/W), bucket write, copy-back), with the loads moved off the
// register file:
//
//   * one producer warp per CTA walks the CTA's slice of the launch and,
//     for every aligned chunk of a segment, issues W one-dimensional bulk
//     copies (cp.async.bulk, global -> shared) into one stage of a ring in
//     shared memory, one lane per copy; an mbarrier per stage counts the
//     landed bytes;
//   * eight consumer warps wait for a stage, sum the W tiles from shared
//     memory in rank order, scale, and stream the means to the arena and
//     the copy-back outputs with 128-bit evict-first stores, then release
//     the stage through a second mbarrier;
//   * with the default ring of 3 stages x 32 KiB a CTA keeps 96 KiB of loads
//     in flight independently of register pressure; two such CTAs fit in an
//     SM, so the next launch's CTAs can start beside a draining one.
//
// Ragged heads/tails and segments whose pointers do not share the arena's
// 16-byte phase bypass the ring (consumers load them directly).  Every
// mbarrier wait is bounded: after ~2 s it records a code in the device
// status word and carries on, so a fault in the pipeline can never hang the
// GPU; lane 0 of the producer warp waits (bounded) for all of the CTA's
// copies to land before the CTA exits.

#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "ddp_device.cuh"
#include "ddp_kernels.h"
#include "ddp_reducer.h"

namespace ddpk {

namespace {

using namespace dev;

constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (1 + kConsumerWarps);
constexpr long long kWaitCycles = 4000000000LL;   // ~2 s at 2 GHz
constexpr int kMaxDynSmem = 232448;                // 227 KiB opt-in per CTA
constexpr int kHeaderBytes = 128;                  // mbarriers, ring starts after
constexpr long long kMinCopyBytes = 4096;          // smallest per-stream copy a stage is sized for
#ifndef DDP_PREFETCH_STAGES
#define DDP_PREFETCH_STAGES 2
#endif
constexpr long long kPrefetchStages = DDP_PREFETCH_STAGES;   // stages prefetched before a launch's wait
#ifndef DDP_PREFETCH_WAVES
#define DDP_PREFETCH_WAVES 2
#endif
constexpr int kPrefetchWaves = DDP_PREFETCH_WAVES;            // waves of CTAs that prefetch (0: every CTA)
constexpr long long kLastMinStages = 8;   // stages per CTA that size an iteration's final launch
constexpr long long kAccLastMinStages = 4;   // ... and the last accumulate launch of a call
constexpr long long kWholeMinStages = 10;   // ... and the single launch of ddp_reduce_all
constexpr long long kWholeMaxWaves = 64;    // its most resident waves

// Launch trace (builds with -DDDP_TRACE only; ddp_read_launch_trace): per
// launch of the bucket pass, per CTA, four %globaltimer stamps -- entry, past
// the wait for the preceding grid (chained launches: past the trigger), the
// first stage the consumers take, and the last -- so that the boundary between
// two launches can be taken apart: the predecessor's tail, the release of the
// wait, the first data.  Release builds record nothing.
#ifdef DDP_TRACE
constexpr bool kTrace = true;
__device__ unsigned long long g_launch_trace[DDP_TRACE_LAUNCHES][DDP_TRACE_CTAS][4];
int g_trace_grid[DDP_TRACE_LAUNCHES];
long long g_trace_seq = 0;
std::mutex g_trace_mutex;
#else
constexpr bool kTrace = false;
#endif

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void trace_stamp(const ReduceParams& p, int which, unsigned long long t) {
#ifdef DDP_TRACE
    if (blockIdx.x < DDP_TRACE_CTAS) g_launch_trace[p.trace_slot][blockIdx.x][which] = t;
#else
    (void)p; (void)which; (void)t;
#endif
}

// status codes written by bounded waits
constexpr int kStatusEmptyTimeout = 1;
constexpr int kStatusDrainTimeout = 2;
constexpr int kStatusFullTimeout = 3;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of `bar` with the given parity to complete; give up
// after kWaitCycles, record `code` and mark the thread failed, after which
// it never waits again (so a broken pipeline costs one time limit per
// thread, not one per chunk).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* status, int code, bool& failed,
                                          long long limit = kWaitCycles) {
    if (mbar_try_wait(bar, parity)) return true;
    if (failed) return false;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) {
            atomicExch(status, code);
            failed = true;
            return false;
        }
    }
    return true;
}

// Bulk prefetch of [src, src + bytes) into L2 (no destination, no barrier):
// a hint that moves no data the program can observe.  src 16-byte aligned,
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// One-dimensional bulk copy global -> shared, completion counted in bytes
// on the mbarrier.  src and dst 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Walk the CTA's slice [x, y) starting in segment s.  Aligned runs of
// vector-capable segments are cut into chunks of at most p.tile elements
// and handed to `body`; everything else goes to `scalar`.  Producer and
// consumers both walk, so they see the same chunk sequence.
template <int N, typename Body, typename Scalar>
__device__ __forceinline__ void walk(const ReduceParams& p, int s, long long x, long long y, Body&& body,
                                     Scalar&& scalar) {
    while (x < y) {
        const long long a0 = __ldg(p.seg_off + s);
        const long long a1 = __ldg(p.seg_off + s + 1);
        const long long e = a1 < y ? a1 : y;
        const long long xb = (x + N - 1) / N * N;
        const long long xe = e / N * N;
        if (!debug_ok(p.status, s < p.s1 && a0 <= x && x < e && e <= a1 && p.lo <= x && e <= p.hi, kDbgSegRange, x))
            return;
        if (__ldg(p.seg_vec + s) && xb < xe) {
            if (x < xb) scalar(s, a0, x, xb);
            for (long long c = xb; c < xe; c += p.tile) {
                const long long L = xe - c < p.tile ? xe - c : p.tile;
                if (!debug_ok(p.status, x <= c && 0 < L && L <= p.tile && c + L <= e && L % N == 0, kDbgChunkRange, c))
                    return;
                body(s, a0, c, L);
            }
            if (xe < e) scalar(s, a0, xe, e);
        } else {
            scalar(s, a0, x, e);
        }
        x = e;
        ++s;
    }
}

// ADD: fused last micro-step of a no_sync block -- a stage holds 2W tiles
// (the W accumulated fields, then the W last-step gradients) and replica r
// contributes fl32(acc_r + g_r).  CMP: the built-in bf16-compression hook
// fused into the pass -- replica r contributes its value rounded to bf16.
template <typename Tin, int WC, typename M, bool ADD, bool CMP = false>
__global__ void __launch_bounds__(kThreads, 1)
bucket_reduce_tma_kernel(const __grid_constant__ ReduceParams p, const __grid_constant__ M mask) {
    extern __shared__ __align__(128) unsigned char smem[];
    using V = Vec<Tin>;
    constexpr int N = V::N;
    const int W = WC > 0 ? WC : p.W;
    const int NS = ADD ? 2 * W : W;   // source streams per segment
    const int S = p.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + S;
    Tin* ring = reinterpret_cast<Tin*>(smem + kHeaderBytes);
    const long long stage_elems = static_cast<long long>(NS) * p.tile;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if constexpr (kTrace) {   // entry; the consumers' stamps start empty (0) for this launch
        if (threadIdx.x == 0) {
            trace_stamp(p, 0, global_ns());
            trace_stamp(p, 2, 0);
            trace_stamp(p, 3, 0);
        }
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(empty + i), kConsumerWarps);
        }
        fence_barrier_init();
    }
    // A chained launch (see pdl_enter) lets its successor start at once.
    if (p.chain) pdl_trigger();

    // The CTA's slice and its first segment come from the library's own
    // segment table, final before the launch: found before the wait for the
    // preceding grid, so a launch that must wait spends none of the time
    // after it on the search.
    long long x = p.base + static_cast<long long>(blockIdx.x) * p.piece;
    long long y = x + p.piece;
    x = x < p.lo ? p.lo : x;
    y = y > p.hi ? p.hi : y;
    const bool idle = x >= y;   // the same for every thread of the CTA
    const int s = idle ? p.s0 : find_segment(p.seg_off, p.s0, p.s1, x);
    // A launch that waits for the preceding grid asks L2 for the inputs of its
    // first stages meanwhile.  Its CTAs become resident only as the preceding
    // launch's CTAs retire (two resident waves fill the SMs until then), so
    // the lines arrive during that launch's tail and the first bulk copies
    // after the wait hit L2.  A prefetch moves nothing the program observes:
    // inputs a preceding grid is still writing are read again, coherently, by
    // the copies after the wait.  The CTAs of the first two waves prefetch:
    // the first wave waits for the preceding grid, the second starts as the
    // first retires and ramps faster with two more stages in flight; later
    // waves gain nothing from it.  GB300, against every CTA prefetching:
    // one reduce_all launch over ResNet-50 W=8 +1.7 %, BERT-large ties in
    // every driving mode; the first wave alone lost 0.7 % per event.
    if (!idle && !p.chain && kPrefetchStages > 0 && warp == 0 &&
        (kPrefetchWaves == 0 || static_cast<int>(blockIdx.x) < kPrefetchWaves * p.first_wave)) {
        long long k = 0;
        walk<N>(
            p, s, x, y,
            [&](int sg, long long a0, long long c, long long L) {
                if (k++ >= kPrefetchStages) return;
                const unsigned long long mk = seg_mask(mask, sg - p.s0);
                const Tin* const* src = reinterpret_cast<const Tin* const*>(p.seg_src) + static_cast<long long>(sg) * NS;
                for (int q = lane; q < NS; q += 32)
                    if (has_replica(mk, q % W))
                        bulk_prefetch_l2(src[q] + (c - a0), static_cast<uint32_t>(L * sizeof(Tin)));
            },
            [](int, long long, long long, long long) {});
    }
    __syncthreads();
    if (!p.chain) pdl_enter(0);   // wait for every earlier grid, then let the successor start
    if constexpr (kTrace) {
        if (threadIdx.x == 0) trace_stamp(p, 1, global_ns());
    }
    if (idle) {   // whole CTA, before any copy is issued
        if (threadIdx.x == 0) pdl_exit(p.chain, p.piece >= kHoldAllPiece);
        return;
    }

    if (warp == 0) {
        // ---------------------------------------------------------- producer warp
        // Every lane walks the same chunk sequence and waits for the stage
        // itself; lane 0 posts the stage's byte count, then lane q issues the
        // copies of streams q, q + 32, ...: a stage's copies go out in
        // parallel instead of one after another from a single thread.
        long long k = 0;
        bool failed = false;
        walk<N>(
            p, s, x, y,
            [&](int sg, long long a0, long long c, long long L) {
                const int st = static_cast<int>(k % S);
                const uint32_t use = static_cast<uint32_t>(k / S);
                if (use > 0) mbar_wait(smem_u32(empty + st), (use - 1) & 1u, p.status, kStatusEmptyTimeout, failed);
                const uint32_t bytes = static_cast<uint32_t>(L * sizeof(Tin));
                const uint32_t fb = smem_u32(full + st);
                // replicas without a gradient for this segment copy nothing
                const unsigned long long mk = seg_mask(mask, sg - p.s0);
                const Tin* const* src = reinterpret_cast<const Tin* const*>(p.seg_src) + static_cast<long long>(sg) * NS;
                Tin* dst = ring + st * stage_elems;
                // debug builds: a stage whose copies would break the bulk-copy
                // alignment rules is posted empty and not copied
                bool issue = true;
                if constexpr (kDebug) {
                    bool ok = (bytes & 15u) == 0;
                    for (int q = lane; q < NS; q += 32)
                        ok = ok && ((reinterpret_cast<uintptr_t>(src[q] + (c - a0)) |
                                     smem_u32(dst + static_cast<long long>(q) * p.tile)) & 15u) == 0;
                    issue = __all_sync(0xffffffffu, ok);
                    if (!issue && lane == 0) debug_record(p.status, kDbgCopyAlign, c);
                }
                if (lane == 0) {
                    uint32_t present = 0;
                    for (int q = 0; q < NS; ++q) present += has_replica(mk, q % W) ? 1u : 0u;
                    mbar_expect_tx(fb, issue ? bytes * present : 0u);
                }
                __syncwarp();
                if (issue)
                    for (int q = lane; q < NS; q += 32)
                        if (has_replica(mk, q % W))
                            bulk_g2s(smem_u32(dst + static_cast<long long>(q) * p.tile), src[q] + (c - a0), bytes, fb);
                ++k;
            },
            [](int, long long, long long, long long) {});
        if (lane != 0) return;
        // every issued copy must land before the CTA may exit
        for (long long j = k > S ? k - S : 0; j < k; ++j)
            mbar_wait(smem_u32(full + j % S), static_cast<uint32_t>(j / S) & 1u, p.status, kStatusDrainTimeout, failed);
        pdl_exit(p.chain, p.piece >= kHoldAllPiece);
        return;
    }

    // -------------------------------------------------------------- consumers
    const int tc = threadIdx.x - 32;
    constexpr int nct = kConsumerWarps * 32;
    long long k = 0;
    bool failed = false;
    walk<N>(
        p, s, x, y,
        [&](int sg, long long a0, long long c, long long L) {
            const int st = static_cast<int>(k % S);
            const uint32_t use = static_cast<uint32_t>(k / S);
            mbar_wait(smem_u32(full + st), use & 1u, p.status, kStatusFullTimeout, failed);
            if constexpr (kTrace) {
                if (k == 0 && tc == 0) trace_stamp(p, 2, global_ns());
            }
            const Tin* base = ring + st * stage_elems;
            float* const* dst = p.seg_dst + static_cast<long long>(sg) * p.n_out;
            const unsigned long long mk = seg_mask(mask, sg - p.s0);
            const bool write_dst = any_replica(mk, W);
            const int nv = static_cast<int>(L / N);
            using Raw = typename V::Raw;
            // replica r's input vector v of this stage (ADD: accumulated + last step)
            auto input = [&](int r, int v, float (&f)[N]) {
                const long long at = static_cast<long long>(r) * p.tile + v * N;
                V::unpack(has_replica(mk, r) ? *reinterpret_cast<const Raw*>(base + at) : Raw{}, f);
                if constexpr (ADD) {
                    float h[N];
                    V::unpack(has_replica(mk, r) ? *reinterpret_cast<const Raw*>(base + at + static_cast<long long>(W) * p.tile)
                                                 : Raw{},
                              h);
#pragma unroll
                    for (int q = 0; q < N; ++q) f[q] = __fadd_rn(f[q], h[q]);
                }
                if constexpr (CMP) {
#pragma unroll
                    for (int q = 0; q < N; ++q) f[q] = round_bf16(f[q]);
                }
            };
            for (int v = tc; v < nv; v += nct) {
                float acc[N], f[N];
                input(0, v, acc);
                if constexpr (WC > 0) {
#pragma unroll
                    for (int r = 1; r < WC; ++r) {
                        input(r, v, f);
#pragma unroll
                        for (int q = 0; q < N; ++q) acc[q] = __fadd_rn(acc[q], f[q]);
                    }
                } else {
                    for (int r = 1; r < W; ++r) {
                        input(r, v, f);
#pragma unroll
                        for (int q = 0; q < N; ++q) acc[q] = __fadd_rn(acc[q], f[q]);
                    }
                }
#pragma unroll
                for (int q = 0; q < N; ++q) acc[q] = __fmul_rn(acc[q], p.inv_w);
                store_vec<N>(p, dst, c + static_cast<long long>(v) * N, c - a0 + static_cast<long long>(v) * N, acc,
                             write_dst);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(empty + st));
            ++k;
        },
        [&](int sg, long long a0, long long lo, long long hi) {
            const Tin* const* src = reinterpret_cast<const Tin* const*>(p.seg_src) + static_cast<long long>(sg) * NS;
            float* const* dst = p.seg_dst + static_cast<long long>(sg) * p.n_out;
            reduce_scalar<Tin, ADD, CMP>(p, src, dst, a0, lo, hi, W, tc, nct, seg_mask(mask, sg - p.s0));
        });
    if constexpr (kTrace) {
        if (tc == 0) trace_stamp(p, 3, global_ns());
    }
}

// ------------------------------------------------------------------ accumulate

// Walk the CTA's slice [x, y) of an accumulate launch's flat space starting
// at pair i: aligned runs of 16-byte-aligned pairs in chunks of at most
// p.tile elements go to `body(i, c, L)`, the rest to `scalar(i, lo, hi)`.
// Padding between pairs (each pair starts at a multiple of 4) is skipped.
template <typename Body, typename Scalar>
__device__ __forceinline__ void walk_pairs(const AccParams& p, int i, long long x, long long y, Body&& body,
                                           Scalar&& scalar) {
    while (x < y && i < p.npairs) {
        const AccPairDev& q = p.pair[i];
        const long long end = q.off + q.len;
        const long long e = end < y ? end : y;
        if (x < e) {
            const bool vec = ((reinterpret_cast<uintptr_t>(q.g) | reinterpret_cast<uintptr_t>(q.acc)) & 15u) == 0;
            const long long xb = (x + 3) / 4 * 4;
            const long long xe = e / 4 * 4;
            if (!debug_ok(p.status, q.off <= x && e <= p.total, kDbgPairRange, x)) return;
            if (vec && xb < xe) {
                if (x < xb) scalar(i, x, xb);
                for (long long c = xb; c < xe; c += p.tile) {
                    const long long L = xe - c < p.tile ? xe - c : p.tile;
                    if (!debug_ok(p.status, x <= c && 0 < L && c + L <= e && L % 4 == 0, kDbgChunkRange, c)) return;
                    body(i, c, L);
                }
                if (xe < e) scalar(i, xe, e);
            } else {
                scalar(i, x, e);
            }
        }
        x = end > x ? end : x;
        ++i;
        if (i < p.npairs && p.pair[i].off > x) x = p.pair[i].off;
    }
}

// no_sync micro-step through the bulk-copy ring: per chunk, the producer
// copies the g tile (and, after the first step, the acc tile) into a stage;
// consumers add in fp32 (acc + g, or take g) and store acc with 128-bit
// evict-first stores.
__global__ void __launch_bounds__(kThreads, 1)
accumulate_tma_kernel(const __grid_constant__ AccParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int S = p.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + S;
    float* ring = reinterpret_cast<float*>(smem + kHeaderBytes);
    const long long stage_elems = 2LL * p.tile;   // [g tile | acc tile]
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(smem_u32(full + i), 1);
            mbar_init(smem_u32(empty + i), kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_enter(p.chain);

    long long x = static_cast<long long>(blockIdx.x) * p.piece;
    long long y = x + p.piece;
    y = y > p.total ? p.total : y;
    if (x >= y) {
        if (threadIdx.x == 0) pdl_exit(p.chain, false);
        return;
    }
    const int i0 = find_pair(p, x);

    if (warp == 0) {
        if (lane != 0) return;
        long long k = 0;
        bool failed = false;
        walk_pairs(
            p, i0, x, y,
            [&](int i, long long c, long long L) {
                const int st = static_cast<int>(k % S);
                const uint32_t use = static_cast<uint32_t>(k / S);
                if (use > 0) mbar_wait(smem_u32(empty + st), (use - 1) & 1u, p.status, kStatusEmptyTimeout, failed);
                const uint32_t bytes = static_cast<uint32_t>(L * sizeof(float));
                const uint32_t fb = smem_u32(full + st);
                const AccPairDev& q = p.pair[i];
                float* dst = ring + st * stage_elems;
                bool issue = true;
                if constexpr (kDebug) {
                    issue = ((bytes | reinterpret_cast<uintptr_t>(q.g + (c - q.off)) |
                              reinterpret_cast<uintptr_t>(q.acc + (c - q.off)) | smem_u32(dst) |
                              smem_u32(dst + p.tile)) & 15u) == 0;
                    if (!issue) debug_record(p.status, kDbgCopyAlign, c);
                }
                mbar_expect_tx(fb, !issue ? 0u : q.assign ? bytes : 2u * bytes);
                if (issue) {
                    bulk_g2s(smem_u32(dst), q.g + (c - q.off), bytes, fb);
                    if (!q.assign) bulk_g2s(smem_u32(dst + p.tile), q.acc + (c - q.off), bytes, fb);
                }
                ++k;
            },
            [](int, long long, long long) {});
        for (long long j = k > S ? k - S : 0; j < k; ++j)
            mbar_wait(smem_u32(full + j % S), static_cast<uint32_t>(j / S) & 1u, p.status, kStatusDrainTimeout, failed);
        pdl_exit(p.chain, false);
        return;
    }

    const int tc = threadIdx.x - 32;
    constexpr int nct = kConsumerWarps * 32;
    long long k = 0;
    bool failed = false;
    walk_pairs(
        p, i0, x, y,
        [&](int i, long long c, long long L) {
            const int st = static_cast<int>(k % S);
            const uint32_t use = static_cast<uint32_t>(k / S);
            mbar_wait(smem_u32(full + st), use & 1u, p.status, kStatusFullTimeout, failed);
            const float* gt = ring + st * stage_elems;
            const float* at = gt + p.tile;
            float* acc = p.pair[i].acc + (c - p.pair[i].off);
            const bool assign = p.pair[i].assign != 0;
            const int nv = static_cast<int>(L / 4);
            for (int v = tc; v < nv; v += nct) {
                const float4 g = *reinterpret_cast<const float4*>(gt + 4 * v);
                if (assign) {
                    st_stream(acc + 4 * v, g);
                } else {
                    const float4 a = *reinterpret_cast<const float4*>(at + 4 * v);
                    st_stream(acc + 4 * v, make_float4(__fadd_rn(a.x, g.x), __fadd_rn(a.y, g.y),
                                                       __fadd_rn(a.z, g.z), __fadd_rn(a.w, g.w)));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(empty + st));
            ++k;
        },
        [&](int i, long long lo, long long hi) {
            const AccPairDev& q = p.pair[i];
            for (long long a = lo + tc; a < hi; a += nct) {
                const long long j = a - q.off;
                q.acc[j] = q.assign ? q.g[j] : __fadd_rn(q.acc[j], q.g[j]);
            }
        });
}

// Bounded-wait self-test: one thread waits on an mbarrier that nothing
// arrives at, with the given cycle budget; the wait must give up, record
// its code in *status and return.
__global__ void wait_selftest_kernel(long long limit, int* status) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
    bool failed = false;
    mbar_wait(smem_u32(&bar), 0u, status, kStatusFullTimeout, failed, limit);
}

template <typename M>
using TmaKernel = void (*)(ReduceParams, M);

template <typename M>
TmaKernel<M> pick_tma(InType in, int W) {
    if (in == IN_F32) {
        switch (W) {
            case 2: return bucket_reduce_tma_kernel<float, 2, M, false>;
            case 4: return bucket_reduce_tma_kernel<float, 4, M, false>;
            case 8: return bucket_reduce_tma_kernel<float, 8, M, false>;
            case 16: return bucket_reduce_tma_kernel<float, 16, M, false>;
            default: return bucket_reduce_tma_kernel<float, 0, M, false>;
        }
    }
    switch (W) {
        case 2: return bucket_reduce_tma_kernel<uint16_t, 2, M, false>;
        case 4: return bucket_reduce_tma_kernel<uint16_t, 4, M, false>;
        case 8: return bucket_reduce_tma_kernel<uint16_t, 8, M, false>;
        case 16: return bucket_reduce_tma_kernel<uint16_t, 16, M, false>;
        default: return bucket_reduce_tma_kernel<uint16_t, 0, M, false>;
    }
}

// bf16-compression variant: fp32 gradients, every replica present.
TmaKernel<NoMask> pick_tma_cmp(int W) {
    switch (W) {
        case 2: return bucket_reduce_tma_kernel<float, 2, NoMask, false, true>;
        case 4: return bucket_reduce_tma_kernel<float, 4, NoMask, false, true>;
        case 8: return bucket_reduce_tma_kernel<float, 8, NoMask, false, true>;
        case 16: return bucket_reduce_tma_kernel<float, 16, NoMask, false, true>;
        default: return bucket_reduce_tma_kernel<float, 0, NoMask, false, true>;
    }
}

// Fused last-step variant: fp32 accumulators, every replica present.
TmaKernel<NoMask> pick_tma_add(int W) {
    switch (W) {
        case 2: return bucket_reduce_tma_kernel<float, 2, NoMask, true>;
        case 4: return bucket_reduce_tma_kernel<float, 4, NoMask, true>;
        case 8: return bucket_reduce_tma_kernel<float, 8, NoMask, true>;
        case 16: return bucket_reduce_tma_kernel<float, 16, NoMask, true>;
        default: return bucket_reduce_tma_kernel<float, 0, NoMask, true>;
    }
}

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// The dynamic shared-memory limit is raised once per kernel and device
// (the cache is shared by every context and host thread).
template <typename K>
cudaError_t ensure_smem_attr(K k) {
    constexpr int kSlots = 64;
    static K done_k[kSlots];
    static int done_dev[kSlots];
    static int n_done = 0;
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_done; ++i)
        if (done_k[i] == k && done_dev[i] == dev) return cudaSuccess;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    // Prefer the largest shared-memory carveout so that the next launch's
    // CTAs (programmatic dependent launch) fit beside this one's.
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess && n_done < kSlots) {
        done_k[n_done] = k;
        done_dev[n_done] = dev;
        ++n_done;
    }
    return e;
}

// CTAs of kernel k with `smem` bytes of dynamic shared memory that fit on
// one SM at once (cached per kernel, size and device; call after
// ensure_smem_attr).  At least 1.
template <typename K>
int resident_ctas(K k, long long smem) {
    constexpr int kSlots = 64;
    static K done_k[kSlots];
    static long long done_smem[kSlots];
    static int done_dev[kSlots];
    static int done_n[kSlots];
    static int n_done = 0;
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_done; ++i)
        if (done_k[i] == k && done_smem[i] == smem && done_dev[i] == dev) return done_n[i];
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kThreads, static_cast<size_t>(smem)) != cudaSuccess)
        n = 1;
    n = n < 1 ? 1 : n;
    if (n_done < kSlots) {
        done_k[n_done] = k;
        done_smem[n_done] = smem;
        done_dev[n_done] = dev;
        done_n[n_done] = n;
        ++n_done;
    }
    return n;
}

// Bulk-copy CTAs per SM of a launch: the caller's count, or cfg.tma_waves
// resident waves (default two).  GB300, chained bucket launches, two waves
// against one CTA per SM: BERT-large W=4 7.05 -> 7.12 TB/s, GPT-2-medium at
// cap 25 and 100 +1.6 / +1.3 %, ResNet-50 W=8 +0.7 %, no_sync ResNet-50 W=16
// micro-steps +6 %.  A single launch over a whole iteration (reduce_all)
// takes at least eight (BERT-large 6.78 (one wave) -> 6.97 (four) -> 7.07
// TB/s), more when its slices stay long (see launch_reduce_tma).
template <typename K>
int tma_ctas(const LaunchCfg& cfg, K k, long long smem) {
    const int waves = cfg.tma_waves > 0 ? cfg.tma_waves : 2;
    return cfg.tma_ctas_per_sm > 0 ? cfg.tma_ctas_per_sm : waves * resident_ctas(k, smem);
}

}  // namespace

cudaError_t launch_wait_selftest(long long limit_cycles, int* status, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_cycles, status);
    return cudaGetLastError();
}

cudaError_t launch_accumulate_tma(const AccPair* pairs, int n, const LaunchCfg& cfg,
                                  cudaStream_t stream, long long* launches) {
    thread_local AccParams p;   // ~32 KiB: kept off the stack, one per host thread
    const int stages = cfg.stages < 2 ? 2 : cfg.stages;
    long long tile = static_cast<long long>(cfg.stage_bytes) / (2 * static_cast<long long>(sizeof(float))) / 4 * 4;
    if (tile < 4) tile = 4;
    while (tile > 4 && kHeaderBytes + stages * 2 * tile * static_cast<long long>(sizeof(float)) > kMaxDynSmem) tile -= 4;
    const long long smem = kHeaderBytes + stages * 2 * tile * static_cast<long long>(sizeof(float));
    if (smem > kMaxDynSmem || 2 * stages * 8 > kHeaderBytes) return cudaErrorInvalidValue;
    cudaError_t e = ensure_smem_attr(accumulate_tma_kernel);
    if (e != cudaSuccess) return e;
    const int per_sm = tma_ctas(cfg, accumulate_tma_kernel, smem);
    int i = 0;
    int issued = 0;
    while (i < n) {
        p.npairs = 0;
        p.chain = cfg.pdl && issued > 0 ? 1 : 0;
        p.stages = stages;
        p.tile = static_cast<int>(tile);
        p.status = cfg.status;
        long long off = 0;
        while (i < n && p.npairs < kMaxAccPairs) {
            if (pairs[i].len > 0) {
                AccPairDev& d = p.pair[p.npairs++];
                d.g = pairs[i].g;
                d.acc = pairs[i].acc;
                d.off = off;
                d.len = pairs[i].len;
                d.assign = pairs[i].assign;
                d.pad = 0;
                off += (pairs[i].len + 3) / 4 * 4;
            }
            ++i;
        }
        if (p.npairs == 0) continue;
        p.total = off;
        long long grid = static_cast<long long>(cfg.sms) * per_sm;
        // The call's last launch has no successor in the call to overlap its
        // tail: as many resident waves (two to eight) as leave every CTA four
        // stages.  GB300, no_sync ResNet-50 W=16 K=8: cycle 7,028 -> 7,051
        // GB/s, adding micro-step 7,043 -> 7,064; eight stages gained less.
        if (i >= n && cfg.tma_ctas_per_sm == 0) {
            const int resident = resident_ctas(accumulate_tma_kernel, smem);
            long long waves = off / (static_cast<long long>(cfg.sms) * resident * kAccLastMinStages * tile);
            waves = waves < 2 ? 2 : waves > 8 ? 8 : waves;
            grid = static_cast<long long>(cfg.sms) * resident * waves;
        }
        grid = grid < ceil_div(off, tile) ? grid : ceil_div(off, tile);
        if (grid < 1) grid = 1;
        p.piece = ceil_div(ceil_div(off, grid), 4) * 4;
        grid = ceil_div(off, p.piece);
        cudaLaunchConfig_t lc = {};
        lc.gridDim = dim3(static_cast<unsigned>(grid));
        lc.blockDim = dim3(kThreads);
        lc.dynamicSmemBytes = static_cast<size_t>(smem);
        lc.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        lc.attrs = attr;
        lc.numAttrs = cfg.pdl ? 1 : 0;
        e = cudaLaunchKernelEx(&lc, accumulate_tma_kernel, p);
        if (e != cudaSuccess) return e;
        ++issued;
        if (launches) ++*launches;
    }
    return cudaSuccess;
}

cudaError_t launch_reduce_tma(const SegTable& t, InType in, int W, int n_out, float* arena,
                              long long lo, long long hi, int s0, int s1, float inv_w,
                              const LaunchCfg& cfg, cudaStream_t stream, long long* launches,
                              const SegMask* mask) {
    if (hi <= lo || s1 <= s0) return cudaSuccess;
    if (t.add && (mask || in != IN_F32)) return cudaErrorInvalidValue;   // no such variant
    if (cfg.compress && (t.add || mask || in != IN_F32)) return cudaErrorInvalidValue;
    const int N = in == IN_F32 ? 4 : 8;
    const int s_in = in == IN_F32 ? 4 : 2;
    const long long NS = t.add ? 2LL * W : W;   // tiles per stage
    // A stage holds one copy per stream.  Copies under a few KiB run into the
    // copy engine's per-request cost (measured on GB300: 1 KiB copies reach
    // ~4.5 TB/s, 4 KiB ones ~6.8), so many streams get larger stages, and
    // fewer of them where the ring would not fit.
    long long stage_bytes = cfg.stage_bytes;
    if (stage_bytes < NS * kMinCopyBytes) stage_bytes = NS * kMinCopyBytes;
    int stages = cfg.stages < 2 ? 2 : cfg.stages;
    while (stages > 2 && kHeaderBytes + stages * stage_bytes > kMaxDynSmem) --stages;
    long long tile = stage_bytes / (NS * s_in) / N * N;
    if (tile < N) tile = N;
    while (tile > N && kHeaderBytes + static_cast<long long>(stages) * NS * tile * s_in > kMaxDynSmem)
        tile -= N;
    const long long smem = kHeaderBytes + static_cast<long long>(stages) * NS * tile * s_in;
    if (smem > kMaxDynSmem || 2 * stages * 8 > kHeaderBytes) return cudaErrorInvalidValue;

    ReduceParams p = {};
    p.seg_off = t.seg_off;
    p.seg_src = t.seg_src;
    p.seg_dst = t.seg_dst;
    p.seg_vec = t.seg_vec;
    p.status = t.status;
    p.arena = arena;
    p.lo = lo;
    p.hi = hi;
    p.base = lo - lo % N;
    p.s0 = s0;
    p.s1 = s1;
    p.W = W;
    p.n_out = n_out;
    p.inv_w = inv_w;
    p.stages = stages;
    p.tile = static_cast<int>(tile);
    p.chain = cfg.chain;
    const TmaKernel<NoMask> plain = t.add ? pick_tma_add(W) : cfg.compress ? pick_tma_cmp(W) : pick_tma<NoMask>(in, W);
    cudaError_t e = mask ? ensure_smem_attr(pick_tma<SegMask>(in, W)) : ensure_smem_attr(plain);
    if (e != cudaSuccess) return e;
    const int resident = mask ? resident_ctas(pick_tma<SegMask>(in, W), smem) : resident_ctas(plain, smem);
    int per_sm = mask ? tma_ctas(cfg, pick_tma<SegMask>(in, W), smem) : tma_ctas(cfg, plain, smem);
    p.first_wave = cfg.sms * resident;
    // The final launch of an iteration has no successor to overlap its tail:
    // it gets as many resident waves (two to eight) as leave every CTA at
    // least kLastMinStages stages of work, so its slices, and its tail, are
    // shorter.  GB300, against two waves: BERT-large W=4 (last launch: the
    // 31M-element word embedding) 7,118 -> 7,173 GB/s, one call per event
    // +0.45 %, GPT-2-medium caps 25 / 100 +1.3 / +1.6 %; ResNet-50 W=8 (a
    // 4.3M-element last bucket: two waves either way) unchanged.  At least
    // four stages per CTA cost ResNet-50 1 %, sixteen gained less.
    // ddp_reduce_all's single launch over the whole iteration (cfg.tma_waves
    // above two) likewise takes eight to 64 waves, as many as leave every CTA
    // kWholeMinStages stages: GB300, against eight waves, BERT-large W=4
    // 7,043 -> 7,156 GB/s at 48 waves (11 stages per CTA), GPT-2-medium at
    // cap 25 6,972 -> 7,171 at 64 (9 stages), ResNet-50 W=8 best at 8-12
    // (7-10 stages) and 12 % slower at 32 waves (3 stages).  Other launches
    // keep two waves unless their slices would exceed kWholeMinStages stages
    // (GPT-2-medium's 100 MiB buckets: 7,127 -> 7,166 GB/s; buckets of 25 MiB
    // and less keep two waves).
    if (cfg.tma_ctas_per_sm == 0) {
        // Grids sized by their slices: as many resident waves, within
        // [lo_w, hi_w], as leave every CTA min_st stages of work.
        long long lo_w = 0, hi_w = 0, min_st = 0;
        if (cfg.last && cfg.tma_waves > 2) {          // ddp_reduce_all: the whole iteration
            lo_w = cfg.tma_waves, hi_w = kWholeMaxWaves, min_st = kWholeMinStages;
        } else if (cfg.last) {                        // an iteration's final launch
            lo_w = 2, hi_w = 8, min_st = kLastMinStages;
        } else if (cfg.tma_waves == 2) {              // any other launch (not W = 1's single wave)
            lo_w = 2, hi_w = kWholeMaxWaves, min_st = kWholeMinStages;
        }
        if (hi_w > 0) {
            long long waves = (hi - lo) / (static_cast<long long>(p.first_wave) * min_st * tile);
            waves = waves < lo_w ? lo_w : waves > hi_w ? hi_w : waves;
            per_sm = static_cast<int>(waves) * resident;
        }
    }

    const long long span = hi - p.base;
    long long grid = static_cast<long long>(cfg.sms) * per_sm;
    grid = grid < ceil_div(span, tile) ? grid : ceil_div(span, tile);
    if (grid < 1) grid = 1;
    p.piece = ceil_div(ceil_div(span, grid), N) * N;
    grid = ceil_div(span, p.piece);

    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(static_cast<unsigned>(grid));
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = static_cast<size_t>(smem);
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = cfg.pdl ? 1 : 0;
#ifdef DDP_TRACE
    {
        std::lock_guard<std::mutex> lock(g_trace_mutex);
        p.trace_slot = static_cast<int>(g_trace_seq % DDP_TRACE_LAUNCHES);
        g_trace_grid[p.trace_slot] = static_cast<int>(grid);
        ++g_trace_seq;
    }
#endif
    e = mask ? cudaLaunchKernelEx(&lc, pick_tma<SegMask>(in, W), p, *mask)
             : cudaLaunchKernelEx(&lc, plain, p, NoMask{});
    if (e == cudaSuccess && launches) ++*launches;
    return e;
}

cudaError_t read_launch_trace(unsigned long long* out, int* grid, long long* seq) {
#ifdef DDP_TRACE
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    if (out) {
        e = cudaMemcpyFromSymbol(out, g_launch_trace, sizeof(g_launch_trace));
        if (e != cudaSuccess) return e;
    }
    std::lock_guard<std::mutex> lock(g_trace_mutex);
    if (grid)
        for (int i = 0; i < DDP_TRACE_LAUNCHES; ++i) grid[i] = g_trace_grid[i];
    if (seq) *seq = g_trace_seq;
#else
    (void)out;
    (void)grid;
    if (seq) *seq = -1;
#endif
    return cudaSuccess;
}

}  // namespace ddpk
