// Device kernels of the DDP Reducer gradient path for sm_103a (GB300).
//
// bucket_reduce_kernel -- the fused bucket pass: for every element of the
//   launched bucket range, read the W replicas' gradients straight from their
//   per-parameter tensors (the gather into the bucket view needs no staging
//   copy), sum them in fp32 in rank order, scale by fl32(1/W), and write the
//   result into the bucket arena and into each copy-back output.  The
//   operation follows the gradient path of "PyTorch Distributed: Experiences
//   on Accelerating Data Parallel Training" (bucket copy, all-reduce to the
//   mean, copy-back) and "Distributed Data Parallel" notes, "Backward pass";
//   the one-GPU emulation turns the all-reduce over W ranks into arithmetic.
//
// accumulate_kernel -- no_sync micro-step: acc = g or acc = fl32(acc + g)
//   ("PyTorch Distributed", Section 3.2.4, gradient accumulation).
//
// Both are HBM-streaming kernels (about 0.2 flop per byte): no tensor cores.
// Design for GB300:
//   * a grid of resident waves (SMs x resident CTAs x waves), each CTA owning
//     one contiguous, equal slice of the launch's flat element range, so a
//     bucket range of any shape (one 125 MiB embedding or hundreds of
//     1024-element LayerNorm vectors) costs one launch and balances across all
//     152 SMs; with more CTAs than fit at once, SMs that finish a slice early
//     take another;
//   * the CTA finds the segment holding its first element with a 32-way
//     warp-ballot search over the segment offsets, then walks the segments;
//   * 128-bit loads through the non-coherent path without L1 allocation,
//     all W replicas x U vectors issued before the first add, and
//     evict-first 128-bit stores: each byte crosses HBM once;
//   * programmatic dependent launch: a launch triggers its successor at
//     entry, so the next bucket range's CTAs are resident when this one
//     drains; every launch still waits (griddepcontrol.wait) for its
//     predecessor before touching memory, so stream order is preserved
//     whatever precedes it.
// Bit exactness: accumulate starts at x_0 (keeps -0.0), adds with __fadd_rn
// in rank order and scales with __fmul_rn, so no FMA contraction and no
// flush-to-zero (the build never uses fast-math).

#include <cstdint>
#include <cuda_runtime.h>

#include "ddp_device.cuh"
#include "ddp_kernels.h"

namespace ddpk {

namespace {

using namespace dev;

constexpr int kMaxBlock = 256;

// Vectors per replica in flight per thread in the fixed-W vector body
// (W x U loads issued before the first add).  U = 2 measured best on GB300
// for W = 4 and W = 8; W = 16 uses 1 to stay within registers.
template <int WC>
__host__ __device__ constexpr int unroll_for() { return WC <= 2 ? 4 : (WC <= 8 ? 2 : 1); }

// The bucket kernel's unroll for NSC streams of Tin: bf16 vectors hold 8
// elements, so half the unroll keeps the loads in flight per SM with half the
// registers and twice the resident warps (GB300, GPT-2-medium W = 8 bf16,
// per-gradient buckets: +1 %; 1 MiB buckets: +2 %).
template <typename Tin, int NSC>
__host__ __device__ constexpr int reduce_unroll() {
    return sizeof(Tin) == 2 && unroll_for<NSC>() > 1 ? unroll_for<NSC>() / 2 : unroll_for<NSC>();
}

// A replica's 16-byte vector, or zeros when the replica has no gradient for
// the segment (its zero-filled bucket slice).
template <typename Raw>
__device__ __forceinline__ Raw zero_raw() { return Raw{}; }

// Vector body, W known at compile time: all NS x U loads in flight at once
// (NS = WC streams, or 2 WC with ADD: the accumulated fields and the last
// micro-step's gradients).  Replica r's input is its vector, or with ADD
// fl32(acc_r + g_r), or with CMP its vector rounded to bf16, added into the
// rank-order sum.
template <typename Tin, int WC, int U, bool ADD, bool CMP>
__device__ __forceinline__ void reduce_vec_fixed(const ReduceParams& p, const Tin* const* src,
                                                 float* const* dst, long long a0, long long kb,
                                                 long long ke, unsigned long long mk) {
    using V = Vec<Tin>;
    constexpr int N = V::N;
    constexpr int NS = ADD ? 2 * WC : WC;
    const bool write_dst = any_replica(mk, WC);
    const Tin* s[NS];
#pragma unroll
    for (int r = 0; r < NS; ++r) s[r] = src[r];
    const long long step = static_cast<long long>(blockDim.x);
    for (long long k = kb + threadIdx.x; k < ke; k += U * step) {
        typename V::Raw raw[U][NS];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long kk = k + u * step;
            if (kk < ke) {
                const long long j = kk * N - a0;
#pragma unroll
                for (int r = 0; r < NS; ++r)
                    raw[u][r] = has_replica(mk, r % WC)
                                    ? ld_stream(reinterpret_cast<const typename V::Raw*>(s[r] + j))
                                    : zero_raw<typename V::Raw>();
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const long long kk = k + u * step;
            if (kk < ke) {
                float acc[N], f[N];
                V::unpack(raw[u][0], acc);
                if constexpr (ADD) {
                    V::unpack(raw[u][WC], f);
#pragma unroll
                    for (int q = 0; q < N; ++q) acc[q] = __fadd_rn(acc[q], f[q]);
                }
                if constexpr (CMP) {
#pragma unroll
                    for (int q = 0; q < N; ++q) acc[q] = round_bf16(acc[q]);
                }
#pragma unroll
                for (int r = 1; r < WC; ++r) {
                    V::unpack(raw[u][r], f);
                    if constexpr (ADD) {
                        float h[N];
                        V::unpack(raw[u][WC + r], h);
#pragma unroll
                        for (int q = 0; q < N; ++q) f[q] = __fadd_rn(f[q], h[q]);
                    }
                    if constexpr (CMP) {
#pragma unroll
                        for (int q = 0; q < N; ++q) f[q] = round_bf16(f[q]);
                    }
#pragma unroll
                    for (int q = 0; q < N; ++q) acc[q] = __fadd_rn(acc[q], f[q]);
                }
#pragma unroll
                for (int q = 0; q < N; ++q) acc[q] = __fmul_rn(acc[q], p.inv_w);
                store_vec<N>(p, dst, kk * N, kk * N - a0, acc, write_dst);
            }
        }
    }
}

// One replica's 16-byte vector of inputs (ADD: accumulated + last step;
// CMP: rounded to bf16).
template <typename Tin, bool ADD, bool CMP>
__device__ __forceinline__ void load_replica(const Tin* const* src, int W, int r, long long j,
                                             unsigned long long mk, float (&f)[Vec<Tin>::N]) {
    using V = Vec<Tin>;
    using Raw = typename V::Raw;
    if (!has_replica(mk, r)) {
        V::unpack(zero_raw<Raw>(), f);
        return;
    }
    V::unpack(ld_stream(reinterpret_cast<const Raw*>(src[r] + j)), f);
    if constexpr (ADD) {
        float h[V::N];
        V::unpack(ld_stream(reinterpret_cast<const Raw*>(src[W + r] + j)), h);
#pragma unroll
        for (int q = 0; q < V::N; ++q) f[q] = __fadd_rn(f[q], h[q]);
    }
    if constexpr (CMP) {
#pragma unroll
        for (int q = 0; q < V::N; ++q) f[q] = round_bf16(f[q]);
    }
}

// Vector body for any W: replicas in groups of 4, still summed in rank order.
template <typename Tin, bool ADD, bool CMP>
__device__ __forceinline__ void reduce_vec_any(const ReduceParams& p, const Tin* const* src,
                                               float* const* dst, long long a0, long long kb,
                                               long long ke, int W, unsigned long long mk) {
    using V = Vec<Tin>;
    constexpr int N = V::N;
    const bool write_dst = any_replica(mk, W);
    for (long long k = kb + threadIdx.x; k < ke; k += blockDim.x) {
        const long long j = k * N - a0;
        float acc[N];
        load_replica<Tin, ADD, CMP>(src, W, 0, j, mk, acc);
        for (int r = 1; r < W; r += 4) {
            float f[4][N];
#pragma unroll
            for (int g = 0; g < 4; ++g)
                if (r + g < W) load_replica<Tin, ADD, CMP>(src, W, r + g, j, mk, f[g]);
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                if (r + g < W) {
#pragma unroll
                    for (int q = 0; q < N; ++q) acc[q] = __fadd_rn(acc[q], f[g][q]);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < N; ++q) acc[q] = __fmul_rn(acc[q], p.inv_w);
        store_vec<N>(p, dst, k * N, j, acc, write_dst);
    }
}

// M = NoMask (every replica has every gradient) or SegMask (unused parameters).
// ADD: fused last micro-step of a no_sync block (2W source streams per
// segment, see SegTable).  CMP: the bf16-compression hook fused into the
// pass (each replica value rounded to bf16 before the sum).
template <typename Tin, int WC, typename M, bool ADD, bool CMP = false>
__global__ void __launch_bounds__(kMaxBlock)
bucket_reduce_kernel(const __grid_constant__ ReduceParams p, const __grid_constant__ M mask) {
    pdl_enter(p.chain);
    using V = Vec<Tin>;
    constexpr int N = V::N;
    constexpr int U = WC == 0 ? 1 : reduce_unroll<Tin, ADD ? 2 * WC : WC>();
    const int W = WC > 0 ? WC : p.W;
    const int NS = ADD ? 2 * W : W;

    long long x = p.base + static_cast<long long>(blockIdx.x) * p.piece;
    long long y = x + p.piece;
    x = x < p.lo ? p.lo : x;
    y = y > p.hi ? p.hi : y;
    if (x >= y) {   // whole CTA leaves together
        if (threadIdx.x == 0) pdl_exit(p.chain, p.piece >= kHoldAllPiece);
        return;
    }

    int s = find_segment(p.seg_off, p.s0, p.s1, x);
    while (x < y) {
        const long long a0 = __ldg(p.seg_off + s);
        const long long a1 = __ldg(p.seg_off + s + 1);
        const long long e = a1 < y ? a1 : y;
        if (!debug_ok(p.status, s < p.s1 && a0 <= x && x < e && e <= a1 && p.lo <= x && e <= p.hi, kDbgSegRange, x))
            break;
        const Tin* const* src = reinterpret_cast<const Tin* const*>(p.seg_src) + static_cast<long long>(s) * NS;
        float* const* dst = p.seg_dst + static_cast<long long>(s) * p.n_out;
        const unsigned long long mk = seg_mask(mask, s - p.s0);
        const long long kb = (x + N - 1) / N;   // first whole vector
        const long long ke = e / N;             // one past the last whole vector
        if (__ldg(p.seg_vec + s) && kb < ke) {
            reduce_scalar<Tin, ADD, CMP>(p, src, dst, a0, x, kb * N, W, threadIdx.x, blockDim.x, mk);
            if constexpr (WC > 0)
                reduce_vec_fixed<Tin, WC, U, ADD, CMP>(p, src, dst, a0, kb, ke, mk);
            else
                reduce_vec_any<Tin, ADD, CMP>(p, src, dst, a0, kb, ke, W, mk);
            reduce_scalar<Tin, ADD, CMP>(p, src, dst, a0, ke * N, e, W, threadIdx.x, blockDim.x, mk);
        } else {
            reduce_scalar<Tin, ADD, CMP>(p, src, dst, a0, x, e, W, threadIdx.x, blockDim.x, mk);
        }
        x = e;
        ++s;
    }
    if (threadIdx.x == 0) pdl_exit(p.chain, p.piece >= kHoldAllPiece);
}

// ------------------------------------------------------------------ accumulate kernel

__global__ void __launch_bounds__(kMaxBlock)
accumulate_kernel(const __grid_constant__ AccParams p) {
    pdl_enter(p.chain);
    long long x = static_cast<long long>(blockIdx.x) * p.piece;
    long long y = x + p.piece;
    y = y > p.total ? p.total : y;
    if (x >= y) {
        if (threadIdx.x == 0) pdl_exit(p.chain, false);
        return;
    }
    int i = find_pair(p, x);
    const long long step = blockDim.x;
    while (x < y && i < p.npairs) {
        const AccPairDev& q = p.pair[i];
        const long long end = q.off + q.len;
        const long long e = end < y ? end : y;
        if (x < e) {
            if (!debug_ok(p.status, q.off <= x && e <= p.total, kDbgPairRange, x)) break;
            const bool assign = q.assign != 0;
            const float* g = q.g - q.off;      // indexed by flat position
            float* acc = q.acc - q.off;
            const bool vec = ((reinterpret_cast<uintptr_t>(q.g) | reinterpret_cast<uintptr_t>(q.acc)) & 15u) == 0;
            long long kb = (x + 3) >> 2, ke = e >> 2;
            if (!vec || kb >= ke) { kb = ke = 0; }
            const long long sc_end = vec && kb < ke ? kb * 4 : e;
            for (long long a = x + threadIdx.x; a < sc_end; a += step)
                acc[a] = assign ? g[a] : __fadd_rn(acc[a], g[a]);
            constexpr int UA = 4;   // vectors per thread per iteration: 2 x 4 loads in flight
            for (long long k = kb + threadIdx.x; k < ke; k += UA * step) {
                float4 gv[UA], cv[UA];
#pragma unroll
                for (int u = 0; u < UA; ++u) {
                    const long long kk = k + u * step;
                    if (kk < ke) {
                        gv[u] = ld_stream(reinterpret_cast<const float4*>(g + 4 * kk));
                        if (!assign) cv[u] = __ldcs(reinterpret_cast<const float4*>(acc + 4 * kk));
                    }
                }
#pragma unroll
                for (int u = 0; u < UA; ++u) {
                    const long long kk = k + u * step;
                    if (kk < ke) {
                        if (assign) {
                            st_stream(acc + 4 * kk, gv[u]);
                        } else {
                            st_stream(acc + 4 * kk, make_float4(__fadd_rn(cv[u].x, gv[u].x), __fadd_rn(cv[u].y, gv[u].y),
                                                                __fadd_rn(cv[u].z, gv[u].z), __fadd_rn(cv[u].w, gv[u].w)));
                        }
                    }
                }
            }
            if (vec && kb < ke)
                for (long long a = ke * 4 + threadIdx.x; a < e; a += step)
                    acc[a] = assign ? g[a] : __fadd_rn(acc[a], g[a]);
        }
        x = end > x ? end : x;
        // skip the padding up to the next pair's start
        ++i;
        if (i < p.npairs && p.pair[i].off > x) x = p.pair[i].off;
    }
    if (threadIdx.x == 0) pdl_exit(p.chain, false);
}

// ------------------------------------------------------------------ hook path kernels

struct CopyParams {
    const long long* seg_off;
    const void* const* seg_src;
    float* const* seg_dst;
    const int* seg_vec;
    const float* arena;
    int* status;
    long long base, lo, hi, piece;
    int s0, s1;
    int W, n_out;
    int mode;   // 0 gather, 1 copy-back
    int elem;   // bytes per element (gather: gradient dtype; copy-back: 4)
    void* rb[kMaxHookReplicas];
};

__device__ __forceinline__ void copy_elem(char* d, const char* s, int elem) {
    if (elem == 4) *reinterpret_cast<float*>(d) = *reinterpret_cast<const float*>(s);
    else *reinterpret_cast<uint16_t*>(d) = *reinterpret_cast<const uint16_t*>(s);
}

// One run: `from` holds the segment's elements starting at its first one,
// `to` is indexed like `from` (both already offset); elements [x, e) of the
// segment, 16-byte vectors where the run is aligned.
__device__ __forceinline__ void copy_run(const char* from, char* to, long long a0, long long x, long long e,
                                         int elem, bool vec) {
    const int n = 16 / elem;
    long long kb = (x + n - 1) / n, ke = e / n;
    if (!vec || kb >= ke) kb = ke = 0;
    const long long sc_end = vec && kb < ke ? kb * n : e;
    for (long long a = x + threadIdx.x; a < sc_end; a += blockDim.x)
        copy_elem(to + (a - a0) * elem, from + (a - a0) * elem, elem);
    // UC independent 16-byte vectors per thread in flight.  One: at 32
    // registers eight 256-thread CTAs fit per SM and the warps keep the loads
    // in flight (GB300, BERT-large W=4 through the gathered hook route:
    // 2,499 -> 2,594 GB/s against four vectors at 80 registers and three
    // CTAs per SM; two and three vectors in between).
#ifndef DDP_COPY_UNROLL
#define DDP_COPY_UNROLL 1
#endif
    constexpr int UC = DDP_COPY_UNROLL;
    const long long step = blockDim.x;
    for (long long k = kb + threadIdx.x; k < ke; k += UC * step) {
        float4 v[UC];
#pragma unroll
        for (int u = 0; u < UC; ++u)
            if (k + u * step < ke) v[u] = __ldcs(reinterpret_cast<const float4*>(from + ((k + u * step) * n - a0) * elem));
#pragma unroll
        for (int u = 0; u < UC; ++u)
            if (k + u * step < ke) st_stream(reinterpret_cast<float*>(to + ((k + u * step) * n - a0) * elem), v[u]);
    }
    if (vec && kb < ke)
        for (long long a = ke * n + threadIdx.x; a < e; a += blockDim.x)
            copy_elem(to + (a - a0) * elem, from + (a - a0) * elem, elem);
}

__global__ void __launch_bounds__(kMaxBlock) seg_copy_kernel(const __grid_constant__ CopyParams p) {
    pdl_enter(0);
    long long x = p.base + static_cast<long long>(blockIdx.x) * p.piece;
    long long y = x + p.piece;
    x = x < p.lo ? p.lo : x;
    y = y > p.hi ? p.hi : y;
    if (x >= y) return;
    int s = find_segment(p.seg_off, p.s0, p.s1, x);
    while (x < y) {
        const long long a0 = __ldg(p.seg_off + s);
        const long long a1 = __ldg(p.seg_off + s + 1);
        const long long e = a1 < y ? a1 : y;
        if (!debug_ok(p.status, s < p.s1 && a0 <= x && x < e && e <= a1 && p.lo <= x && e <= p.hi, kDbgSegRange, x))
            break;
        const bool vec = __ldg(p.seg_vec + s) != 0;
        if (p.mode == 0) {
            for (int r = 0; r < p.W; ++r) {
                const char* from = static_cast<const char*>(p.seg_src[static_cast<long long>(s) * p.W + r]);
                char* to = static_cast<char*>(p.rb[r]) + a0 * p.elem;
                copy_run(from, to, a0, x, e, p.elem, vec);
            }
        } else {
            const char* from = reinterpret_cast<const char*>(p.arena + a0);
            for (int o = 0; o < p.n_out; ++o)
                copy_run(from, reinterpret_cast<char*>(p.seg_dst[static_cast<long long>(s) * p.n_out + o]), a0, x,
                         e, 4, vec);
        }
        x = e;
        ++s;
    }
}

struct FlatMeanParams {
    float* out;
    long long n;
    float inv_w;
    int W;
    int compress;
    const void* src[kMaxHookReplicas];
};

template <typename Tin>
__device__ __forceinline__ float flat_term(const FlatMeanParams& p, int r, long long i) {
    const float x = widen1(static_cast<const Tin*>(p.src[r])[i]);
    return p.compress ? round_bf16(x) : x;
}

// vec != 0: every pointer 16-byte aligned; 16-byte loads over whole vectors,
// the tail element by element.  WC > 0: W known at compile time, W x U
// loads in flight per thread before the first add (as in the fused pass).
template <typename Tin, int WC>
__global__ void __launch_bounds__(kMaxBlock) flat_mean_kernel(const __grid_constant__ FlatMeanParams p, int vec) {
    pdl_enter(0);
    using V = Vec<Tin>;
    using Raw = typename V::Raw;
    constexpr int N = V::N;
    constexpr int U = WC == 0 ? 1 : unroll_for<WC>();
    const int W = WC > 0 ? WC : p.W;
    const long long step = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long t0 = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long nv = vec ? p.n / N : 0;
    auto term = [&](float x) { return p.compress ? round_bf16(x) : x; };
    if constexpr (WC > 0) {
        for (long long k = t0; k < nv; k += U * step) {
            Raw raw[U][WC];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (k + u * step < nv)
#pragma unroll
                    for (int r = 0; r < WC; ++r)
                        raw[u][r] = ld_stream(reinterpret_cast<const Raw*>(static_cast<const Tin*>(p.src[r]) +
                                                                           (k + u * step) * N));
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const long long kk = k + u * step;
                if (kk < nv) {
                    float acc[N], f[N];
                    V::unpack(raw[u][0], acc);
#pragma unroll
                    for (int q = 0; q < N; ++q) acc[q] = term(acc[q]);
#pragma unroll
                    for (int r = 1; r < WC; ++r) {
                        V::unpack(raw[u][r], f);
#pragma unroll
                        for (int q = 0; q < N; ++q) acc[q] = __fadd_rn(acc[q], term(f[q]));
                    }
#pragma unroll
                    for (int q = 0; q < N; q += 4)
                        st_stream(p.out + kk * N + q,
                                  make_float4(__fmul_rn(acc[q], p.inv_w), __fmul_rn(acc[q + 1], p.inv_w),
                                              __fmul_rn(acc[q + 2], p.inv_w), __fmul_rn(acc[q + 3], p.inv_w)));
                }
            }
        }
    } else {
        for (long long k = t0; k < nv; k += step) {
            float acc[N], f[N];
            V::unpack(ld_stream(reinterpret_cast<const Raw*>(static_cast<const Tin*>(p.src[0]) + k * N)), acc);
#pragma unroll
            for (int q = 0; q < N; ++q) acc[q] = term(acc[q]);
            for (int r = 1; r < W; ++r) {
                V::unpack(ld_stream(reinterpret_cast<const Raw*>(static_cast<const Tin*>(p.src[r]) + k * N)), f);
#pragma unroll
                for (int q = 0; q < N; ++q) acc[q] = __fadd_rn(acc[q], term(f[q]));
            }
#pragma unroll
            for (int q = 0; q < N; q += 4)
                st_stream(p.out + k * N + q, make_float4(__fmul_rn(acc[q], p.inv_w), __fmul_rn(acc[q + 1], p.inv_w),
                                                         __fmul_rn(acc[q + 2], p.inv_w), __fmul_rn(acc[q + 3], p.inv_w)));
        }
    }
    for (long long i = nv * N + t0; i < p.n; i += step) {
        float acc = flat_term<Tin>(p, 0, i);
        for (int r = 1; r < W; ++r) acc = __fadd_rn(acc, flat_term<Tin>(p, r, i));
        p.out[i] = __fmul_rn(acc, p.inv_w);
    }
}

// ------------------------------------------------------------------ launch helpers

template <typename Kernel, typename... Params>
cudaError_t launch(Kernel k, int grid, int block, bool pdl, cudaStream_t st, const Params&... params) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(block));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, params...);
}

template <typename M>
using ReduceKernel = void (*)(ReduceParams, M);

template <typename M>
ReduceKernel<M> pick_reduce(InType in, int W) {
    if (in == IN_F32) {
        switch (W) {
            case 2: return bucket_reduce_kernel<float, 2, M, false>;
            case 4: return bucket_reduce_kernel<float, 4, M, false>;
            case 8: return bucket_reduce_kernel<float, 8, M, false>;
            case 16: return bucket_reduce_kernel<float, 16, M, false>;
            default: return bucket_reduce_kernel<float, 0, M, false>;
        }
    }
    switch (W) {
        case 2: return bucket_reduce_kernel<uint16_t, 2, M, false>;
        case 4: return bucket_reduce_kernel<uint16_t, 4, M, false>;
        case 8: return bucket_reduce_kernel<uint16_t, 8, M, false>;
        case 16: return bucket_reduce_kernel<uint16_t, 16, M, false>;
        default: return bucket_reduce_kernel<uint16_t, 0, M, false>;
    }
}

// bf16-compression variant: fp32 gradients, every replica present.
ReduceKernel<NoMask> pick_reduce_cmp(int W) {
    switch (W) {
        case 2: return bucket_reduce_kernel<float, 2, NoMask, false, true>;
        case 4: return bucket_reduce_kernel<float, 4, NoMask, false, true>;
        case 8: return bucket_reduce_kernel<float, 8, NoMask, false, true>;
        case 16: return bucket_reduce_kernel<float, 16, NoMask, false, true>;
        default: return bucket_reduce_kernel<float, 0, NoMask, false, true>;
    }
}

// Fused last-step variant: fp32 accumulators, every replica present.
ReduceKernel<NoMask> pick_reduce_add(int W) {
    switch (W) {
        case 2: return bucket_reduce_kernel<float, 2, NoMask, true>;
        case 4: return bucket_reduce_kernel<float, 4, NoMask, true>;
        case 8: return bucket_reduce_kernel<float, 8, NoMask, true>;
        case 16: return bucket_reduce_kernel<float, 16, NoMask, true>;
        default: return bucket_reduce_kernel<float, 0, NoMask, true>;
    }
}

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

}  // namespace

int reduce_max_ctas_per_sm(InType in, int W, int block, bool add) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, add ? pick_reduce_add(W) : pick_reduce<NoMask>(in, W),
                                                      block, 0) != cudaSuccess)
        return 1;
    return n > 0 ? n : 1;
}

int accumulate_max_ctas_per_sm(int block) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, accumulate_kernel, block, 0) != cudaSuccess)
        return 1;
    return n > 0 ? n : 1;
}

cudaError_t launch_reduce(const SegTable& t, InType in, int W, int n_out, float* arena,
                          long long lo, long long hi, int s0, int s1, float inv_w,
                          const LaunchCfg& cfg, cudaStream_t stream, long long* launches,
                          const SegMask* mask) {
    if (hi <= lo || s1 <= s0) return cudaSuccess;
    if (cfg.kernel == KERNEL_TMA)
        return launch_reduce_tma(t, in, W, n_out, arena, lo, hi, s0, s1, inv_w, cfg, stream, launches, mask);
    const int N = in == IN_F32 ? 4 : 8;
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
    p.chain = cfg.chain;
    // One slice per CTA, at least two vectors per thread so tiny ranges use
    // few CTAs; slices are multiples of the vector width so no vector is split.
    const long long span = hi - p.base;
    const long long min_piece = static_cast<long long>(cfg.block) * N * 2;
    long long grid = static_cast<long long>(cfg.sms) * cfg.ctas_per_sm;
    grid = grid < ceil_div(span, min_piece) ? grid : ceil_div(span, min_piece);
    if (grid < 1) grid = 1;
    p.piece = ceil_div(ceil_div(span, grid), N) * N;
    grid = ceil_div(span, p.piece);
    if (t.add && (mask || in != IN_F32)) return cudaErrorInvalidValue;   // no such variant
    if (cfg.compress && (t.add || mask || in != IN_F32)) return cudaErrorInvalidValue;
    const ReduceKernel<NoMask> plain = t.add ? pick_reduce_add(W) : cfg.compress ? pick_reduce_cmp(W)
                                                                               : pick_reduce<NoMask>(in, W);
    cudaError_t err = mask ? launch(pick_reduce<SegMask>(in, W), static_cast<int>(grid), cfg.block, cfg.pdl,
                                    stream, p, *mask)
                           : launch(plain, static_cast<int>(grid), cfg.block, cfg.pdl, stream, p, NoMask{});
    if (err == cudaSuccess && launches) ++*launches;
    return err;
}

cudaError_t launch_seg_copy(const SegTable& t, int mode, int elem, int W, int n_out, const float* arena,
                            void* const* rb, long long lo, long long hi, int s0, int s1,
                            const LaunchCfg& cfg, cudaStream_t stream, long long* launches) {
    if (hi <= lo || s1 <= s0 || (mode == 1 && n_out == 0)) return cudaSuccess;
    if (W > kMaxHookReplicas) return cudaErrorInvalidValue;
    CopyParams p = {};
    p.seg_off = t.seg_off;
    p.seg_src = t.seg_src;
    p.seg_dst = t.seg_dst;
    p.seg_vec = t.seg_vec;
    p.arena = arena;
    p.status = t.status;
    p.lo = lo;
    p.hi = hi;
    const int n = 16 / (mode == 0 ? elem : 4);
    p.base = lo - lo % n;
    p.s0 = s0;
    p.s1 = s1;
    p.W = W;
    p.n_out = n_out;
    p.mode = mode;
    p.elem = mode == 0 ? elem : 4;
    for (int r = 0; r < W && mode == 0; ++r) p.rb[r] = rb[r];
    const long long span = hi - p.base;
    const long long min_piece = static_cast<long long>(cfg.block) * n * 2;
    // one resident wave of CTAs (a second, partial wave would only add a tail)
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, seg_copy_kernel, cfg.block, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    long long grid = static_cast<long long>(cfg.sms) * per_sm;
    grid = grid < ceil_div(span, min_piece) ? grid : ceil_div(span, min_piece);
    if (grid < 1) grid = 1;
    p.piece = ceil_div(ceil_div(span, grid), n) * n;
    grid = ceil_div(span, p.piece);
    cudaError_t err = launch(seg_copy_kernel, static_cast<int>(grid), cfg.block, cfg.pdl, stream, p);
    if (err == cudaSuccess && launches) ++*launches;
    return err;
}

cudaError_t launch_flat_mean(InType in, int W, const void* const* src, float* out, long long n, float inv_w,
                             int compress, int sms, cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    if (W < 1 || W > kMaxHookReplicas) return cudaErrorInvalidValue;
    FlatMeanParams p = {};
    p.out = out;
    p.n = n;
    p.inv_w = inv_w;
    p.W = W;
    p.compress = compress;
    int vec = (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
    for (int r = 0; r < W; ++r) {
        p.src[r] = src[r];
        vec = vec && (reinterpret_cast<uintptr_t>(src[r]) & 15u) == 0;
    }
    const int N = in == IN_F32 ? 4 : 8;
    using K = void (*)(FlatMeanParams, int);
    auto pick = [&](auto tag) -> K {
        using T = decltype(tag);
        switch (W) {
            case 2: return flat_mean_kernel<T, 2>;
            case 4: return flat_mean_kernel<T, 4>;
            case 8: return flat_mean_kernel<T, 8>;
            case 16: return flat_mean_kernel<T, 16>;
            default: return flat_mean_kernel<T, 0>;
        }
    };
    const K k = in == IN_F32 ? pick(float{}) : pick(uint16_t{});
    // one resident wave: the grid-stride loop covers the rest
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, 256, 0) != cudaSuccess || per_sm < 1) per_sm = 1;
    long long grid = ceil_div(vec ? ceil_div(n, N) : n, 256);
    const long long cap = static_cast<long long>(sms > 0 ? sms : 152) * per_sm;
    grid = grid < cap ? grid : cap;
    if (grid < 1) grid = 1;
    return launch(k, static_cast<int>(grid), 256, true, stream, p, vec);
}

cudaError_t launch_accumulate(const AccPair* pairs, int n, const LaunchCfg& cfg,
                              cudaStream_t stream, long long* launches) {
    if (cfg.kernel == KERNEL_TMA) return launch_accumulate_tma(pairs, n, cfg, stream, launches);
    thread_local AccParams p;   // ~32 KiB: kept off the stack, one per host thread
    int i = 0;
    int issued = 0;
    while (i < n) {
        p.npairs = 0;
        // launches after the first of this call directly follow it on the
        // stream and touch other pairs: no need to wait for it on entry
        p.chain = cfg.pdl && issued > 0 ? 1 : 0;
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
        const long long min_piece = static_cast<long long>(cfg.block) * 8;
        long long grid = static_cast<long long>(cfg.sms) * cfg.ctas_per_sm;
        grid = grid < ceil_div(off, min_piece) ? grid : ceil_div(off, min_piece);
        if (grid < 1) grid = 1;
        p.piece = ceil_div(ceil_div(off, grid), 4) * 4;
        grid = ceil_div(off, p.piece);
        cudaError_t err = launch(accumulate_kernel, static_cast<int>(grid), cfg.block, cfg.pdl, stream, p);
        if (err != cudaSuccess) return err;
        ++issued;
        if (launches) ++*launches;
    }
    return cudaSuccess;
}

}  // namespace ddpk
