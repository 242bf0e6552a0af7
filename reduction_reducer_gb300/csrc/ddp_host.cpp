// Host core of the DDP Reducer gradient path: bucket builder, readiness state
// machine, bind-time segment tables and the C ABI declared in ddp_reducer.h.
//
// Bucket assignment follows "NCCL 专家课程 30: DDP Reducer、Bucket 与计算通信重叠"
// (section "`bucket_cap_mb` 不是张量切分器": whole tensors, close once the size
// reaches the cap) and "PyTorch Distributed: Experiences on Accelerating Data
// Parallel Training" (Section 3.2.2: reverse registration order).  The state
// machine follows the same course page, sections "Variable 到 Bucket" and
// "Bucket 必须按序发起" (pending counts, next-bucket cursor, parking), and the
// prior-reduction check of "Distributed Data Parallel" notes, "When a
// parameter never receives a gradient".

#include "ddp_reducer.h"

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "ddp_kernels.h"

namespace {

thread_local std::string g_build_error;

}  // namespace

struct ddp_ctx {
    // ---- construction (host only)
    int32_t P = 0;
    ddp_dtype dtype = DDP_F32;
    int elem = 4;
    int64_t cap = 0;
    std::vector<int64_t> numel;
    std::vector<std::vector<int32_t>> members;   // per bucket, push order
    std::vector<ddp_locator> loc;                 // per variable
    std::vector<int64_t> bucket_off;              // B+1 arena offsets
    int32_t B = 0;

    // ---- iteration state
    bool active = false;
    std::vector<int32_t> pending;
    std::vector<uint8_t> ready;
    int32_t next = 0;

    int64_t first_cap = 0;
    std::vector<int32_t> trace_cur;               // ready events of the current iteration
    std::vector<int32_t> trace_last;              // ... of the last finished iteration

    // ---- unused parameters (DDP_OPT_FIND_UNUSED)
    bool opt_find_unused = false;
    std::vector<uint8_t> pending_used;            // W*P: OR of local-use bits since the last reduction
    bool pending_set = false;
    std::vector<uint8_t> iter_used;               // W*P: bits of the current iteration
    std::vector<uint8_t> gused;                   // P: used on some replica
    bool iter_masked = false;                     // some replica lacks some gradient
    bool unused_marked = false;                   // globally unused variables marked ready
    std::vector<uint8_t> has_grad;                // W*P: accumulator holds a gradient (no_sync block)

    // ---- communication hook
    ddp_comm_hook_fn hook = nullptr;
    void* hook_state = nullptr;
    std::vector<void*> hook_rb;                   // W replica bucket buffers (empty: gradients are bucket views)
    bool hook_alias = false;                      // the hook reads the gradients in place
    int hook_builtin = 0;                         // 1: ddp_hook_mean, 2: ddp_hook_bf16_compress, 0: another hook
    bool opt_hook_fused = true;                   // built-in hooks run inside the fused bucket pass

    // ---- binding
    bool bound = false;
    std::vector<const void*> bind_grads;          // W*P, kept for rebuilds
    std::vector<const void*> bind_last;           // W*P last-step gradients (fused last micro-step), or empty
    std::vector<float*> bind_outs;                // n_out*P
    int W = 0;
    int n_out = 0;
    int device = -1;
    float* arena = nullptr;
    float inv_w = 1.0f;
    void* dev_table = nullptr;
    ddpk::SegTable tab{};
    std::vector<int32_t> bucket_seg;              // B+1 segment ranges
    std::vector<int64_t> seg_off_h;               // host copy of the segment offsets (S+1)
    std::vector<int32_t> seg_var;                 // first variable of each segment

    // ---- options and counters
    bool dry = false;
    bool pdl = true;
    int opt_ctas = 0;
    int opt_block = 0;              // 0: 128 threads for the bucket kernel, 256 for accumulate and hook copies
    // Defaults from the GB300 sweeps: the kernel is chosen per context from
    // the median bucket length (bulk-copy pipeline with 3 stages of 32 KiB
    // from 6 x 2^20 elements up, register streaming below).  Both kernels
    // launch more CTAs than fit at once (two or more resident waves for bulk
    // copy, three for register streaming): SMs that finish a slice early take
    // another, so a launch ends with a short tail and consecutive launches
    // interleave.  One kernel for all launches of a context, so consecutive
    // launches can overlap (one call per ready event, where every launch
    // waits, takes the bulk-copy kernel: see launch_range).
    int opt_kernel = ddpk::KERNEL_AUTO;
    int opt_stages = 3;
    int opt_stage_bytes = 32 * 1024;
    int opt_tma_ctas = 0;           // 0: resident waves sized by the launch (two by default)
    long long opt_auto_min = 6LL << 20;
    bool opt_chain = false;
    // Within one ddp_mark_ready_many call, consecutive released bucket runs
    // go out as one launch until it spans this many elements (0: one launch
    // per releasing event).  Every listed gradient is final when the call is
    // made, so a later launch start delays nothing that could overlap.
    // GB300, GPT-2-medium W=8 bf16, reverse order: per-gradient buckets
    // (292 launches) 6.92 -> 7.17 TB/s at 2^21, equal to 5 MiB buckets;
    // 1 MiB buckets 7.15 -> 7.17; 2^20 gains less, 2^22 and 2^23 the same.
    int64_t opt_coalesce = 1LL << 21;
    int64_t iter_launches = 0;      // launches issued in the current iteration
    void* iter_stream = nullptr;    // stream of the last of them
    int64_t call_launches = 0;      // launches issued by the current API call
    bool event_call = false;        // the current call is ddp_mark_ready or ddp_reduce_bucket
    ddpk::LaunchCfg cfg{};
    int acc_ctas = 1;
    int aux_block = 256;            // threads per CTA of the accumulate and hook copy kernels
    int64_t launches = 0;
    std::string err;
};

namespace {

int fail(ddp_ctx* c, int status, const std::string& msg) {
    if (c) c->err = msg;
    return status;
}

int cuda_fail(ddp_ctx* c, cudaError_t e, const char* where) {
    std::string m = std::string(where) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
    return fail(c, DDP_ERR_CUDA, m);
}

void reset_iteration(ddp_ctx* c) {
    c->pending.assign(c->B, 0);
    for (int32_t b = 0; b < c->B; ++b) c->pending[b] = static_cast<int32_t>(c->members[b].size());
    c->ready.assign(c->P, 0);
    c->next = 0;
}

void start_iteration(ddp_ctx* c) {
    reset_iteration(c);
    c->active = c->B > 0;
    c->iter_launches = 0;
    c->trace_cur.clear();
    c->iter_masked = false;
    c->unused_marked = false;
    if (c->pending_set) {
        // the local-use bits gathered since the last reduction serve this one
        c->iter_used.swap(c->pending_used);
        c->pending_used.assign(c->iter_used.size(), 0);
        c->pending_set = false;
        c->gused.assign(c->P, 0);
        for (int r = 0; r < c->W; ++r)
            for (int32_t v = 0; v < c->P; ++v) {
                const uint8_t u = c->iter_used[static_cast<size_t>(r) * c->P + v];
                c->gused[v] |= u;
                if (!u) c->iter_masked = true;
            }
    }
}

// Globally unused variables count as ready from the iteration's first event.
void mark_unused(ddp_ctx* c) {
    if (!c->iter_masked || c->unused_marked) return;
    c->unused_marked = true;
    for (int32_t v = 0; v < c->P; ++v)
        if (!c->gused[v] && !c->ready[v]) {
            c->ready[v] = 1;
            --c->pending[c->loc[v].bucket];
        }
}

// The iteration launched its last bucket: keep its ready order for a rebuild.
void finish_iteration(ddp_ctx* c) {
    c->active = false;
    c->trace_last = c->trace_cur;
}

// Layout from a walk over `order` (every variable once): append, close the
// bucket once its bytes reach the limit (first_cap for bucket 0, cap after).
void assign_layout(ddp_ctx* c, const int32_t* order, int64_t first_cap, int64_t cap) {
    c->members.clear();
    c->loc.assign(c->P, ddp_locator{-1, -1, 0, 0});
    std::vector<int32_t> cur;
    int64_t size = 0;
    for (int32_t i = 0; i < c->P; ++i) {
        const int32_t v = order[i];
        cur.push_back(v);
        size += c->numel[v] * c->elem;
        const int64_t limit = c->members.empty() ? first_cap : cap;
        if (size >= limit) {
            c->members.push_back(std::move(cur));
            cur.clear();
            size = 0;
        }
    }
    if (!cur.empty()) c->members.push_back(std::move(cur));
    c->B = static_cast<int32_t>(c->members.size());
    c->bucket_off.assign(c->B + 1, 0);
    for (int32_t b = 0; b < c->B; ++b) {
        int64_t off = 0;
        for (size_t i = 0; i < c->members[b].size(); ++i) {
            const int32_t v = c->members[b][i];
            c->loc[v] = ddp_locator{b, static_cast<int32_t>(i), off, c->numel[v]};
            off += c->numel[v];
        }
        c->bucket_off[b + 1] = c->bucket_off[b] + off;
    }
    c->cap = cap;
    c->first_cap = first_cap;
}

// Starts an iteration implicitly when the previous one has finished.
void ensure_started(ddp_ctx* c) {
    if (!c->active) start_iteration(c);
}

void free_binding(ddp_ctx* c) {
    if (c->dev_table) cudaFree(c->dev_table);
    c->dev_table = nullptr;
    c->tab = ddpk::SegTable{};
    c->bound = false;
}

int refresh_launch_cfg(ddp_ctx* c) {
    if (!c->bound || c->dry) return DDP_OK;
    int sms = 0;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, c->device);
    if (e != cudaSuccess) return cuda_fail(c, e, "cudaDeviceGetAttribute");
    const ddpk::InType in = c->dtype == DDP_F32 ? ddpk::IN_F32 : ddpk::IN_BF16;
    c->cfg.sms = sms;
    // GB300 sweeps of the register-streaming kernel: 128-thread CTAs beat 256
    // on small buckets (per-gradient and 1 MiB caps) and tie on large ones
    const int block = c->opt_block > 0 ? c->opt_block : 128;
    c->aux_block = c->opt_block > 0 ? c->opt_block : 256;
    c->cfg.block = block;
    c->cfg.pdl = c->pdl;
    // default grid: three resident waves (GB300, chained launches: GPT-2-medium
    // W=8 bf16 at cap 0 6.6 -> 7.0 TB/s against one wave)
    c->cfg.ctas_per_sm = c->opt_ctas > 0 ? c->opt_ctas
                                         : 3 * ddpk::reduce_max_ctas_per_sm(in, c->W, block, c->tab.add != 0);
    if (c->opt_kernel == ddpk::KERNEL_AUTO) {
        std::vector<int64_t> lens;
        for (int32_t b = 0; b < c->B; ++b) lens.push_back(c->bucket_off[b + 1] - c->bucket_off[b]);
        int64_t median = 0;
        if (!lens.empty()) {
            std::nth_element(lens.begin(), lens.begin() + lens.size() / 2, lens.end());
            median = lens[lens.size() / 2];
        }
        c->cfg.kernel = median >= c->opt_auto_min ? ddpk::KERNEL_TMA : ddpk::KERNEL_LDG;
    } else {
        c->cfg.kernel = c->opt_kernel;
    }
    c->cfg.stages = c->opt_stages;
    c->cfg.stage_bytes = c->opt_stage_bytes;
    c->cfg.tma_ctas_per_sm = c->opt_tma_ctas;
    c->cfg.tma_waves = 2;
    c->cfg.status = c->tab.status;

    c->acc_ctas = c->opt_ctas > 0 ? c->opt_ctas : ddpk::accumulate_max_ctas_per_sm(c->aux_block);
    return DDP_OK;
}

int check_device(ddp_ctx* c) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(c, e, "cudaGetDevice");
    if (dev != c->device)
        return fail(c, DDP_ERR_INVALID_ARG, "current CUDA device differs from the device the context was bound on");
    return DDP_OK;
}

// The hook path for buckets [b0, b1): per bucket, gather into the replica
// buffers, the hook, copy-back.
// Gradient as bucket view: replica r's gradients of bucket b lie at one base
// address plus each member's offset.  Fills base[r] (nullptr for a bucket
// without elements) and returns false when some member lies elsewhere.
bool bucket_view_bases(const ddp_ctx* c, int32_t b, const void** base) {
    for (int r = 0; r < c->W; ++r) {
        const char* b0 = nullptr;
        for (int32_t v : c->members[b]) {
            if (c->numel[v] == 0) continue;
            const char* g = static_cast<const char*>(c->bind_grads[static_cast<int64_t>(r) * c->P + v]);
            const char* at = g - c->loc[v].offset * c->elem;
            if (!b0) b0 = at;
            else if (at != b0) return false;
        }
        base[r] = b0;
    }
    return true;
}

int hook_range(ddp_ctx* c, int32_t b0, int32_t b1, const ddpk::LaunchCfg& launch_cfg, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    ddpk::LaunchCfg cfg = launch_cfg;
    cfg.block = c->aux_block;
    std::vector<const void*> reps(c->W);
    std::vector<int64_t> offs, lens;
    for (int32_t b = b0; b < b1; ++b) {
        const long long lo = c->bucket_off[b], hi = c->bucket_off[b + 1];
        const int s0 = c->bucket_seg[b], s1 = c->bucket_seg[b + 1];
        long long n = 0;
        if (c->hook_alias) {
            // the replicas' buckets are their gradients: nothing to gather
            if (!bucket_view_bases(c, b, reps.data()))
                return fail(c, DDP_ERR_INVALID_ARG, "bucket " + std::to_string(b) +
                                                        ": the bound gradients are not views of the bucket layout");
        } else {
            cudaError_t e = ddpk::launch_seg_copy(c->tab, 0, c->elem, c->W, c->n_out, c->arena, c->hook_rb.data(), lo,
                                                  hi, s0, s1, cfg, st, &n);
            c->launches += n;
            if (e != cudaSuccess) return cuda_fail(c, e, "hook gather launch");
            for (int r = 0; r < c->W; ++r)
                reps[r] = static_cast<const char*>(c->hook_rb[r]) + lo * c->elem;
        }
        const auto& vs = c->members[b];
        offs.resize(vs.size());
        lens.resize(vs.size());
        for (size_t i = 0; i < vs.size(); ++i) {
            offs[i] = c->loc[vs[i]].offset;
            lens[i] = c->loc[vs[i]].length;
        }
        ddp_grad_bucket gb;
        gb.index = b;
        gb.num_buckets = c->B;
        gb.is_last = b == c->B - 1;
        gb.W = c->W;
        gb.dtype = c->dtype;
        gb.n_vars = static_cast<int32_t>(vs.size());
        gb.numel = hi - lo;
        gb.replicas = reps.data();
        gb.result = c->arena + lo;
        gb.variables = vs.data();
        gb.offsets = offs.data();
        gb.lengths = lens.data();
        const int hr = c->hook(c->hook_state, &gb, stream);
        if (hr != 0) return fail(c, DDP_ERR_HOOK, "communication hook returned " + std::to_string(hr) + " for bucket " +
                                                      std::to_string(b));
        n = 0;
        const cudaError_t e =
            ddpk::launch_seg_copy(c->tab, 1, 4, c->W, c->n_out, c->arena, nullptr, lo, hi, s0, s1, cfg, st, &n);
        c->launches += n;
        if (e != cudaSuccess) return cuda_fail(c, e, "hook copy-back launch");
    }
    c->iter_launches += 1;
    c->iter_stream = stream;
    return DDP_OK;
}

// One kernel launch over buckets [b0, b1); tma_waves > 0 overrides the
// bulk-copy kernel's default number of resident waves.
int launch_range(ddp_ctx* c, int32_t b0, int32_t b1, void* stream, int tma_waves = 0) {
    if (c->dry || b1 <= b0) return DDP_OK;
    const long long lo = c->bucket_off[b0], hi = c->bucket_off[b1];
    const int s0 = c->bucket_seg[b0], s1 = c->bucket_seg[b1];
    if (hi <= lo || s1 <= s0) return DDP_OK;     // only zero-length tensors
    int st = check_device(c);
    if (st != DDP_OK) return st;
    const ddpk::InType in = c->dtype == DDP_F32 ? ddpk::IN_F32 : ddpk::IN_BF16;
    ddpk::LaunchCfg cfg = c->cfg;
    // One replica reads a third of what it writes (bucket and copy-back), and
    // its bulk-copy launches do best as one resident wave of long slices
    // (GB300, BERT-large shapes, one mark_ready_many call: 6,779 against 6,475
    // GB/s with two waves; one CTA per SM 6,574).
    if (tma_waves > 0) cfg.tma_waves = tma_waves;
    else if (c->W == 1) cfg.tma_waves = 1;
    // the iteration's final launch has no successor to overlap its tail
    cfg.last = b1 == c->B ? 1 : 0;
    // Chained launches: a launch that directly follows this iteration's
    // previous launch on the same stream need not wait for it when nothing
    // else can sit between them -- always within one API call (the call
    // enqueues only its own launches), across calls only when the caller
    // opted in (DDP_OPT_CHAINED).
    const bool follows_own = c->iter_launches > 0 && stream == c->iter_stream;
    cfg.chain = c->pdl && follows_own && (c->call_launches > 0 || c->opt_chain) ? 1 : 0;
    // One call per ready event (ddp_mark_ready, ddp_reduce_bucket), calls not
    // chained: every launch of the iteration waits for the preceding grid,
    // and with the automatic choice they all take the bulk-copy kernel, whose
    // CTAs ask L2 for their first stages during the wait (the register-
    // streaming kernel does not).  GB300, GPT-2-medium W=8 bf16, one
    // mark_ready call per event: caps 0 / 1 / 5 MiB +10.8 / +5.3 / +3.6 %
    // against register streaming; Linear(10,10) W=2 (one launch) equal.
    // Batched calls keep the context's kernel for every launch: a bulk-copy
    // first launch followed by chained register-streaming launches cost
    // GPT-2-medium at cap 0 17 % (7.14 -> 5.94 TB/s).
    if (c->opt_kernel == ddpk::KERNEL_AUTO && c->event_call && !c->opt_chain) cfg.kernel = ddpk::KERNEL_TMA;
    // The bulk-copy ring holds two stages of at least 16 bytes per stream
    // (one per replica, two with a bound last step) in the 227 KiB of shared
    // memory a CTA can have; past that the automatic choice streams through
    // registers (an explicit bulk-copy choice fails the launch).
    constexpr int64_t kTmaMaxStreams = (227 * 1024 - 128) / (2 * 16);
    if (c->opt_kernel == ddpk::KERNEL_AUTO && static_cast<int64_t>(c->W) * (c->tab.add ? 2 : 1) > kTmaMaxStreams)
        cfg.kernel = ddpk::KERNEL_LDG;
    // A built-in hook's arithmetic is the fused pass's (the default hook) or
    // the fused pass with every replica value rounded to bf16 first (the
    // compression hook): it runs inside the one-pass kernel, with nothing
    // gathered into the replica buffers and no separate copy-back.
    const bool fused_hook = c->hook && c->hook_builtin != 0 && c->opt_hook_fused;
    if (c->hook && !fused_hook) return hook_range(c, b0, b1, cfg, stream);
    cfg.compress = fused_hook && c->hook_builtin == 2 && c->dtype == DDP_F32 ? 1 : 0;
    if (!c->iter_masked) {
        long long n = 0;
        cudaError_t e = ddpk::launch_reduce(c->tab, in, c->W, c->n_out, c->arena, lo, hi, s0, s1, c->inv_w,
                                            cfg, static_cast<cudaStream_t>(stream), &n);
        c->launches += n;
        c->iter_launches += n;
        c->call_launches += n;
        c->iter_stream = stream;
        if (e != cudaSuccess) return cuda_fail(c, e, "bucket reduce launch");
        return DDP_OK;
    }
    // Unused parameters: the replicas' local-use masks travel in the launch's
    // parameter block, at most kMaxMaskSegs segments per launch.
    thread_local ddpk::SegMask mask;
    for (int sa = s0; sa < s1; sa += ddpk::kMaxMaskSegs) {
        const int sb = std::min(s1, sa + ddpk::kMaxMaskSegs);
        mask.n = sb - sa;
        for (int sg = sa; sg < sb; ++sg) {
            const int32_t v = c->seg_var[sg];
            unsigned long long bits = 0;
            for (int r = 0; r < c->W; ++r)
                if (c->iter_used[static_cast<size_t>(r) * c->P + v]) bits |= 1ull << r;
            mask.bits[sg - sa] = bits;
        }
        if (sa > s0) cfg.chain = c->pdl ? 1 : 0;   // follows this call's previous launch
        long long n = 0;
        cudaError_t e = ddpk::launch_reduce(c->tab, in, c->W, c->n_out, c->arena, c->seg_off_h[sa],
                                            c->seg_off_h[sb], sa, sb, c->inv_w, cfg,
                                            static_cast<cudaStream_t>(stream), &n, &mask);
        c->launches += n;
        c->iter_launches += n;
        c->call_launches += n;
        c->iter_stream = stream;
        if (e != cudaSuccess) return cuda_fail(c, e, "bucket reduce launch (unused parameters)");
    }
    return DDP_OK;
}

// In-order release starting at the cursor: one launch for the whole run of
// consecutive complete buckets.
int release(ddp_ctx* c, int32_t* launched, int32_t* n_launched, void* stream) {
    const int32_t first = c->next;
    while (c->next < c->B && c->pending[c->next] == 0) ++c->next;
    if (launched)
        for (int32_t b = first; b < c->next; ++b) launched[b - first] = b;
    if (n_launched) *n_launched = c->next - first;
    if (c->next == c->B) finish_iteration(c);
    return launch_range(c, first, c->next, stream);
}

bool is_aligned16(uintptr_t p) { return (p & 15u) == 0; }

}  // namespace

extern "C" {

const char* ddp_status_string(int status) {
    switch (status) {
        case DDP_OK: return "DDP_OK";
        case DDP_ERR_INVALID_ARG: return "DDP_ERR_INVALID_ARG";
        case DDP_ERR_ALREADY_READY: return "DDP_ERR_ALREADY_READY";
        case DDP_ERR_OUT_OF_ORDER: return "DDP_ERR_OUT_OF_ORDER";
        case DDP_ERR_PRIOR_REDUCTION_UNFINISHED:
            return "DDP_ERR_PRIOR_REDUCTION_UNFINISHED: Expected to have finished reduction in the prior "
                   "iteration before starting a new one";
        case DDP_ERR_NOT_BOUND: return "DDP_ERR_NOT_BOUND";
        case DDP_ERR_CUDA: return "DDP_ERR_CUDA";
        case DDP_ERR_NO_MEMORY: return "DDP_ERR_NO_MEMORY";
        case DDP_ERR_HOOK: return "DDP_ERR_HOOK";
        default: return "unknown ddp status";
    }
}

const char* ddp_last_error(const ddp_ctx* ctx) {
    return ctx ? ctx->err.c_str() : g_build_error.c_str();
}

int ddp_build_buckets(const int64_t* numel, int32_t P, ddp_dtype grad_dtype, int64_t cap_bytes,
                      ddp_ctx** out) {
    g_build_error.clear();
    if (!out) { g_build_error = "out is NULL"; return DDP_ERR_INVALID_ARG; }
    *out = nullptr;
    if (P < 0 || (P > 0 && !numel)) { g_build_error = "bad P or numel"; return DDP_ERR_INVALID_ARG; }
    if (grad_dtype != DDP_F32 && grad_dtype != DDP_BF16) { g_build_error = "bad dtype"; return DDP_ERR_INVALID_ARG; }
    if (cap_bytes < 0) { g_build_error = "negative cap"; return DDP_ERR_INVALID_ARG; }
    for (int32_t v = 0; v < P; ++v)
        if (numel[v] < 0) { g_build_error = "negative numel at " + std::to_string(v); return DDP_ERR_INVALID_ARG; }

    ddp_ctx* c = new (std::nothrow) ddp_ctx();
    if (!c) { g_build_error = "out of host memory"; return DDP_ERR_NO_MEMORY; }
    try {
        c->P = P;
        c->dtype = grad_dtype;
        c->elem = grad_dtype == DDP_F32 ? 4 : 2;
        c->cap = cap_bytes;
        c->numel.assign(numel, numel + P);
        // Walk the parameters in reverse registration order; close a bucket
        // as soon as its byte size reaches the cap (tensors never split).
        std::vector<int32_t> order(P);
        for (int32_t i = 0; i < P; ++i) order[i] = P - 1 - i;
        assign_layout(c, order.data(), cap_bytes, cap_bytes);
        reset_iteration(c);
    } catch (const std::bad_alloc&) {
        delete c;
        g_build_error = "out of host memory";
        return DDP_ERR_NO_MEMORY;
    }
    *out = c;
    return DDP_OK;
}

int ddp_get_locators(const ddp_ctx* ctx, ddp_locator* out) {
    if (!ctx || (!out && ctx->P > 0)) return DDP_ERR_INVALID_ARG;
    std::copy(ctx->loc.begin(), ctx->loc.end(), out);
    return DDP_OK;
}

int ddp_get_bucket_info(const ddp_ctx* ctx, int32_t* B, int64_t* bucket_offsets) {
    if (!ctx || !B) return DDP_ERR_INVALID_ARG;
    *B = ctx->B;
    if (bucket_offsets) std::copy(ctx->bucket_off.begin(), ctx->bucket_off.end(), bucket_offsets);
    return DDP_OK;
}

}  // extern "C"

namespace {

// Build the segment table of the current layout for the given pointers and
// upload it (replacing any previous table).
// Consistency of the layout a table is built from, checked at every bind and
// rebuild (O(P + S)): every variable sits in exactly one bucket at the prefix
// sum of the earlier members' lengths, the buckets tile the arena, and the
// segments of each bucket tile exactly its non-empty range in order.
std::string layout_problem(const ddp_ctx* c, const std::vector<int64_t>& seg_off,
                           const std::vector<int64_t>& seg_len, const std::vector<int32_t>& bucket_seg) {
    std::vector<uint8_t> seen(c->P, 0);
    if (c->bucket_off.size() != static_cast<size_t>(c->B) + 1 || c->bucket_off[0] != 0) return "bucket offsets";
    for (int32_t b = 0; b < c->B; ++b) {
        int64_t off = 0;
        for (size_t i = 0; i < c->members[b].size(); ++i) {
            const int32_t v = c->members[b][i];
            if (v < 0 || v >= c->P || seen[v]) return "variable " + std::to_string(v) + " placed twice or out of range";
            seen[v] = 1;
            const ddp_locator& l = c->loc[v];
            if (l.bucket != b || l.intra != static_cast<int32_t>(i) || l.offset != off || l.length != c->numel[v])
                return "locator of variable " + std::to_string(v);
            off += c->numel[v];
        }
        if (c->bucket_off[b + 1] != c->bucket_off[b] + off) return "bucket " + std::to_string(b) + " length";
        int64_t at = c->bucket_off[b];   // segments tile [bucket_off[b], bucket_off[b+1]) in order
        for (int32_t sg = bucket_seg[b]; sg < bucket_seg[b + 1]; ++sg) {
            if (seg_off[sg] != at || seg_len[sg] <= 0) return "segment " + std::to_string(sg) + " of bucket " + std::to_string(b);
            at += seg_len[sg];
        }
        if (at != c->bucket_off[b + 1]) return "segments of bucket " + std::to_string(b) + " do not cover it";
    }
    for (int32_t v = 0; v < c->P; ++v)
        if (!seen[v]) return "variable " + std::to_string(v) + " in no bucket";
    if (bucket_seg[c->B] != static_cast<int32_t>(seg_len.size()) || seg_off.back() != c->bucket_off[c->B])
        return "segment table end";
    return "";
}

// last: W*P last-step gradients (fused last micro-step; fp32) or nullptr.
int build_table(ddp_ctx* c, int32_t W, const void* const* grads, const void* const* last, float* bucket_arena,
                float* const* grad_out, int32_t n_out) {
    const int64_t total = c->bucket_off[c->B];
    // source streams per segment: the W gradients, then the W last-step gradients
    const int NS = last ? 2 * W : W;
    auto source = [&](int q, int32_t v) -> const void* {
        return q < W ? grads[static_cast<int64_t>(q) * c->P + v] : last[static_cast<int64_t>(q - W) * c->P + v];
    };

    // Host segment table: merge consecutive members of a bucket whose
    // gradients (every replica) and outputs (every copy) are contiguous.
    std::vector<int64_t> seg_off;
    std::vector<const void*> seg_src;
    std::vector<float*> seg_dst;
    std::vector<int32_t> seg_vec;
    std::vector<int32_t> bucket_seg(c->B + 1, 0);
    std::vector<int64_t> seg_len;
    std::vector<int32_t> seg_var;
    try {
        for (int32_t b = 0; b < c->B; ++b) {
            bucket_seg[b] = static_cast<int32_t>(seg_off.size());
            for (int32_t v : c->members[b]) {
                const int64_t n = c->numel[v];
                if (n == 0) continue;
                const int64_t a0 = c->bucket_off[b] + c->loc[v].offset;
                for (int q = 0; q < NS; ++q)
                    if (!source(q, v))
                        return fail(c, DDP_ERR_INVALID_ARG,
                                    std::string(q < W ? "NULL gradient" : "NULL last-step gradient") + " for replica " +
                                        std::to_string(q % W) + " variable " + std::to_string(v));
                for (int o = 0; o < n_out; ++o)
                    if (!grad_out[static_cast<int64_t>(o) * c->P + v])
                        return fail(c, DDP_ERR_INVALID_ARG, "NULL output for copy " + std::to_string(o) +
                                                                " variable " + std::to_string(v));
                const size_t S = seg_off.size();
                // with unused parameters every segment is one variable (one mask each)
                bool merge = !c->opt_find_unused && static_cast<int32_t>(S) > bucket_seg[b];
                if (merge) {
                    const int64_t plen = seg_len[S - 1];
                    for (int q = 0; q < NS && merge; ++q) {
                        const char* prev = static_cast<const char*>(seg_src[(S - 1) * NS + q]);
                        merge = static_cast<const char*>(source(q, v)) == prev + plen * c->elem;
                    }
                    for (int o = 0; o < n_out && merge; ++o)
                        merge = grad_out[static_cast<int64_t>(o) * c->P + v] == seg_dst[(S - 1) * n_out + o] + plen;
                }
                if (merge) {
                    seg_len[S - 1] += n;
                    continue;
                }
                // 128-bit path: element a of the arena is 16-byte aligned when a is
                // a multiple of the vector width; require the same of every stream.
                bool vec = true;
                for (int q = 0; q < NS; ++q) {
                    const uintptr_t p = reinterpret_cast<uintptr_t>(source(q, v));
                    vec = vec && is_aligned16(p - static_cast<uintptr_t>(a0 * c->elem));
                }
                for (int o = 0; o < n_out; ++o) {
                    const uintptr_t p = reinterpret_cast<uintptr_t>(grad_out[static_cast<int64_t>(o) * c->P + v]);
                    vec = vec && is_aligned16(p - static_cast<uintptr_t>(a0 * 4));
                }
                seg_off.push_back(a0);
                seg_len.push_back(n);
                seg_var.push_back(v);
                for (int q = 0; q < NS; ++q) seg_src.push_back(source(q, v));
                for (int o = 0; o < n_out; ++o) seg_dst.push_back(grad_out[static_cast<int64_t>(o) * c->P + v]);
                seg_vec.push_back(vec ? 1 : 0);
            }
        }
        bucket_seg[c->B] = static_cast<int32_t>(seg_off.size());
        seg_off.push_back(total);
        const std::string bad = layout_problem(c, seg_off, seg_len, bucket_seg);
        if (!bad.empty()) return fail(c, DDP_ERR_INVALID_ARG, "internal layout check failed: " + bad);
    } catch (const std::bad_alloc&) {
        return fail(c, DDP_ERR_NO_MEMORY, "out of host memory");
    }

    if (c->dry) {   // dry run: the host-side state only, no device table
        free_binding(c);
        c->bucket_seg = std::move(bucket_seg);
        c->seg_off_h = seg_off;
        c->seg_var = std::move(seg_var);
        c->W = W;
        c->n_out = n_out;
        c->arena = bucket_arena;
        c->inv_w = 1.0f / static_cast<float>(W);
        c->bound = true;
        return DDP_OK;
    }

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(c, e, "cudaGetDevice");

    // One device block: offsets | source pointers | output pointers | flags.
    const size_t S = seg_vec.size();
    auto up16 = [](size_t x) { return (x + 15) / 16 * 16; };
    const size_t b_off = up16(seg_off.size() * sizeof(int64_t));
    const size_t b_src = up16(seg_src.size() * sizeof(void*));
    const size_t b_dst = up16(seg_dst.size() * sizeof(float*));
    const size_t b_vec = up16(std::max<size_t>(S, 1) * sizeof(int32_t));
    const size_t b_status = 16;
    const size_t bytes = b_off + b_src + b_dst + b_vec + b_status;
    std::vector<unsigned char> host(bytes, 0);
    std::memcpy(host.data(), seg_off.data(), seg_off.size() * sizeof(int64_t));
    if (!seg_src.empty()) std::memcpy(host.data() + b_off, seg_src.data(), seg_src.size() * sizeof(void*));
    if (!seg_dst.empty()) std::memcpy(host.data() + b_off + b_src, seg_dst.data(), seg_dst.size() * sizeof(float*));
    if (S) std::memcpy(host.data() + b_off + b_src + b_dst, seg_vec.data(), S * sizeof(int32_t));

    free_binding(c);
    void* d = nullptr;
    e = cudaMalloc(&d, bytes);
    if (e != cudaSuccess) return cuda_fail(c, e, "cudaMalloc(segment table)");
    // A copy from pageable memory may return before its DMA has landed, and
    // it is ordered only with the default stream, not with the caller's
    // (non-blocking) streams: wait for it here, so that any later launch on
    // any stream reads the whole table.
    e = cudaMemcpyAsync(d, host.data(), bytes, cudaMemcpyHostToDevice, nullptr);
    if (e == cudaSuccess) e = cudaStreamSynchronize(nullptr);
    if (e != cudaSuccess) {
        cudaFree(d);
        return cuda_fail(c, e, "upload of the segment table");
    }
    auto* base = static_cast<unsigned char*>(d);
    c->dev_table = d;
    c->tab.seg_off = reinterpret_cast<const long long*>(base);
    c->tab.seg_src = reinterpret_cast<const void* const*>(base + b_off);
    c->tab.seg_dst = reinterpret_cast<float* const*>(base + b_off + b_src);
    c->tab.seg_vec = reinterpret_cast<const int*>(base + b_off + b_src + b_dst);
    c->tab.status = reinterpret_cast<int*>(base + b_off + b_src + b_dst + b_vec);
    c->tab.add = last ? 1 : 0;
    c->bucket_seg = std::move(bucket_seg);
    c->seg_off_h = seg_off;
    c->seg_var = std::move(seg_var);
    c->W = W;
    c->n_out = n_out;
    c->arena = bucket_arena;
    c->device = dev;
    c->inv_w = 1.0f / static_cast<float>(W);   // correctly rounded fp32 quotient
    c->bound = true;
    return refresh_launch_cfg(c);
}

}  // namespace

extern "C" {

int ddp_bind(ddp_ctx* c, int32_t W, const void* const* grads, float* bucket_arena, float* const* grad_out,
             int32_t n_out) {
    if (!c) return DDP_ERR_INVALID_ARG;
    if (W < 1) return fail(c, DDP_ERR_INVALID_ARG, "W must be >= 1");
    if (n_out != 0 && n_out != 1 && n_out != W) return fail(c, DDP_ERR_INVALID_ARG, "n_out must be 0, 1 or W");
    if (c->P > 0 && !grads) return fail(c, DDP_ERR_INVALID_ARG, "grads is NULL");
    if (n_out > 0 && c->P > 0 && !grad_out) return fail(c, DDP_ERR_INVALID_ARG, "grad_out is NULL with n_out > 0");
    const int64_t total = c->bucket_off[c->B];
    if (total > 0 && !bucket_arena) return fail(c, DDP_ERR_INVALID_ARG, "bucket_arena is NULL");
    if (!is_aligned16(reinterpret_cast<uintptr_t>(bucket_arena)))
        return fail(c, DDP_ERR_INVALID_ARG, "bucket_arena must be 16-byte aligned");
    std::vector<const void*> g_copy;
    std::vector<float*> o_copy;
    try {
        g_copy.assign(grads, grads + static_cast<int64_t>(W) * c->P);
        if (n_out > 0) o_copy.assign(grad_out, grad_out + static_cast<int64_t>(n_out) * c->P);
    } catch (const std::bad_alloc&) {
        return fail(c, DDP_ERR_NO_MEMORY, "out of host memory");
    }
    if (c->opt_find_unused && W > 64)
        return fail(c, DDP_ERR_INVALID_ARG, "unused-parameter tracking supports W <= 64");
    const int st = build_table(c, W, g_copy.data(), nullptr, bucket_arena, o_copy.empty() ? nullptr : o_copy.data(),
                               n_out);
    if (st != DDP_OK) return st;
    c->bind_grads = std::move(g_copy);
    c->bind_last.clear();
    c->bind_outs = std::move(o_copy);
    c->pending_used.clear();
    c->pending_set = false;
    c->has_grad.clear();
    return DDP_OK;
}

int ddp_bind_last_step(ddp_ctx* c, const void* const* g_last) {
    if (!c) return DDP_ERR_INVALID_ARG;
    if (!c->bound) return fail(c, DDP_ERR_NOT_BOUND, "bind the accumulated gradients first");
    if (c->active) return fail(c, DDP_ERR_INVALID_ARG, "the last step changes between iterations only");
    std::vector<const void*> last;
    if (g_last) {
        if (c->dtype != DDP_F32) return fail(c, DDP_ERR_INVALID_ARG, "the fused last step needs fp32 gradients");
        if (c->hook) return fail(c, DDP_ERR_INVALID_ARG, "a bound last step does not combine with hooks");
        if (c->opt_find_unused)
            return fail(c, DDP_ERR_INVALID_ARG, "a bound last step does not combine with DDP_OPT_FIND_UNUSED");
        try {
            last.assign(g_last, g_last + static_cast<int64_t>(c->W) * c->P);
        } catch (const std::bad_alloc&) {
            return fail(c, DDP_ERR_NO_MEMORY, "out of host memory");
        }
    }
    const int st = build_table(c, c->W, c->bind_grads.data(), last.empty() ? nullptr : last.data(), c->arena,
                               c->bind_outs.empty() ? nullptr : c->bind_outs.data(), c->n_out);
    if (st != DDP_OK) return st;
    c->bind_last = std::move(last);
    return DDP_OK;
}

int ddp_register_comm_hook(ddp_ctx* c, ddp_comm_hook_fn hook, void* state, void* const* replica_buffers) {
    if (!c) return DDP_ERR_INVALID_ARG;
    if (!hook) return fail(c, DDP_ERR_INVALID_ARG, "hook is NULL");
    if (c->hook) return fail(c, DDP_ERR_INVALID_ARG, "a communication hook is registered already");
    if (!c->bound) return fail(c, DDP_ERR_NOT_BOUND, "register the hook after ddp_bind");
    if (c->launches > 0 || c->active) return fail(c, DDP_ERR_INVALID_ARG, "register the hook before the first launch");
    if (c->W > ddpk::kMaxHookReplicas) return fail(c, DDP_ERR_INVALID_ARG, "hooks support W <= 64");
    if (c->opt_find_unused) return fail(c, DDP_ERR_INVALID_ARG, "hooks do not combine with DDP_OPT_FIND_UNUSED");
    if (!c->bind_last.empty()) return fail(c, DDP_ERR_INVALID_ARG, "hooks do not combine with a bound last step");
    const bool alias = !replica_buffers;
    std::vector<void*> rb;
    if (alias) {
        // the gradients must already be views of the bucket layout
        std::vector<const void*> base(c->W);
        for (int32_t b = 0; b < c->B; ++b)
            if (!bucket_view_bases(c, b, base.data()))
                return fail(c, DDP_ERR_INVALID_ARG, "replica_buffers is NULL but bucket " + std::to_string(b) +
                                                        " is not laid out as a view of the bound gradients");
    } else {
        rb.assign(c->W, nullptr);
        for (int r = 0; r < c->W && c->bucket_off[c->B] > 0; ++r) {
            if (!replica_buffers[r] || !is_aligned16(reinterpret_cast<uintptr_t>(replica_buffers[r])))
                return fail(c, DDP_ERR_INVALID_ARG,
                            "replica buffer " + std::to_string(r) + " is NULL or not 16-byte aligned");
            rb[r] = replica_buffers[r];
        }
    }
    c->hook = hook;
    c->hook_state = state;
    c->hook_rb = std::move(rb);
    c->hook_alias = alias;
    c->hook_builtin = hook == &ddp_hook_mean ? 1 : hook == &ddp_hook_bf16_compress ? 2 : 0;
    return DDP_OK;
}

namespace {
int builtin_mean(const ddp_grad_bucket* b, void* stream, int compress) {
    if (!b || b->W < 1 || b->W > ddpk::kMaxHookReplicas) return 1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 2;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 2;
    const ddpk::InType in = b->dtype == DDP_F32 ? ddpk::IN_F32 : ddpk::IN_BF16;
    const cudaError_t e = ddpk::launch_flat_mean(in, b->W, b->replicas, b->result, b->numel,
                                                 1.0f / static_cast<float>(b->W), compress, sms,
                                                 static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? 0 : 3;
}
}  // namespace

int ddp_hook_mean(void* state, const ddp_grad_bucket* bucket, void* stream) {
    (void)state;
    return builtin_mean(bucket, stream, 0);
}

int ddp_hook_bf16_compress(void* state, const ddp_grad_bucket* bucket, void* stream) {
    (void)state;
    return builtin_mean(bucket, stream, 1);
}

int ddp_get_ready_trace(const ddp_ctx* c, int32_t* order, int32_t* n) {
    if (!c || !n) return DDP_ERR_INVALID_ARG;
    *n = static_cast<int32_t>(c->trace_last.size());
    if (order) std::copy(c->trace_last.begin(), c->trace_last.end(), order);
    return DDP_OK;
}

int ddp_rebuild_buckets(ddp_ctx* c, const int32_t* order, int64_t first_cap_bytes, int64_t cap_bytes) {
    if (!c) return DDP_ERR_INVALID_ARG;
    if (c->active) return fail(c, DDP_ERR_INVALID_ARG, "rebuild inside an unfinished iteration");
    if (first_cap_bytes < 0 || cap_bytes < 0) return fail(c, DDP_ERR_INVALID_ARG, "negative cap");
    std::vector<int32_t> ord;
    try {
        if (order) ord.assign(order, order + c->P);
        else ord = c->trace_last;
    } catch (const std::bad_alloc&) {
        return fail(c, DDP_ERR_NO_MEMORY, "out of host memory");
    }
    if (static_cast<int32_t>(ord.size()) != c->P)
        return fail(c, DDP_ERR_INVALID_ARG, "the order must list every variable once (no complete recorded iteration)");
    std::vector<uint8_t> seen(c->P, 0);
    for (int32_t v : ord) {
        if (v < 0 || v >= c->P || seen[v]) return fail(c, DDP_ERR_INVALID_ARG, "the order is not a permutation");
        seen[v] = 1;
    }
    try {
        assign_layout(c, ord.data(), first_cap_bytes, cap_bytes);
    } catch (const std::bad_alloc&) {
        return fail(c, DDP_ERR_NO_MEMORY, "out of host memory");
    }
    reset_iteration(c);
    c->active = false;
    if (!c->bound) return DDP_OK;
    return build_table(c, c->W, c->bind_grads.data(), c->bind_last.empty() ? nullptr : c->bind_last.data(), c->arena,
                       c->bind_outs.empty() ? nullptr : c->bind_outs.data(), c->n_out);
}

int ddp_begin_iteration(ddp_ctx* c) {
    if (!c) return DDP_ERR_INVALID_ARG;
    if (c->active)
        return fail(c, DDP_ERR_PRIOR_REDUCTION_UNFINISHED,
                    "Expected to have finished reduction in the prior iteration before starting a new one: "
                    "bucket " + std::to_string(c->next) + " of " + std::to_string(c->B) + " never launched");
    start_iteration(c);
    return DDP_OK;
}

int ddp_abort_iteration(ddp_ctx* c) {
    if (!c) return DDP_ERR_INVALID_ARG;
    reset_iteration(c);
    c->active = false;
    return DDP_OK;
}

int ddp_mark_ready(ddp_ctx* c, int32_t var, int32_t* launched, int32_t* n_launched, void* stream) {
    if (!c) return DDP_ERR_INVALID_ARG;
    c->call_launches = 0;
    c->event_call = true;
    if (n_launched) *n_launched = 0;
    if (var < 0 || var >= c->P) return fail(c, DDP_ERR_INVALID_ARG, "variable index out of range");
    if (!c->dry && !c->bound) return fail(c, DDP_ERR_NOT_BOUND, "mark_ready before bind");
    ensure_started(c);
    if (c->ready[var] || (c->iter_masked && !c->gused[var]))
        return fail(c, DDP_ERR_ALREADY_READY, "variable " + std::to_string(var) + " already ready");
    mark_unused(c);
    c->ready[var] = 1;
    c->trace_cur.push_back(var);
    --c->pending[c->loc[var].bucket];
    if (c->next < c->B && c->pending[c->next] == 0) return release(c, launched, n_launched, stream);
    return DDP_OK;
}

int ddp_mark_ready_many(ddp_ctx* c, const int32_t* vars, int32_t n, int32_t* n_done, void* stream) {
    if (!c) return DDP_ERR_INVALID_ARG;
    if (n_done) *n_done = 0;
    if (n < 0 || (n > 0 && !vars)) return fail(c, DDP_ERR_INVALID_ARG, "bad event list");
    if (!c->dry && !c->bound) return fail(c, DDP_ERR_NOT_BOUND, "mark_ready_many before bind");
    c->call_launches = 0;
    c->event_call = false;
    // Released buckets [pend0, pend1) not launched yet: the runs released by
    // consecutive events of this call are adjacent (the cursor only moves
    // forward), so they merge into one launch (DDP_OPT_COALESCE_ELEMS).
    int32_t pend0 = -1, pend1 = -1;
    auto flush = [&]() -> int {
        if (pend0 < 0) return DDP_OK;
        const int st = launch_range(c, pend0, pend1, stream);
        pend0 = pend1 = -1;
        return st;
    };
    // an error at event i leaves events 0 .. i-1 applied: their buckets go out first
    auto stop = [&](int status, const std::string& msg) -> int {
        const int st = flush();
        return st != DDP_OK ? st : fail(c, status, msg);
    };
    for (int32_t i = 0; i < n; ++i) {
        const int32_t var = vars[i];
        if (var < 0 || var >= c->P) return stop(DDP_ERR_INVALID_ARG, "variable index out of range at event " + std::to_string(i));
        ensure_started(c);
        if (c->ready[var] || (c->iter_masked && !c->gused[var]))
            return stop(DDP_ERR_ALREADY_READY, "variable " + std::to_string(var) + " already ready at event " + std::to_string(i));
        mark_unused(c);
        c->ready[var] = 1;
        c->trace_cur.push_back(var);
        --c->pending[c->loc[var].bucket];
        if (c->next < c->B && c->pending[c->next] == 0) {
            const int32_t first = c->next;
            while (c->next < c->B && c->pending[c->next] == 0) ++c->next;
            if (c->next == c->B) finish_iteration(c);
            if (pend0 < 0) pend0 = first;
            pend1 = c->next;
            if (c->opt_coalesce <= 0 || c->bucket_off[pend1] - c->bucket_off[pend0] >= c->opt_coalesce ||
                c->next == c->B) {
                const int st = flush();
                if (st != DDP_OK) return st;
            }
        }
        if (n_done) *n_done = i + 1;
    }
    return flush();
}

int ddp_reduce_bucket(ddp_ctx* c, int32_t bucket, void* stream) {
    if (!c) return DDP_ERR_INVALID_ARG;
    c->call_launches = 0;
    c->event_call = true;
    if (bucket < 0 || bucket >= c->B) return fail(c, DDP_ERR_INVALID_ARG, "bucket index out of range");
    if (!c->dry && !c->bound) return fail(c, DDP_ERR_NOT_BOUND, "reduce_bucket before bind");
    ensure_started(c);
    if (bucket != c->next)
        return fail(c, DDP_ERR_OUT_OF_ORDER, "bucket " + std::to_string(bucket) + " is not next (next is " +
                                                 std::to_string(c->next) + ")");
    mark_unused(c);
    for (int32_t v : c->members[bucket]) c->ready[v] = 1;
    c->pending[bucket] = 0;
    return release(c, nullptr, nullptr, stream);
}

int ddp_reduce_all(ddp_ctx* c, void* stream) {
    if (!c) return DDP_ERR_INVALID_ARG;
    c->call_launches = 0;
    c->event_call = false;
    if (!c->dry && !c->bound) return fail(c, DDP_ERR_NOT_BOUND, "reduce_all before bind");
    ensure_started(c);
    const int32_t first = c->next;
    for (int32_t b = first; b < c->B; ++b) {
        for (int32_t v : c->members[b]) c->ready[v] = 1;
        c->pending[b] = 0;
    }
    c->next = c->B;
    finish_iteration(c);
    // one launch over the whole remaining iteration: at least eight resident
    // waves of the bulk-copy kernel, more while every CTA keeps ten stages
    // (launch_reduce_tma), shorten its tail (two suit the shorter launches of
    // a readiness-driven iteration).  GB300, BERT-large W=4: 6,967 GB/s with
    // four waves, 7,012 with six, 7,041 with eight; ResNet-50 W=8 +0.2 %.
    return launch_range(c, first, c->B, stream, 8);
}

int ddp_get_progress(const ddp_ctx* c, int32_t* next_bucket, int32_t* parked, int32_t* n_parked) {
    if (!c) return DDP_ERR_INVALID_ARG;
    if (next_bucket) *next_bucket = c->next;
    int32_t n = 0;
    for (int32_t b = c->next; b < c->B; ++b)
        if (c->pending[b] == 0) {
            if (parked) parked[n] = b;
            ++n;
        }
    if (n_parked) *n_parked = n;
    return DDP_OK;
}

int ddp_accumulate_nosync_used(ddp_ctx* c, void* const* acc, const void* const* g, const uint8_t* used,
                               int32_t first_step, void* stream) {
    if (!c) return DDP_ERR_INVALID_ARG;
    if (c->dtype != DDP_F32) return fail(c, DDP_ERR_INVALID_ARG, "no_sync accumulation supports fp32 gradients only");
    if (!c->bound) return fail(c, DDP_ERR_NOT_BOUND, "accumulate_nosync before bind (W unknown)");
    if (c->P > 0 && (!acc || !g)) return fail(c, DDP_ERR_INVALID_ARG, "acc or g is NULL");
    if (used && !c->opt_find_unused)
        return fail(c, DDP_ERR_INVALID_ARG, "local-use bits need DDP_OPT_FIND_UNUSED");
    const size_t WP = static_cast<size_t>(c->W) * c->P;
    std::vector<ddpk::AccPair> pairs;
    std::vector<uint8_t> has;   // the block record after this step, committed once the step is accepted
    try {
        // A gradient field that is empty in this block takes the gradient;
        // a filled one adds it.  Without a block record every field counts
        // as filled after the first step.
        if (first_step || c->has_grad.size() != WP) has.assign(WP, first_step ? 0 : 1);
        else has = c->has_grad;
        pairs.reserve(WP);
        for (int r = 0; r < c->W; ++r)
            for (int32_t v = 0; v < c->P; ++v) {
                const size_t i = static_cast<size_t>(r) * c->P + v;
                if (used && !used[i]) continue;
                if (c->numel[v] == 0) {
                    has[i] = 1;
                    continue;
                }
                if (!acc[i] || !g[i])
                    return fail(c, DDP_ERR_INVALID_ARG, "NULL accumulator or gradient at replica " +
                                                            std::to_string(r) + " variable " + std::to_string(v));
                pairs.push_back(ddpk::AccPair{static_cast<const float*>(g[i]), static_cast<float*>(acc[i]),
                                              c->numel[v], has[i] ? 0 : 1});
                has[i] = 1;
            }
        if (c->opt_find_unused && c->pending_used.size() != WP) c->pending_used.assign(WP, 0);
    } catch (const std::bad_alloc&) {
        return fail(c, DDP_ERR_NO_MEMORY, "out of host memory");
    }
    if (!c->dry && !pairs.empty()) {
        const int st = check_device(c);
        if (st != DDP_OK) return st;
        ddpk::LaunchCfg cfg = c->cfg;
        cfg.ctas_per_sm = c->acc_ctas;
        cfg.block = c->aux_block;
        long long n = 0;
        const cudaError_t e = ddpk::launch_accumulate(pairs.data(), static_cast<int>(pairs.size()), cfg,
                                                      static_cast<cudaStream_t>(stream), &n);
        c->launches += n;
        if (e != cudaSuccess) return cuda_fail(c, e, "accumulate launch");
    }
    c->has_grad.swap(has);
    if (c->opt_find_unused) {   // the local-use bitmap accumulates until the next reduction
        for (size_t i = 0; i < WP; ++i) c->pending_used[i] |= used ? (used[i] ? 1 : 0) : 1;
        c->pending_set = true;
    }
    return DDP_OK;
}

int ddp_accumulate_nosync(ddp_ctx* c, void* const* acc, const void* const* g, int32_t first_step, void* stream) {
    return ddp_accumulate_nosync_used(c, acc, g, nullptr, first_step, stream);
}

int ddp_set_local_used(ddp_ctx* c, const uint8_t* used) {
    if (!c) return DDP_ERR_INVALID_ARG;
    if (!c->opt_find_unused) return fail(c, DDP_ERR_INVALID_ARG, "local-use bits need DDP_OPT_FIND_UNUSED");
    if (!c->bound) return fail(c, DDP_ERR_NOT_BOUND, "set_local_used before bind (W unknown)");
    if (c->W > 64) return fail(c, DDP_ERR_INVALID_ARG, "unused-parameter tracking supports W <= 64");
    const size_t WP = static_cast<size_t>(c->W) * c->P;
    try {
        if (c->pending_used.size() != WP) c->pending_used.assign(WP, 0);
    } catch (const std::bad_alloc&) {
        return fail(c, DDP_ERR_NO_MEMORY, "out of host memory");
    }
    for (size_t i = 0; i < WP; ++i) c->pending_used[i] |= used ? (used[i] ? 1 : 0) : 1;
    c->pending_set = true;
    return DDP_OK;
}

int ddp_set_option(ddp_ctx* c, int32_t option, int64_t value) {
    if (!c) return DDP_ERR_INVALID_ARG;
    switch (option) {
        case DDP_OPT_DRY_RUN: c->dry = value != 0; return DDP_OK;
        case DDP_OPT_CTAS_PER_SM:
            if (value < 0 || value > 64) return fail(c, DDP_ERR_INVALID_ARG, "ctas_per_sm out of range");
            c->opt_ctas = static_cast<int>(value);
            return refresh_launch_cfg(c);
        case DDP_OPT_PDL:
            c->pdl = value != 0;
            c->cfg.pdl = c->pdl;
            return DDP_OK;
        case DDP_OPT_AUTO_MIN_ELEMS:
            if (value < 0) return fail(c, DDP_ERR_INVALID_ARG, "auto threshold must be >= 0");
            c->opt_auto_min = value;
            return refresh_launch_cfg(c);
        case DDP_OPT_CHAINED:
            c->opt_chain = value != 0;
            return DDP_OK;
        case DDP_OPT_HOOK_FUSED:
            if (c->active) return fail(c, DDP_ERR_INVALID_ARG, "the hook route changes between iterations only");
            c->opt_hook_fused = value != 0;
            return DDP_OK;
        case DDP_OPT_COALESCE_ELEMS:
            if (value < 0) return fail(c, DDP_ERR_INVALID_ARG, "coalescing threshold must be >= 0");
            c->opt_coalesce = value;
            return DDP_OK;
        case DDP_OPT_QUERY_KERNEL:
            return fail(c, DDP_ERR_INVALID_ARG, "DDP_OPT_QUERY_KERNEL is read with ddp_get_option");
        case DDP_OPT_FIND_UNUSED: {
            if (c->active) return fail(c, DDP_ERR_INVALID_ARG, "find_unused changes between iterations only");
            if (value != 0 && c->hook)
                return fail(c, DDP_ERR_INVALID_ARG, "hooks do not combine with DDP_OPT_FIND_UNUSED");
            if (value != 0 && !c->bind_last.empty())
                return fail(c, DDP_ERR_INVALID_ARG, "a bound last step does not combine with DDP_OPT_FIND_UNUSED");
            const bool on = value != 0;
            if (on && c->bound && c->W > 64)
                return fail(c, DDP_ERR_INVALID_ARG, "unused-parameter tracking supports W <= 64");
            if (on == c->opt_find_unused) return DDP_OK;
            c->opt_find_unused = on;
            c->pending_used.clear();
            c->pending_set = false;
            c->has_grad.clear();
            if (!c->bound) return DDP_OK;   // a bound context gets an unmerged (or merged) table now
            return build_table(c, c->W, c->bind_grads.data(), nullptr, c->arena,
                               c->bind_outs.empty() ? nullptr : c->bind_outs.data(), c->n_out);
        }
        case DDP_OPT_KERNEL:
            if (value != ddpk::KERNEL_LDG && value != ddpk::KERNEL_TMA && value != ddpk::KERNEL_AUTO)
                return fail(c, DDP_ERR_INVALID_ARG, "kernel must be 0 (register streaming), 1 (bulk copy) or 2 (by size)");
            c->opt_kernel = static_cast<int>(value);
            return refresh_launch_cfg(c);
        case DDP_OPT_STAGES:
            if (value < 2 || value > 8) return fail(c, DDP_ERR_INVALID_ARG, "stages must be 2..8");
            c->opt_stages = static_cast<int>(value);
            return refresh_launch_cfg(c);
        case DDP_OPT_STAGE_BYTES:
            if (value < 4096 || value > 112 * 1024)
                return fail(c, DDP_ERR_INVALID_ARG, "stage bytes must be 4 KiB..112 KiB");
            c->opt_stage_bytes = static_cast<int>(value);
            return refresh_launch_cfg(c);
        case DDP_OPT_TMA_CTAS_PER_SM:
            if (value < 0 || value > 8)
                return fail(c, DDP_ERR_INVALID_ARG, "bulk-copy CTAs per SM must be 0 (resident waves sized by the launch) .. 8");
            c->opt_tma_ctas = static_cast<int>(value);
            return refresh_launch_cfg(c);
        case DDP_OPT_BLOCK_THREADS:
            if (value != 0 && value != 128 && value != 256)
                return fail(c, DDP_ERR_INVALID_ARG, "block threads must be 0 (automatic), 128 or 256");
            c->opt_block = static_cast<int>(value);
            return refresh_launch_cfg(c);
        default: return fail(c, DDP_ERR_INVALID_ARG, "unknown option");
    }
}

int ddp_get_device_status(ddp_ctx* c, int32_t* status) {
    if (!c || !status) return DDP_ERR_INVALID_ARG;
    *status = 0;
    if (!c->bound) return fail(c, DDP_ERR_NOT_BOUND, "device status before bind");
    int32_t v = 0;
    // every stream's launches, not only the default stream's, must be done
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&v, c->tab.status, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(c, e, "read device status");
    if (v != 0) {
        const int32_t zero = 0;   // landed before returning, like the table upload
        e = cudaMemcpyAsync(c->tab.status, &zero, sizeof(zero), cudaMemcpyHostToDevice, nullptr);
        if (e == cudaSuccess) e = cudaStreamSynchronize(nullptr);
        if (e != cudaSuccess) return cuda_fail(c, e, "clear device status");
    }
    *status = v;
    return DDP_OK;
}

int ddp_get_debug_record(ddp_ctx* c, int32_t* code, int64_t* index) {
    if (!c || !code || !index) return DDP_ERR_INVALID_ARG;
    *code = 0;
    *index = 0;
    if (!c->bound) return fail(c, DDP_ERR_NOT_BOUND, "debug record before bind");
    if (c->dry) return DDP_OK;
    int32_t words[4] = {0, 0, 0, 0};
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(words, c->tab.status, sizeof(words), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(c, e, "read debug record");
    if (words[1] != 0) {
        const int32_t zero[3] = {0, 0, 0};
        e = cudaMemcpyAsync(c->tab.status + 1, zero, sizeof(zero), cudaMemcpyHostToDevice, nullptr);
        if (e == cudaSuccess) e = cudaStreamSynchronize(nullptr);
        if (e != cudaSuccess) return cuda_fail(c, e, "clear debug record");
    }
    *code = words[1];
    int64_t idx = 0;
    std::memcpy(&idx, &words[2], sizeof(idx));
    *index = idx;
    return DDP_OK;
}

int ddp_selftest_bounded_wait(int64_t limit_cycles, int32_t* code) {
    if (!code) return DDP_ERR_INVALID_ARG;
    *code = 0;
    if (limit_cycles <= 0 || limit_cycles > 4000000000LL) return DDP_ERR_INVALID_ARG;
    int* d = nullptr;
    cudaError_t e = cudaMalloc(&d, sizeof(int));
    if (e != cudaSuccess) return DDP_ERR_CUDA;
    e = cudaMemset(d, 0, sizeof(int));
    if (e == cudaSuccess) e = ddpk::launch_wait_selftest(limit_cycles, d, nullptr);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    int32_t v = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&v, d, sizeof(v), cudaMemcpyDeviceToHost);
    cudaFree(d);
    if (e != cudaSuccess) return DDP_ERR_CUDA;
    *code = v;
    return DDP_OK;
}

int ddp_get_option(const ddp_ctx* c, int32_t option, int64_t* value) {
    if (!c || !value) return DDP_ERR_INVALID_ARG;
    switch (option) {
        case DDP_OPT_DRY_RUN: *value = c->dry; return DDP_OK;
        case DDP_OPT_CTAS_PER_SM: *value = c->opt_ctas; return DDP_OK;
        case DDP_OPT_PDL: *value = c->pdl; return DDP_OK;
        case DDP_OPT_BLOCK_THREADS: *value = c->opt_block; return DDP_OK;
        case DDP_OPT_KERNEL: *value = c->opt_kernel; return DDP_OK;
        case DDP_OPT_STAGES: *value = c->opt_stages; return DDP_OK;
        case DDP_OPT_STAGE_BYTES: *value = c->opt_stage_bytes; return DDP_OK;
        case DDP_OPT_TMA_CTAS_PER_SM: *value = c->opt_tma_ctas; return DDP_OK;
        case DDP_OPT_AUTO_MIN_ELEMS: *value = c->opt_auto_min; return DDP_OK;
        case DDP_OPT_CHAINED: *value = c->opt_chain; return DDP_OK;
        case DDP_OPT_QUERY_KERNEL: *value = c->bound ? c->cfg.kernel : -1; return DDP_OK;
        case DDP_OPT_FIND_UNUSED: *value = c->opt_find_unused; return DDP_OK;
        case DDP_OPT_HOOK_FUSED: *value = c->opt_hook_fused; return DDP_OK;
        case DDP_OPT_COALESCE_ELEMS: *value = c->opt_coalesce; return DDP_OK;
        default: return DDP_ERR_INVALID_ARG;
    }
}

int ddp_read_launch_trace(uint64_t* out, int32_t* grid, int64_t* seq) {
    long long n = -1;
    static_assert(sizeof(uint64_t) == sizeof(unsigned long long), "trace stamps are 64-bit");
    const cudaError_t e = ddpk::read_launch_trace(reinterpret_cast<unsigned long long*>(out), grid, &n);
    if (seq) *seq = n;
    return e == cudaSuccess ? DDP_OK : cuda_fail(nullptr, e, "launch trace");
}

int ddp_get_launch_count(const ddp_ctx* c, int64_t* launches) {
    if (!c || !launches) return DDP_ERR_INVALID_ARG;
    *launches = c->launches;
    return DDP_OK;
}

void ddp_destroy(ddp_ctx* c) {
    if (!c) return;
    free_binding(c);
    delete c;
}

}  // extern "C"

// ---------------------------------------------------------------- internal layout access
// Read-only view of a context's bucket layout for other translation units of
// the library (declared in ddp_layout.h).

#include "ddp_layout.h"

namespace ddp_internal {

Layout layout(const ddp_ctx* c) {
    Layout l;
    l.P = c->P;
    l.B = c->B;
    l.elem = c->elem;
    l.bf16 = c->dtype == DDP_BF16;
    l.numel = c->numel.data();
    l.loc = c->loc.data();
    l.bucket_off = c->bucket_off.data();
    l.members = &c->members;
    return l;
}

}  // namespace ddp_internal

namespace ddp_internal {

void set_error(ddp_ctx* c, const std::string& msg) {
    if (c) c->err = msg;
}

}  // namespace ddp_internal
