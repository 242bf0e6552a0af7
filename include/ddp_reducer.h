/*
 * ddp_reducer.h -- C ABI of the GB300 DDP Reducer gradient path.
 *
 * The library reproduces the gradient path of PyTorch DistributedDataParallel's
 * Reducer as described in "PyTorch Distributed: Experiences on Accelerating Data
 * Parallel Training" (Li et al., VLDB 2020), the "Distributed Data Parallel"
 * notes (section "Internal Design") and "NCCL 专家课程 30: DDP Reducer、Bucket 与
 * 计算通信重叠":
 *   - parameters are packed into flat gradient buckets at construction time;
 *   - during an iteration each ready gradient is copied into its bucket view
 *     and buckets are launched strictly in index order (early ones park);
 *   - every bucket is averaged over the W data-parallel replicas and the mean
 *     is copied back into the parameters' gradients;
 *   - under no_sync, gradients accumulate locally for several micro-steps.
 *
 * On one GPU the W replicas are W gradient sets resident in device memory, so
 * the cross-replica reduction is arithmetic in a kernel, not communication.
 *
 * Conventions for every entry point
 *   - Every call returns a status (enum ddp_status); nothing aborts or throws
 *     across the ABI.  ddp_last_error() gives a one-line detail.
 *   - Device pointers are plain CUDA device addresses owned by the caller;
 *     "host array" arguments are host memory read during the call only.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Kernels run asynchronously on it; results are ordered in that stream only.
 *   - A context is not thread-safe: one thread drives it at a time.
 *   - Element offsets and lengths are in elements, not bytes.
 */
#ifndef DDP_REDUCER_H
#define DDP_REDUCER_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ddp_ctx ddp_ctx;

/* Gradient element type.  Buckets and copied-back gradients are always fp32;
 * bf16 gradients are widened exactly and summed in fp32. */
typedef enum ddp_dtype { DDP_F32 = 0, DDP_BF16 = 1 } ddp_dtype;

/* Where variable v lives: bucket index, position in the bucket's push order,
 * and the [offset, offset + length) element range inside the flat bucket
 * ("NCCL 专家课程 30", section "Variable 到 Bucket"). */
typedef struct ddp_locator {
    int32_t bucket;
    int32_t intra;
    int64_t offset;
    int64_t length;
} ddp_locator;

enum ddp_status {
    DDP_OK = 0,
    DDP_ERR_INVALID_ARG = -1,                 /* bad index, size, pointer, alignment */
    DDP_ERR_ALREADY_READY = -2,               /* variable reported twice in one iteration */
    DDP_ERR_OUT_OF_ORDER = -3,                /* explicit launch of a bucket that is not next */
    DDP_ERR_PRIOR_REDUCTION_UNFINISHED = -4,  /* previous iteration left buckets unlaunched */
    DDP_ERR_NOT_BOUND = -5,                   /* launch requested before ddp_bind */
    DDP_ERR_CUDA = -6,                        /* a CUDA runtime call failed */
    DDP_ERR_NO_MEMORY = -7,                   /* host or library-owned device allocation failed */
    DDP_ERR_HOOK = -8                         /* a communication hook returned nonzero */
};

/* ---------------------------------------------------------------- construction */

/* Assign P parameters to buckets ("PyTorch Distributed", Section 3.2.2 bucketing;
 * "NCCL 专家课程 30", section "`bucket_cap_mb` 不是张量切分器").
 * Walk v = P-1 .. 0 (reverse registration order), append v to the open bucket,
 * add numel[v] * sizeof(grad_dtype) bytes; close the bucket once its size is
 * >= cap_bytes; a non-empty remainder closes last.  Tensors are never split, so
 * a bucket may exceed the cap; cap_bytes = 0 gives one bucket per tensor.
 *   numel      host array [P] of element counts (>= 0; 0 joins the open bucket)
 *   P          >= 0 (P = 0 gives zero buckets)
 *   cap_bytes  >= 0 (bucket_cap_mb * 2^20)
 *   out        receives a new context (host memory only; no CUDA call is made)
 * Errors: INVALID_ARG (negative sizes, NULL out, bad dtype), NO_MEMORY. */
int ddp_build_buckets(const int64_t* numel, int32_t P, ddp_dtype grad_dtype,
                      int64_t cap_bytes, ddp_ctx** out);

/* Copy the locator table into out[P] (host array). */
int ddp_get_locators(const ddp_ctx* ctx, ddp_locator* out);

/* Number of buckets, and optionally the bucket arena layout: bucket b occupies
 * elements [bucket_offsets[b], bucket_offsets[b+1]) of the flat fp32 arena
 * (buckets back to back in index order, no padding).  bucket_offsets is a host
 * array of B+1 entries or NULL. */
int ddp_get_bucket_info(const ddp_ctx* ctx, int32_t* B, int64_t* bucket_offsets);

/* Bind the W replicas' gradients and the outputs.
 *   grads        host array [W*P]: grads[r*P + v] = device address of replica r's
 *                gradient of v (numel[v] elements of grad_dtype, contiguous);
 *                may be NULL for numel[v] == 0
 *   bucket_arena device fp32 array of bucket_offsets[B] elements, 16-byte aligned;
 *                receives every reduced bucket (the GradBucket buffer)
 *   grad_out     host array [n_out*P] of device fp32 addresses, or NULL when
 *                n_out == 0: grad_out[o*P + v] receives the mean gradient of v
 *                (the copy-back).  n_out = 0 is gradient_as_bucket_view: the
 *                caller uses arena views as the gradients and nothing is
 *                copied back; n_out = 1 writes one shared copy; n_out = W
 *                writes every replica's copy.
 * Builds the device segment table (library-owned, freed by ddp_destroy or the
 * next bind).  Synchronous.  Pointers must stay valid while bound.  Any W >= 1
 * reduces; the bulk-copy kernel holds up to 7,260 streams (W, or 2W with a
 * bound last step), so with more the automatic kernel choice streams through
 * registers and an explicit bulk-copy choice fails its launches (CUDA).
 * Errors: INVALID_ARG (W < 1, NULL pointers, misaligned arena, n_out not in
 * {0, 1, W}), CUDA, NO_MEMORY. */
int ddp_bind(ddp_ctx* ctx, int32_t W, const void* const* grads, float* bucket_arena,
             float* const* grad_out, int32_t n_out);

/* ---------------------------------------------------------------- iteration */

/* Start an iteration: every bucket pending = member count, cursor = 0.
 * Fails with PRIOR_REDUCTION_UNFINISHED if the previous iteration did not launch
 * every bucket ("Distributed Data Parallel" notes, "When a parameter never
 * receives a gradient"); the context is left unchanged -- call
 * ddp_abort_iteration to discard it.  The launch calls below start an iteration
 * implicitly when the previous one finished. */
int ddp_begin_iteration(ddp_ctx* ctx);

/* Discard an unfinished iteration (nothing is launched); local-use bits the
 * iteration took at its start (ddp_set_local_used) are dropped with it.
 * Buckets already launched by it stay launched (their results are in the
 * arena and outputs). */
int ddp_abort_iteration(ddp_ctx* ctx);

/* Variable `var`'s gradient is final ("NCCL 专家课程 30", section "Autograd Hook
 * 状态机" / "Bucket 必须按序发起"): --pending of its bucket; at zero the bucket
 * is ready; if it is the next to launch, it and every following bucket already
 * ready go out in index order, as ONE kernel launch over that bucket range on
 * `stream` (gather of the W replicas' gradients, fp32 mean, bucket write and
 * copy-back); otherwise it parks.
 *   launched    host array [B] or NULL: receives the launched bucket indices
 *   n_launched  receives their count (may be NULL)
 * Errors: INVALID_ARG (var out of range), ALREADY_READY, NOT_BOUND, CUDA.  On
 * ALREADY_READY the state is unchanged. */
int ddp_mark_ready(ddp_ctx* ctx, int32_t var, int32_t* launched, int32_t* n_launched,
                   void* stream);

/* A batch of ready events, processed in order exactly as that many
 * ddp_mark_ready calls would be (an autograd engine reports its hooks one by
 * one; a batch serves callers that know the order up front, like the one-GPU
 * emulation whose replicas' gradients are all resident).  The gradients of
 * every listed variable must be final on `stream` when the call is made.
 * Launches after the first one of the call follow it directly on the stream
 * (nothing else can be enqueued in between), so they start without waiting
 * for it and wait only before exiting.  Consecutive bucket runs released by
 * the call's events merge into one launch until it spans DDP_OPT_COALESCE_ELEMS
 * elements (the state and the results are those of one launch per event).
 *   vars    host array [n] of variable indices
 *   n_done  receives the number of events processed (all of them on success;
 *           on error, the failing event's index; earlier events stay applied
 *           and their released buckets are launched before the call returns)
 * Errors: as ddp_mark_ready. */
int ddp_mark_ready_many(ddp_ctx* ctx, const int32_t* vars, int32_t n, int32_t* n_done, void* stream);

/* Explicit launch of bucket `bucket`, which must be the next one (else
 * OUT_OF_ORDER): its members count as ready, it is launched, and any parked
 * buckets right after it follow in the same launch. */
int ddp_reduce_bucket(ddp_ctx* ctx, int32_t bucket, void* stream);

/* Launch every bucket not yet launched in this iteration, in index order, as one
 * kernel launch over their whole range (its CTAs each walk their slice of the
 * segment table); the iteration is then finished. */
int ddp_reduce_all(ddp_ctx* ctx, void* stream);

/* Cursor and parked set: *next_bucket = index of the next bucket to launch
 * (B when all are out); parked (host array [B] or NULL) receives the ready but
 * unlaunched buckets, *n_parked their count. */
int ddp_get_progress(const ddp_ctx* ctx, int32_t* next_bucket, int32_t* parked,
                     int32_t* n_parked);

/* ---------------------------------------------------------------- unused parameters */

/* Local-use bits of the replicas (find_unused_parameters; "Distributed Data
 * Parallel" notes, "Forward pass"; "PyTorch Distributed" summary, the
 * globally-unused bitmap).  used: host array [W*P], used[r*P+v] != 0 when
 * replica r's backward produces a gradient for v (NULL = all used).  The bits
 * are OR-ed into the bitmap that the next reduction uses (the bitmap also
 * collects the no_sync micro-steps' bits, see ddp_accumulate_nosync_used) and
 * that reduction then:
 *   - counts a replica without the gradient as a zero-filled slice (+0.0 in
 *     the rank-order sum; the mean is still over all W replicas);
 *   - marks every variable used on no replica ready at its first event
 *     (first mark_ready / explicit launch), before that event, so its bucket
 *     can launch; reporting such a variable is DDP_ERR_ALREADY_READY;
 *   - leaves the copy-back of such a variable untouched (its bucket slice
 *     receives the reduced zeros).
 * Needs DDP_OPT_FIND_UNUSED and a bound context.  Errors: INVALID_ARG,
 * NOT_BOUND, NO_MEMORY. */
int ddp_set_local_used(ddp_ctx* ctx, const uint8_t* used);

/* ddp_accumulate_nosync with the micro-step's local-use bits (host array
 * [W*P] or NULL = all used).  An unused (r, v) leaves acc untouched; a used
 * one takes g when its field is still empty in this no_sync block
 * (first_step != 0 starts a block: every field empty) and adds g otherwise.
 * With DDP_OPT_FIND_UNUSED the bits are OR-ed into the bitmap of the next
 * reduction ("PyTorch Distributed" summary, the conflict between no_sync and
 * unused-parameter marking).  Non-NULL bits need DDP_OPT_FIND_UNUSED. */
int ddp_accumulate_nosync_used(ddp_ctx* ctx, void* const* acc, const void* const* g, const uint8_t* used,
                               int32_t first_step, void* stream);

/* ---------------------------------------------------------------- communication hooks */

/* One ready bucket as a hook sees it ("Distributed Data Parallel" notes,
 * "Custom gradient aggregation"; "NCCL 专家课程 30", section "从 Bucket 到
 * AllReduce Future": index, bucket count, flat buffer, per-parameter views).
 * Host arrays are valid during the hook call only. */
typedef struct ddp_grad_bucket {
    int32_t index;                 /* bucket index */
    int32_t num_buckets;
    int32_t is_last;               /* index == num_buckets - 1 */
    int32_t W;                     /* replicas */
    int32_t dtype;                 /* ddp_dtype of the replica buffers */
    int32_t n_vars;
    int64_t numel;                 /* elements in the bucket */
    const void* const* replicas;   /* host [W] of device pointers: replica r's gradients of this bucket, gathered
                                      into the bucket layout (numel elements of dtype) */
    float* result;                 /* device fp32 [numel]: the hook writes the reduced bucket here (the arena slice) */
    const int32_t* variables;      /* host [n_vars]: the bucket's variables in push order */
    const int64_t* offsets;        /* host [n_vars]: element offset of each variable in the bucket */
    const int64_t* lengths;        /* host [n_vars]: element count of each variable */
} ddp_grad_bucket;

/* A hook enqueues its reduction on `stream` and returns 0 (nonzero aborts the
 * launch with DDP_ERR_HOOK).  It owns the averaging: the result is what the
 * parameters' gradients receive. */
typedef int (*ddp_comm_hook_fn)(void* state, const ddp_grad_bucket* bucket, void* stream);

/* Replace the fused bucket pass by: gather (each replica's gradients copied
 * into its bucket buffer), hook, copy-back (the result into the gradient
 * outputs), per launched bucket in index order.  Register once, after
 * ddp_bind and before the first launch.
 *   replica_buffers  host array [W] of device pointers, caller-owned, each 16-byte
 *                    aligned with room for bucket_offsets[B] elements of the
 *                    gradient dtype (bucket b of replica r lives at
 *                    replica_buffers[r] + bucket_offsets[b]);
 *                    or NULL when the bound gradients are views of the bucket
 *                    layout ("Distributed Data Parallel" notes,
 *                    gradient_as_bucket_view): every member v of bucket b of
 *                    replica r at one base address + its locator offset.  Then
 *                    nothing is gathered, the hook's replica pointers are those
 *                    bases (the gradients themselves; NULL for a bucket without
 *                    elements), and a launch whose bound gradients no longer
 *                    form such views fails with INVALID_ARG.
 * W <= 64; not with DDP_OPT_FIND_UNUSED or a bound last step.  The two
 * built-in hooks below keep the fused pass instead (DDP_OPT_HOOK_FUSED): the
 * buffers are then left as they are, and the view check is not made.
 * Errors: INVALID_ARG, NOT_BOUND. */
int ddp_register_comm_hook(ddp_ctx* ctx, ddp_comm_hook_fn hook, void* state, void* const* replica_buffers);

/* Built-in hooks (state unused): the default, the rank-order fp32 mean of the
 * replicas' buffers x fl32(1/W) -- the fused pass's arithmetic -- and a
 * compression variant that first rounds every replica value to bf16 (round to
 * nearest even), i.e. averages what a bf16 wire would carry.  Registered on a
 * context, they are not called per bucket: with DDP_OPT_HOOK_FUSED (default)
 * their arithmetic runs inside the fused bucket pass, which reads the bound
 * gradients where they lie, so the replica buffers are neither needed nor
 * written and the result equals the gather, hook, copy-back route bit for
 * bit.  Called directly, they launch their mean on `stream` as any hook. */
int ddp_hook_mean(void* state, const ddp_grad_bucket* bucket, void* stream);
int ddp_hook_bf16_compress(void* state, const ddp_grad_bucket* bucket, void* stream);

/* ---------------------------------------------------------------- rebuild */

/* The ready events of the last finished iteration, in order (the hooks'
 * record of the actual gradient-ready order; "NCCL 专家课程 30", section
 * "第一次迭代为何不同").  order: host array [P] or NULL; *n receives the count
 * (P when every variable reported through ddp_mark_ready/_many; fewer when
 * buckets went out through explicit launches). */
int ddp_get_ready_trace(const ddp_ctx* ctx, int32_t* order, int32_t* n);

/* Re-pack the buckets in a recorded ready order (same source): walk `order`
 * (host array [P], every variable once; NULL = the last finished iteration's
 * trace), append whole tensors, close a bucket once its bytes reach
 * first_cap_bytes (bucket 0) or cap_bytes (every later bucket).  Call between
 * iterations.  Locators, bucket count and arena layout change (the arena size
 * does not); a bound context keeps its pointers and gets a new device segment
 * table (synchronous).
 * Errors: INVALID_ARG (inside an iteration, not a permutation, no complete
 * trace, negative caps), CUDA, NO_MEMORY. */
int ddp_rebuild_buckets(ddp_ctx* ctx, const int32_t* order, int64_t first_cap_bytes, int64_t cap_bytes);

/* ---------------------------------------------------------------- no_sync */

/* One local accumulation micro-step for all W replicas ("PyTorch Distributed",
 * Section 3.2.4; "Distributed Data Parallel" notes, "Gradient sync you can turn
 * off"): acc[r*P+v] = g[r*P+v] when first_step != 0, else
 * acc[r*P+v] = fl32(acc[r*P+v] + g[r*P+v]).  fp32 only; W is the bound W.
 *   acc, g  host arrays [W*P] of device fp32 addresses (numel[v] elements each)
 * No bucket copy and no reduction happens; the accumulated gradients are reduced
 * by a later iteration whose bound grads are the accumulators.
 * Errors: INVALID_ARG (bf16 context, NULL pointers), NOT_BOUND, CUDA. */
int ddp_accumulate_nosync(ddp_ctx* ctx, void* const* acc, const void* const* g,
                          int32_t first_step, void* stream);

/* The synchronizing micro-step that ends a no_sync block, fused into the bucket
 * pass ("PyTorch Distributed", Section 3.2.4: the first backward after the
 * block accumulates its gradient into the same fields and then reduces them).
 * With g_last bound, every reduction of this context (ddp_mark_ready,
 * ddp_mark_ready_many, ddp_reduce_bucket, ddp_reduce_all) takes replica r's
 * input for variable v as fl32(grads[r*P+v] + g_last[r*P+v]), formed per
 * replica before the rank-order sum: the result equals ddp_accumulate_nosync
 * (first_step = 0) followed by the reduction, bit for bit, while each operand
 * is read once and the accumulated fields are not written.
 *   g_last  host array [W*P] of device fp32 addresses (numel[v] elements each;
 *           W = the bound W), copied; NULL unbinds it (reductions read the bound
 *           gradients alone again).  The caller owns the memory.
 * ddp_bind drops a bound last step.  Between iterations only.
 * Errors: INVALID_ARG (bf16 context, a NULL entry for a non-empty variable, a
 *         communication hook registered, DDP_OPT_FIND_UNUSED on, inside an
 *         unfinished iteration), NOT_BOUND, NO_MEMORY, CUDA. */
int ddp_bind_last_step(ddp_ctx* ctx, const void* const* g_last);

/* ---------------------------------------------------------------- no allocation */

/* The fused pass of ddp_reduce_all over every bucket, for callers that may not
 * allocate device memory: a framework whose caching allocator already owns the
 * device memory budget (a cudaMalloc beside it can fail or fragment what it
 * holds), and real-time loops where an allocation and the device
 * synchronisation it implies are not allowed.  The pages have no counterpart
 * of this call; it exists for such callers.
 *
 * It needs no ddp_bind: the caller passes the replicas' gradients and the
 * outputs exactly as ddp_bind takes them (grads [W*P], bucket_arena, grad_out
 * [n_out*P], n_out in {0, 1, W}), and the segment table that ddp_bind keeps in
 * cudaMalloc'd memory lives here in one file-scope static device array of
 * 256 KiB that every GPU which loads the library holds until the process
 * exits.  The context's binding and iteration state are neither used nor
 * changed.  No cudaMalloc, cudaFree or other allocating routine is called.
 *   - Limit: one table entry per non-empty parameter of
 *     8 + 8*W + 8*n_out + 4 bytes (plus 32 bytes); a layout that does not fit
 *     in 256 KiB is rejected with DDP_ERR_INVALID_ARG before anything runs.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture begins.
 *   - Every call copies its table into the shared array (the copy also zeroes
 *     the status word) and the array keeps the last call's contents; calls
 *     whose work can overlap on the GPU (other streams, other host threads)
 *     race on it.  Calls on one stream are ordered and safe.
 *   - Launch shape: always the bulk-copy kernel with 3 stages of 32 KiB and
 *     one CTA per SM; the context's launch options (ddp_set_option) are not
 *     used.  W is at most 7,260 (the ring's streams); more fail with CUDA.
 *   - The status word of the kernel's bounded waits lives in the shared array
 *     and is not reported: ddp_get_device_status reads a bound context's own
 *     word, not this one.
 * Errors: INVALID_ARG, CUDA. */
int ddp_reduce_all_noalloc(ddp_ctx* ctx, int32_t W, const void* const* grads, float* bucket_arena,
                           float* const* grad_out, int32_t n_out, void* stream);

/* ---------------------------------------------------------------- ranks that each hold some of the replicas */

/* Ownership plan of the bucket all-reduce split across G ranks ("PyTorch
 * Distributed Training Internals", section "3. The All-Reduce Itself": a
 * reduce-scatter, in which every rank ends up owning the reduced values of one
 * contiguous chunk of the bucket's flat range, then an all-gather of the
 * chunks; "NCCL 专家课程 30", section "Bucket 必须按序发起": every rank issues
 * the buckets' collectives in bucket-index order).  For a range of n elements
 * every chunk has *chunk = ceil(n / G) elements rounded up to a multiple of 8
 * (16-byte aligned chunk starts for fp32 and bf16); rank g owns
 * [*lo, *hi) = [min(n, g * chunk), min(n, (g + 1) * chunk)), so the chunks
 * tile [0, n) in rank order and ranks past the last non-empty chunk own
 * nothing.  Pure host arithmetic; any pointer may be NULL.
 * Errors: INVALID_ARG (n < 0, G < 1, g outside [0, G)). */
int ddp_shard_range(int64_t n, int32_t G, int32_t g, int64_t* chunk, int64_t* lo, int64_t* hi);

/* The owner's step of that all-reduce: out[i] = fl32(1/G) x the fp32 sum, in
 * order c = 0 .. G-1 starting from chunks[0][i], of the widened values
 * chunks[c][i], i < n -- the one-GPU pass's arithmetic over G replicas, so
 * the sharded result equals it bit for bit when the reduce-scatter moves the
 * replicas' raw chunks (all-to-alls) instead of partial sums.  With Wl
 * replicas on each rank, G here is the number of replicas in all (ranks x
 * Wl) and chunks[c] is replica c in the one-GPU order.
 *   chunks  host array [G] of device pointers: replica c's n values of the
 *           owned chunk, in `dtype` (16-byte aligned for 128-bit loads; any
 *           alignment is correct)
 *   out     device fp32 [n]
 * Asynchronous on `stream`.  G <= 64.  Errors: INVALID_ARG, CUDA. */
int ddp_shard_mean(int32_t G, ddp_dtype dtype, const void* const* chunks, float* out, int64_t n, void* stream);

/* ---------------------------------------------------------------- options, info */

enum ddp_option {
    DDP_OPT_DRY_RUN = 0,          /* 1: run the state machine, launch nothing; ddp_bind records the
                                     pointers without a device table (host tests) */
    DDP_OPT_CTAS_PER_SM = 1,      /* register-streaming kernels: CTAs per SM; 0 (default) = three times the
                                     bucket kernel's occupancy maximum (three resident waves: SMs that finish
                                     a slice early take another) and one resident wave of the accumulate
                                     kernel */
    DDP_OPT_PDL = 2,              /* 1 (default): programmatic dependent launch */
    DDP_OPT_BLOCK_THREADS = 3,    /* threads per CTA of the register-streaming kernels: 128 or 256 for
                                     all of them, or 0 (default): 128 for the bucket kernel, 256 for
                                     the accumulate and hook copy kernels */
    DDP_OPT_KERNEL = 4,           /* 0: register-streaming kernel, 1: bulk-copy (TMA) pipeline,
                                     2 (default): per context, bulk copy when the median bucket has at
                                     least DDP_OPT_AUTO_MIN_ELEMS elements, register streaming below;
                                     the launches of ddp_mark_ready and ddp_reduce_bucket calls, which
                                     each wait for the preceding grid, take the bulk-copy kernel either
                                     way unless DDP_OPT_CHAINED is set */
    DDP_OPT_STAGES = 5,           /* bulk-copy kernel: ring depth, 2..8 (default 3); fewer when the
                                     stages would not fit in shared memory */
    DDP_OPT_STAGE_BYTES = 6,      /* bulk-copy kernel: bytes of one stage, all W tiles (default 32 KiB);
                                     raised to 4 KiB per tile for many streams (W > 8, or W > 4 with
                                     a bound last step) */
    DDP_OPT_TMA_CTAS_PER_SM = 7,  /* bulk-copy kernels: CTAs per SM, 1..8, or 0 (default): resident
                                     waves sized by the launch's slices -- two, or up to 64 while every
                                     CTA keeps ten stages of work; one for a single replica (W = 1); an
                                     iteration's final launch two to eight, as many as leave every CTA
                                     eight stages; the single launch of ddp_reduce_all eight to 64 */
    DDP_OPT_AUTO_MIN_ELEMS = 8,   /* kernel 2: median bucket length (elements) from which the bulk-copy
                                     kernel is used (default 6 x 2^20) */
    DDP_OPT_CHAINED = 9,          /* 1: chained launches (default 0).  The caller guarantees that every
                                     gradient of an iteration is final before its first launch and that
                                     nothing else is enqueued on the stream until its last launch (true
                                     when the replicas' gradients are resident before the iteration, not
                                     when backward kernels run between hooks).  Then a launch that follows
                                     the iteration's previous launch on the same stream starts at once and
                                     waits for it only before exiting; stream order still holds for any
                                     work after the iteration. */
    DDP_OPT_QUERY_KERNEL = 10,    /* read only (ddp_get_option): kernel the bound context chose at bind
                                     (every launch of ddp_mark_ready_many and ddp_reduce_all), 0 or 1;
                                     -1 before ddp_bind */
    DDP_OPT_FIND_UNUSED = 11,     /* 1: track unused parameters (find_unused_parameters; default 0):
                                     enables ddp_set_local_used and the local-use bits of
                                     ddp_accumulate_nosync_used; segments are never merged; W <= 64 */
    DDP_OPT_HOOK_FUSED = 12,      /* 1 (default): a registered built-in hook (ddp_hook_mean,
                                     ddp_hook_bf16_compress) runs inside the fused bucket pass -- one
                                     launch per released bucket range, nothing gathered into the replica
                                     buffers, no separate copy-back; 0: the gather, hook call and
                                     copy-back route of every other hook.  Between iterations only. */
    DDP_OPT_COALESCE_ELEMS = 13   /* ddp_mark_ready_many: consecutive bucket runs released by the events
                                     of one call go out as one launch until it spans at least this many
                                     elements (default 2^21; 0: one launch per releasing event); results,
                                     readiness state and hook order are unchanged, only launch boundaries
                                     move.  Every listed gradient is final when the call is made, so no
                                     launch is held back behind work it could overlap. */
};
int ddp_set_option(ddp_ctx* ctx, int32_t option, int64_t value);
int ddp_get_option(const ddp_ctx* ctx, int32_t option, int64_t* value);

/* Read and clear the device status word of a bound context (synchronous:
 * waits for the device).  0 = every bounded wait inside the kernels finished
 * normally; a nonzero code names a wait that gave up after its time limit
 * (the results of that launch are not to be trusted). */
int ddp_get_device_status(ddp_ctx* ctx, int32_t* status);

/* Read and clear the bounds-check record of a bound context (synchronous:
 * waits for the device).
 * Only a library built with -DDDP_DEBUG (libddpreducer_debug.so) checks, in
 * every kernel, that each range it walks lies inside its segment, launch and
 * stage and that every bulk copy is 16-byte aligned and sized; the first
 * failed check stores its code (101 segment range, 102 staged chunk range,
 * 103 bulk-copy alignment, 104 accumulate pair range) and the element index
 * there and the access is skipped.  A release build never writes the record:
 * *code = 0.  The pages have no counterpart (a stand-in for a sanitizer run).
 * Errors: INVALID_ARG, NOT_BOUND, CUDA. */
int ddp_get_debug_record(ddp_ctx* ctx, int32_t* code, int64_t* index);

/* Self-test of the kernels' bounded waits on the current device: one CTA
 * waits on an mbarrier that nothing completes, for at most limit_cycles SM
 * clock cycles (1 .. 4e9); the wait gives up, writes its timeout code into a
 * status word, and the kernel returns.  *code receives that word (3 when the
 * wait ended as designed).  Synchronous; allocates and frees 4 bytes.  The
 * pages have no counterpart.  Errors: INVALID_ARG (limit out of range), CUDA. */
int ddp_selftest_bounded_wait(int64_t limit_cycles, int32_t* code);

/* Launch trace of a library built with -DDDP_TRACE (libddpreducer_trace.so,
 * `python -m reduction_reducer_gb300.build --trace`): for the last
 * DDP_TRACE_LAUNCHES launches of the bulk-copy bucket kernel (all contexts of
 * the process), per CTA (the first DDP_TRACE_CTAS of each grid), four
 * %globaltimer stamps in ns: entry, past the wait for the preceding grid (a
 * chained launch: past its trigger), the consumers' first stage and their
 * last.  Launch number i (from 0) sits in slot i % DDP_TRACE_LAUNCHES.
 *   out   host array [DDP_TRACE_LAUNCHES * DDP_TRACE_CTAS * 4] or NULL
 *   grid  host array [DDP_TRACE_LAUNCHES] or NULL: CTAs of each slot's launch
 *   seq   receives the number of launches traced so far (-1: not a trace build)
 * Synchronous (waits for the device).  Diagnostics only; the pages have no
 * counterpart.  Errors: CUDA. */
#define DDP_TRACE_LAUNCHES 64
#define DDP_TRACE_CTAS 4096
int ddp_read_launch_trace(uint64_t* out, int32_t* grid, int64_t* seq);

/* Kernel launches issued by this context since creation. */
int ddp_get_launch_count(const ddp_ctx* ctx, int64_t* launches);

const char* ddp_status_string(int status);
/* Detail of the last failure on ctx (or of the last failed ddp_build_buckets in
 * this thread when ctx is NULL). */
const char* ddp_last_error(const ddp_ctx* ctx);

void ddp_destroy(ddp_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* DDP_REDUCER_H */
