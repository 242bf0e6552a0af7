"""GPU parity of the CUDA path against the CPU oracle, through the C ABI.

Every comparison is bitwise (0 ULP; NaN compared as a class): the kernels
use the oracle's summation order, so the tolerance the gradient path allows
for a tree order (2e-7 relative per element) is not needed.

* small and reduced workloads: every element of the bucket arena and of every
  copied-back gradient against the oracle, plus guard words around them;
* full-size workloads (BERT-large W=4 in every launch mode, including the
  bench's own configuration; GPT-2-medium W=8 bf16 at every cap; the no_sync
  ResNet-50 W=16 K=8 block): every element of the arena, of every copied-back
  gradient and of the accumulated fields against the oracle run on the same
  inputs, read back from the device buffers;
* one tensor of 2^31 + 37 elements (64-bit offsets, not a benchmark
  configuration): sampled elements, random positions plus the first and last
  40 elements of every parameter.
"""

import numpy as np
import pytest
import torch

from oracle.buckets import assign_buckets
from oracle.nosync import accumulate_steps
from oracle.reduce import reduce_buckets
from reduction_reducer_gb300 import InvalidArg, Reducer, _lib
from workloads import gen, shapes

from gpu_util import (bits_equal, check_every_element, first_mismatch, host_grads, host_to_device_views,
                      layout, nosync_full_size_check, run_path, sampled_check, to_host)

pytestmark = pytest.mark.gpu

DEV = "cuda"
GUARD = np.uint32(0x7FC0DEAD)      # a NaN payload no kernel writes
MIB = 1 << 20


@pytest.fixture(scope="module", autouse=True)
def _built():
    import os
    from reduction_reducer_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    _lib.load()
    torch.cuda.set_device(0)


def guarded(n, pad=64):
    """fp32 device buffer of n elements with `pad` guard words on each side
    (16-byte alignment preserved); returns (whole, view)."""
    whole = torch.from_numpy(np.full(n + 2 * pad, GUARD, np.uint32).view(np.float32)).to(DEV)
    return whole, whole[pad:pad + n]


def guards_intact(whole, pad, n):
    h = whole.cpu().numpy().view(np.uint32)
    return np.all(h[:pad] == GUARD) and np.all(h[pad + n:] == GUARD)


def make_order(kind, numel, members, seed=0):
    if kind == "reverse":
        return gen.reverse_order(len(numel))
    if kind == "straggler":
        return gen.straggler_order(members, p=0.5, seed=seed)
    if kind == "random":
        rng = np.random.default_rng(seed)
        return [int(v) for v in rng.permutation(len(numel))]
    raise ValueError(kind)


def set_kernel(red, kernel):
    """ldg | tma | auto (size-based choice) | chained (bulk copy + chained launches)."""
    if kernel == "chained":
        red.set_option(_lib.OPT_KERNEL, _lib.KERNEL_TMA)
        red.set_option(_lib.OPT_CHAINED, 1)
    elif kernel == "auto":
        red.set_option(_lib.OPT_KERNEL, _lib.KERNEL_AUTO)
        red.set_option(_lib.OPT_AUTO_MIN_ELEMS, 50_000)
    else:
        red.set_option(_lib.OPT_KERNEL, _lib.KERNEL_TMA if kernel == "tma" else _lib.KERNEL_LDG)


def full_compare(numel, W, dtype, cap, order="straggler", n_out=1, mode="mark_ready", odd=False,
                 special=False, stream=None, iterations=1, out_odd=False, kernel="ldg", options=None):
    elem = 4 if dtype == "f32" else 2
    flats, views, offs = host_grads(numel, W, dtype, odd=odd, special=special)
    members, locs = assign_buckets(numel, elem, cap)
    want_arena, want_outs = reduce_buckets(views, members, locs, numel, n_out=max(n_out, 1))
    flat_dev, grads_dev = host_to_device_views(flats, numel, offs, dtype, DEV)

    red = Reducer(numel, dtype, cap)
    set_kernel(red, kernel)
    for opt, value in (options or {}).items():
        red.set_option(opt, value)
    N = red.arena_numel()
    arena_whole, arena = guarded(N)
    out_offs, out_total = layout(numel, 64, out_odd)
    out_bufs, outs = [], []
    for o in range(n_out):
        whole, flat = guarded(out_total)
        out_bufs.append((whole, flat))
        outs.append([flat[off:off + n] for off, n in zip(out_offs, numel)])
    grad_out = None if n_out == 0 else (outs[0] if n_out == 1 else outs)
    ordr = make_order(order, numel, members)
    for _ in range(iterations):
        run_path(red, grads_dev, arena, grad_out, order=ordr, mode=mode, stream=stream)

    got = arena.cpu().numpy()
    assert bits_equal(got, want_arena), first_mismatch(got, want_arena)
    assert guards_intact(arena_whole, 64, N)
    covered = np.zeros(out_total, bool)
    for off, n in zip(out_offs, numel):
        covered[off:off + n] = True
    for o in range(n_out):
        whole, flat = out_bufs[o]
        host = flat.cpu().numpy()
        for v, (off, n) in enumerate(zip(out_offs, numel)):
            assert bits_equal(host[off:off + n], want_outs[0][v]), (o, v, first_mismatch(host[off:off + n], want_outs[0][v]))
        assert np.all(host.view(np.uint32)[~covered] == GUARD), "copy-back wrote outside the views"
        assert guards_intact(whole, 64, out_total)
    # the inputs are read only
    for r in range(W):
        back = flat_dev[r].view(torch.int16).cpu().numpy().view(np.uint16) if dtype == "bf16" else flat_dev[r].cpu().numpy()
        assert np.array_equal(back.view(np.uint8), flats[r].view(np.uint8))
    launches = red.launch_count()
    assert red.device_status() == 0
    red.destroy()
    return launches


# ---------------------------------------------------------------- the worked example

def test_linear_example_bitexact_and_full_batch():
    numel = shapes.numels(shapes.linear_10x10())
    ex = gen.linear_example(W=2, n=20, seed=0)
    members, locs = assign_buckets(numel, 4, 25 * MIB)
    want_arena, want_outs = reduce_buckets(ex["grads"], members, locs, numel)
    red = Reducer(numel, "f32", 25 * MIB)
    grads = [[torch.from_numpy(g).to(DEV) for g in ex["grads"][r]] for r in range(2)]
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    outs = [torch.full((n,), float("nan"), device=DEV) for n in numel]
    run_path(red, grads, arena, outs, order=[1, 0])
    assert bits_equal(arena.cpu().numpy(), want_arena)
    for v in range(2):
        assert bits_equal(outs[v].cpu().numpy(), want_outs[0][v])
    # and the mean is the full-batch gradient of the 40 x 10 batch (fp64)
    x = np.concatenate([xi.astype(np.float64) for xi in ex["x"]])
    out = x @ ex["weight"].astype(np.float64).T + ex["bias"].astype(np.float64)
    dw = (2.0 / out.size) * out.T @ x
    assert np.allclose(outs[0].cpu().numpy(), dw.reshape(-1), rtol=1e-4, atol=1e-7)


def test_replicas_identical_after_step():
    """Broadcast form (n_out = W): every replica receives the same bits and
    the SGD step keeps the replicas identical."""
    W = 4
    numel = shapes.numels(shapes.linear_10x10())
    ex = gen.linear_example(W=W, n=20, seed=0)
    red = Reducer(numel, "f32", 25 * MIB)
    grads = [[torch.from_numpy(g).to(DEV) for g in ex["grads"][r]] for r in range(W)]
    arena = torch.empty(red.arena_numel(), device=DEV)
    outs = [[torch.full((n,), float("nan"), device=DEV) for n in numel] for _ in range(W)]
    run_path(red, grads, arena, outs, order=[1, 0])
    params = [[torch.from_numpy(ex["weight"].reshape(-1).copy()).to(DEV), torch.from_numpy(ex["bias"].copy()).to(DEV)]
              for _ in range(W)]
    for r in range(W):
        for p, g in zip(params[r], outs[r]):
            p.sub_(0.001 * g)
    for r in range(1, W):
        for v in range(2):
            assert torch.equal(outs[r][v].view(torch.int32), outs[0][v].view(torch.int32))
            assert torch.equal(params[r][v].view(torch.int32), params[0][v].view(torch.int32))


# ---------------------------------------------------------------- ragged lists, every W

RAGGED = [0, 1, 2, 3, 5, 7, 8, 13, 64, 67, 100, 1000, 4095, 4097, 70001, 0, 9, 300007, 16, 31]


KERNELS = ["ldg", "tma", "auto", "chained"]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("W", [1, 2, 3, 4, 5, 8, 16])
def test_ragged_every_W(W, dtype, kernel):
    full_compare(RAGGED, W, dtype, cap=64 * 1024, order="straggler", n_out=1, kernel=kernel)


@pytest.mark.parametrize("kernel", ["ldg", "tma"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("W", [32, 64, 100, 256])
def test_many_replicas(W, dtype, kernel):
    """W beyond the compiled-in widths: the generic replica loop; from W = 100
    on, the bulk-copy ring no longer fits 4 KiB per stream and its tiles
    shrink (256 streams: 2 stages of 112-element tiles)."""
    numel = [3, 4097, 0, 70001, 16, 1000]
    full_compare(numel, W, dtype, cap=32 * 1024, order="random", n_out=1, kernel=kernel)


@pytest.mark.parametrize("mode", ["mark_ready", "mark_ready_many"])
def test_more_replicas_than_the_bulk_copy_ring_holds(mode):
    """7,300 replicas: more streams than the bulk-copy ring has room for
    (7,260).  The automatic kernel choice streams them through registers,
    bit for bit; an explicit bulk-copy choice fails its launch with a CUDA
    status before anything runs, and the device stays usable."""
    from reduction_reducer_gb300 import CudaError
    numel = [16, 5, 33]
    full_compare(numel, 7300, "f32", cap=1 << 20, order="random", n_out=1, mode=mode, kernel="auto")
    flats, views, offs = host_grads(numel, 7300, "f32")
    _, grads_dev = host_to_device_views(flats, numel, offs, "f32", DEV)
    red = Reducer(numel, "f32", 1 << 20)
    red.set_option(_lib.OPT_KERNEL, _lib.KERNEL_TMA)
    arena = torch.zeros(red.arena_numel(), device=DEV)
    red.bind(grads_dev, arena, None)
    red.begin_iteration()
    with pytest.raises(CudaError):
        red.mark_ready_many([2, 1, 0])
    red.destroy()
    full_compare(numel, 3, "f32", cap=1 << 20, order="random", n_out=1, kernel="tma")


# Launch shapes other than the defaults: ring depth and stage bytes (a 112 KiB
# stage leaves room for fewer stages and, at many streams, smaller tiles), two
# bulk-copy CTAs per SM, 256-thread register-streaming CTAs, a fixed number of
# CTAs per SM, and no programmatic dependent launch.  Each changes the tile,
# grid and slice arithmetic the kernels index with.
O = _lib
SHAPES = {
    "tma_2x4k": ("tma", {O.OPT_STAGES: 2, O.OPT_STAGE_BYTES: 4096}),
    "tma_8x16k": ("tma", {O.OPT_STAGES: 8, O.OPT_STAGE_BYTES: 16 * 1024}),
    "tma_3x112k": ("tma", {O.OPT_STAGES: 3, O.OPT_STAGE_BYTES: 112 * 1024}),
    "tma_4x32k_2cta": ("tma", {O.OPT_STAGES: 4, O.OPT_STAGE_BYTES: 32 * 1024, O.OPT_TMA_CTAS_PER_SM: 2}),
    "tma_nopdl": ("tma", {O.OPT_PDL: 0}),
    "chained_6x16k_2cta": ("chained", {O.OPT_STAGES: 6, O.OPT_STAGE_BYTES: 16 * 1024, O.OPT_TMA_CTAS_PER_SM: 2}),
    "ldg_256": ("ldg", {O.OPT_BLOCK_THREADS: 256}),
    "ldg_1cta": ("ldg", {O.OPT_CTAS_PER_SM: 1}),
    "ldg_256_3cta": ("ldg", {O.OPT_BLOCK_THREADS: 256, O.OPT_CTAS_PER_SM: 3}),
    "ldg_nopdl": ("ldg", {O.OPT_PDL: 0}),
}


@pytest.mark.parametrize("shape", list(SHAPES))
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("W,mode", [(3, "mark_ready_many"), (8, "mark_ready"), (16, "reduce_all")])
def test_launch_shapes(shape, dtype, W, mode):
    kernel, options = SHAPES[shape]
    full_compare(RAGGED, W, dtype, cap=64 * 1024, order="straggler", n_out=1, mode=mode, kernel=kernel,
                 options=options, odd=(W == 3))


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n_out", [0, 1, "W"])
def test_output_modes(dtype, n_out, kernel):
    W = 4
    full_compare(RAGGED, W, dtype, cap=32 * 1024, order="random", n_out=W if n_out == "W" else n_out,
                 kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("W", [2, 3, 8])
def test_misaligned_views(W, dtype, kernel):
    """Parameters at odd offsets of their buffers (no common 16-byte phase)
    take the scalar path; outputs at odd offsets too."""
    full_compare(RAGGED, W, dtype, cap=16 * 1024, order="straggler", odd=True, out_odd=True, kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_special_values(dtype, kernel):
    full_compare(RAGGED, 4, dtype, cap=64 * 1024, special=True, kernel=kernel)
    full_compare(RAGGED, 3, dtype, cap=64 * 1024, special=True, kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("W", [3, 4, 8])
def test_mark_ready_many(W, dtype, kernel):
    """A whole ready order in one call: launches after the first chain."""
    full_compare(RAGGED, W, dtype, cap=16 * 1024, order="straggler", mode="mark_ready_many", kernel=kernel,
                 iterations=2)
    full_compare(RAGGED, W, dtype, cap=0, order="random", mode="mark_ready_many", kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("mode", ["reduce_all", "reduce_bucket"])
def test_explicit_launch_modes(mode, kernel):
    full_compare(RAGGED, 8, "f32", cap=16 * 1024, mode=mode, kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_repeated_iterations_and_side_stream(kernel):
    s = torch.cuda.Stream()
    full_compare(RAGGED, 4, "f32", cap=16 * 1024, iterations=3, stream=s, kernel=kernel)


def test_cap_zero_per_gradient():
    n = full_compare(RAGGED, 4, "bf16", cap=0, order="reverse")
    # one launch per non-empty bucket: reverse order releases each at once
    assert n == sum(1 for x in RAGGED if x > 0)


def test_mixed_hooks_then_reduce_all():
    numel = RAGGED
    W = 4
    flats, views, offs = host_grads(numel, W, "f32")
    members, locs = assign_buckets(numel, 4, 16 * 1024)
    want_arena, want_outs = reduce_buckets(views, members, locs, numel)
    flat_dev, grads_dev = host_to_device_views(flats, numel, offs, "f32", DEV)
    red = Reducer(numel, "f32", 16 * 1024)
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    outs = [torch.full((n,), float("nan"), device=DEV) for n in numel]
    red.bind(grads_dev, arena, outs)
    red.begin_iteration()
    for v in gen.reverse_order(len(numel))[:7]:
        red.mark_ready(v)
    red.reduce_all()
    torch.cuda.synchronize()
    assert bits_equal(arena.cpu().numpy(), want_arena)
    for v in range(len(numel)):
        assert bits_equal(outs[v].cpu().numpy(), want_outs[0][v])


def test_bucket_order_contiguous_replicas_merge():
    """Replicas laid out in bucket order (gradient-as-bucket-view style):
    consecutive members merge into one segment per bucket."""
    numel = RAGGED
    W = 4
    members, locs = assign_buckets(numel, 4, 64 * 1024)
    lens = [sum(numel[v] for v in m) for m in members]
    starts = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    offs = [int(starts[locs[v].bucket] + locs[v].offset) for v in range(len(numel))]
    total = int(starts[-1])
    flats = [gen.draw_flat_np(total, r) for r in range(W)]
    views = [[f[o:o + n] for o, n in zip(offs, numel)] for f in flats]
    want_arena, _ = reduce_buckets(views, members, locs, numel)
    flat_dev, grads_dev = host_to_device_views(flats, numel, offs, "f32", DEV)
    red = Reducer(numel, "f32", 64 * 1024)
    arena = torch.full((total,), float("nan"), device=DEV)
    run_path(red, grads_dev, arena, None, mode="reduce_all")
    assert bits_equal(arena.cpu().numpy(), want_arena)


def test_bind_rejects_misaligned_arena():
    red = Reducer([8, 8], "f32", 1 << 20)
    g = [[torch.zeros(8, device=DEV), torch.zeros(8, device=DEV)]]
    buf = torch.zeros(20, device=DEV)
    with pytest.raises(InvalidArg):
        red.bind(g, buf[1:], None)


@pytest.mark.parametrize("mode", ["mark_ready", "mark_ready_many"])
@pytest.mark.parametrize("cap", [0, 1 << 20])
def test_many_small_parameters(cap, mode):
    """20,000 parameters of 0-40 elements: a segment table of ~19,500
    entries that every CTA searches; per-gradient buckets (cap 0: one bucket
    per parameter, one launch per event, or coalesced runs in one call) and
    1 MiB buckets."""
    rng = np.random.default_rng(20_000)
    numel = [int(x) for x in rng.integers(0, 41, size=20_000)]
    full_compare(numel, 4, "f32", cap=cap, order="random", n_out=1, mode=mode, kernel="auto")


def test_empty_and_zero_length_models():
    red = Reducer([], "f32", 25 * MIB)
    red.bind([[]], torch.zeros(4, device=DEV), None)
    red.reduce_all()
    assert red.launch_count() == 0
    red = Reducer([0, 0, 0], "f32", 0)
    z = torch.zeros(0, device=DEV)
    red.bind([[z, z, z], [z, z, z]], torch.zeros(4, device=DEV), [z, z, z])
    red.begin_iteration()
    for v in (2, 1, 0):
        red.mark_ready(v)
    torch.cuda.synchronize()
    assert red.launch_count() == 0


# ---------------------------------------------------------------- reduced workloads, every element

@pytest.mark.parametrize("kernel", KERNELS)
def test_resnet50_full_size_every_element(kernel):
    numel = shapes.numels(shapes.resnet50())
    full_compare(numel, 8, "f32", 25 * MIB, order="reverse", n_out=1, kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_bert_reduced_straggler_every_element(kernel):
    numel = shapes.numels(shapes.bert_large(layers=3, vocab=4096))
    full_compare(numel, 4, "f32", 2 * MIB, order="straggler", n_out=1, kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("cap_mib", [0, 1, 5, 25, 100])
def test_gpt2_reduced_caps_every_element(cap_mib, kernel):
    numel = shapes.numels(shapes.gpt2_medium(layers=2, vocab=3000, n_ctx=256))
    full_compare(numel, 8, "bf16", cap_mib * MIB, order="reverse", n_out=1, kernel=kernel)


@pytest.mark.parametrize("kernel", ["ldg", "tma"])
def test_nosync_small_every_element(kernel):
    numel = RAGGED
    W, K = 3, 4
    steps_np = [host_grads(numel, W, "f32", step=k)[1] for k in range(K)]
    offs = host_grads(numel, W, "f32", step=0)[2]
    acc_np = [accumulate_steps([steps_np[k][r] for k in range(K)]) for r in range(W)]
    members, locs = assign_buckets(numel, 4, 64 * 1024)
    want_arena, want_outs = reduce_buckets(acc_np, members, locs, numel)
    dev_steps = []
    for k in range(K):
        fl, _, _ = host_grads(numel, W, "f32", step=k)
        dev_steps.append(host_to_device_views(fl, numel, offs, "f32", DEV)[1])
    acc_dev = [[torch.full((n,), float("nan"), device=DEV) for n in numel] for _ in range(W)]
    red = Reducer(numel, "f32", 64 * 1024)
    set_kernel(red, kernel)
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    outs = [torch.full((n,), float("nan"), device=DEV) for n in numel]
    red.bind(acc_dev, arena, outs)
    for k in range(K):
        red.accumulate_nosync(acc_dev, dev_steps[k], first_step=(k == 0))
    red.begin_iteration()
    for v in gen.reverse_order(len(numel)):
        red.mark_ready(v)
    torch.cuda.synchronize()
    assert red.device_status() == 0
    for r in range(W):
        for v in range(len(numel)):
            assert bits_equal(acc_dev[r][v].cpu().numpy(), acc_np[r][v])
    assert bits_equal(arena.cpu().numpy(), want_arena)
    for v in range(len(numel)):
        assert bits_equal(outs[v].cpu().numpy(), want_outs[0][v])


# ---------------------------------------------------------------- full-size workloads, every element

def device_replicas(numel, W, dtype, step=0):
    offs, total = gen.packed_offsets(numel, 64)
    flat = [gen.draw_flat_torch(total, r, step, dtype, DEV) for r in range(W)]
    views = [[f[o:o + n] for o, n in zip(offs, numel)] for f in flat]
    return flat, views, offs


# The inputs of one full-size workload at a time (device buffers drawn by the
# seeded generator and their host copies), and the oracle's result for one
# bucket cap at a time: the tests of a workload run back to back and share
# them.  The kernels never write their inputs.
_FULL = {}


def full_size_inputs(name, numel, W, dtype):
    key = (name, W, dtype)
    if key not in _FULL:
        _FULL.clear()
        torch.cuda.empty_cache()
        flat, views, offs = device_replicas(numel, W, dtype)
        host = [to_host(f, dtype) for f in flat]
        _FULL[key] = {"flat": flat, "views": views, "offs": offs, "oracle": {},
                      "host": [[h[o:o + n] for o, n in zip(offs, numel)] for h in host]}
    return _FULL[key]


def oracle_result(inp, numel, dtype, cap):
    if cap not in inp["oracle"]:
        inp["oracle"].clear()
        members, locs = assign_buckets(numel, 4 if dtype == "f32" else 2, cap)
        inp["oracle"][cap] = reduce_buckets(inp["host"], members, locs, numel)
    return inp["oracle"][cap]


def full_size_run(name, numel, W, dtype, cap, order, mode="mark_ready", kernel="ldg"):
    """One iteration of a full-size workload through the C ABI, every element
    of the bucket arena and of the copied-back gradients against the oracle
    run on the same inputs (read back from the device buffers)."""
    inp = full_size_inputs(name, numel, W, dtype)
    red = Reducer(numel, dtype, cap)
    if kernel is not None:        # None: the library's defaults
        set_kernel(red, kernel)
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    out_offs, out_total = gen.packed_offsets(numel, 64)
    out_flat = torch.full((out_total,), float("nan"), device=DEV)
    outs = [out_flat[o:o + n] for o, n in zip(out_offs, numel)]
    run_path(red, inp["views"], arena, outs, order=order, mode=mode)
    assert red.device_status() == 0
    launches = red.launch_count()
    red.destroy()
    want_arena, want_outs = oracle_result(inp, numel, dtype, cap)
    check_every_element(numel, want_arena, want_outs, arena, out_flat, out_offs)
    return launches


def bert_order():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "bert_large_ready_order.txt")
    return [int(l) for l in open(path) if l.strip() and not l.startswith("#")]


@pytest.mark.parametrize("kernel", KERNELS)
def test_bert_large_full_size_every_element(kernel):
    numel = shapes.numels(shapes.bert_large())
    full_size_run("bert_large", numel, 4, "f32", 25 * MIB, bert_order(), kernel=kernel)


def test_bert_large_full_size_bench_configuration():
    """Exactly what bench.py times: library defaults, the stored straggler
    order reported in one mark_ready_many call, one copy-back."""
    numel = shapes.numels(shapes.bert_large())
    n = full_size_run("bert_large", numel, 4, "f32", 25 * MIB, bert_order(), mode="mark_ready_many", kernel=None)
    assert n == 35          # 37 buckets in 35 launches: two parked buckets go out with the ones that release them


@pytest.mark.parametrize("kernel", KERNELS)
def test_bert_large_full_size_reduce_all(kernel):
    numel = shapes.numels(shapes.bert_large())
    full_size_run("bert_large", numel, 4, "f32", 25 * MIB, None, mode="reduce_all", kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("cap_mib", [0, 1, 5, 25, 100])
def test_gpt2_medium_full_size_every_element(cap_mib, kernel):
    numel = shapes.numels(shapes.gpt2_medium())
    full_size_run("gpt2_medium", numel, 8, "bf16", cap_mib * MIB, gen.reverse_order(len(numel)), kernel=kernel,
                  mode="mark_ready_many")


def test_nosync_resnet50_full_size_every_element():
    _FULL.clear()
    numel = shapes.numels(shapes.resnet50())
    W, K = 16, 8
    steps = [device_replicas(numel, W, "f32", step=k) for k in range(K)]
    offs = steps[0][2]
    acc_flat = [torch.full_like(steps[0][0][r], float("nan")) for r in range(W)]
    acc = [[f[o:o + n] for o, n in zip(offs, numel)] for f in acc_flat]
    red = Reducer(numel, "f32", 25 * MIB)
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    out_flat = torch.full_like(steps[0][0][0], float("nan"))
    outs = [out_flat[o:o + n] for o, n in zip(offs, numel)]
    red.bind(acc, arena, outs)
    for k in range(K):
        red.accumulate_nosync(acc, steps[k][1], first_step=(k == 0))
    red.begin_iteration()
    red.mark_ready_many(gen.reverse_order(len(numel)))
    torch.cuda.synchronize()
    assert red.device_status() == 0
    red.destroy()
    nosync_full_size_check(numel, offs, [[f for f in s[0]] for s in steps], acc_flat, arena, out_flat, K, False)


@pytest.mark.parametrize("kernel", KERNELS)
def test_largest_tensor_64bit_offsets(kernel):
    """One tensor of 2^31 + 37 bf16 elements (past 32-bit indexing) behind a
    small one, W = 2: sampled check including both ends."""
    numel = [1000, (1 << 31) + 37]
    _FULL.clear()
    torch.cuda.empty_cache()
    flat, views, offs = device_replicas(numel, 2, "bf16")
    red = Reducer(numel, "bf16", 25 * MIB)
    set_kernel(red, kernel)
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    out_offs, out_total = gen.packed_offsets(numel, 64)
    out_flat = torch.full((out_total,), float("nan"), device=DEV)
    run_path(red, views, arena, [out_flat[o:o + n] for o, n in zip(out_offs, numel)], order=[1, 0])
    assert sampled_check(numel, "bf16", 2, 25 * MIB, flat, offs, arena, [(out_flat, out_offs)], 1) > 100_000
    assert not torch.isnan(arena).any(), "arena not fully written"
    assert red.device_status() == 0
    red.destroy()


def test_automatic_kernel_choice():
    """Default kernel choice per context: the bulk-copy pipeline when the
    median bucket has >= 2^20 elements (BERT-large, 25 MiB buckets), register
    streaming for per-gradient buckets (GPT-2-medium at cap 0)."""
    def chosen(numel, dtype, cap):
        red = Reducer(numel, dtype, cap)
        assert red.get_option(_lib.OPT_QUERY_KERNEL) == -1
        W = 2
        offs, total = gen.packed_offsets(numel, 64)
        flat = [torch.zeros(total, dtype=torch.float32 if dtype == "f32" else torch.bfloat16, device=DEV) for _ in range(W)]
        grads = [[f[o:o + n] for o, n in zip(offs, numel)] for f in flat]
        red.bind(grads, torch.empty(red.arena_numel(), device=DEV), None)
        k = red.get_option(_lib.OPT_QUERY_KERNEL)
        red.destroy()
        return k
    assert chosen(shapes.numels(shapes.bert_large()), "f32", 25 * MIB) == _lib.KERNEL_TMA
    assert chosen(shapes.numels(shapes.gpt2_medium()), "bf16", 0) == _lib.KERNEL_LDG


@pytest.mark.parametrize("kernel", ["ldg", "tma"])
def test_nosync_misaligned_and_special(kernel):
    """Accumulators and gradients at odd offsets (no 16-byte alignment) and
    special values: scalar paths, first step copies bits (incl. -0.0)."""
    numel = RAGGED
    W, K = 2, 3
    steps = [host_grads(numel, W, "f32", step=k, odd=True, special=True) for k in range(K)]
    offs = steps[0][2]
    acc_np = [accumulate_steps([steps[k][1][r] for k in range(K)]) for r in range(W)]
    dev_steps = [host_to_device_views(steps[k][0], numel, offs, "f32", DEV)[1] for k in range(K)]
    acc_off, acc_total = layout(numel, 64, odd=True)
    acc_flat = [torch.full((acc_total,), float("nan"), device=DEV) for _ in range(W)]
    acc_dev = [[f[o:o + n] for o, n in zip(acc_off, numel)] for f in acc_flat]
    red = Reducer(numel, "f32", 64 * 1024)
    set_kernel(red, kernel)
    red.bind(acc_dev, torch.empty(red.arena_numel() + 4, device=DEV), None)
    for k in range(K):
        red.accumulate_nosync(acc_dev, dev_steps[k], first_step=(k == 0))
    torch.cuda.synchronize()
    assert red.device_status() == 0
    for r in range(W):
        for v in range(len(numel)):
            assert bits_equal(acc_dev[r][v].cpu().numpy(), acc_np[r][v]), (r, v)


@pytest.mark.parametrize("kernel", KERNELS)
def test_rebuild_then_reduce(kernel):
    """Iteration 1 records the ready order; the buckets are re-packed from it
    with a smaller first bucket; iteration 2 must match the oracle on the
    rebuilt layout, bit for bit, through the same binding."""
    from oracle.rebuild import rebuild_buckets
    numel = shapes.numels(shapes.bert_large(layers=2, vocab=2048))
    W = 4
    flats, views, offs = host_grads(numel, W, "f32")
    flat_dev, grads_dev = host_to_device_views(flats, numel, offs, "f32", DEV)
    red = Reducer(numel, "f32", 4 * MIB)
    set_kernel(red, kernel)
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    outs = [torch.full((n,), float("nan"), device=DEV) for n in numel]
    rng = np.random.default_rng(5)
    order = [int(v) for v in rng.permutation(len(numel))]
    run_path(red, grads_dev, arena, outs, order=order, mode="mark_ready_many")
    assert red.get_ready_trace() == order
    red.rebuild_buckets(None, 1 * MIB, 4 * MIB)
    arena.fill_(float("nan"))
    red.begin_iteration()
    red.mark_ready_many(order)
    torch.cuda.synchronize()
    members, locs = rebuild_buckets(numel, 4, order, 1 * MIB, 4 * MIB)
    want_arena, want_outs = reduce_buckets(views, members, locs, numel)
    assert red.B == len(members)
    assert bits_equal(arena.cpu().numpy(), want_arena), first_mismatch(arena.cpu().numpy(), want_arena)
    for v in range(len(numel)):
        assert bits_equal(outs[v].cpu().numpy(), want_outs[0][v])
    assert red.device_status() == 0


@pytest.mark.parametrize("kernel", ["ldg", "tma"])
def test_iteration_captured_in_cuda_graph(kernel):
    """An iteration's launches (PDL-chained) captured into a CUDA graph and
    replayed on new gradient values in the same buffers: each replay matches
    the oracle on those values.  A warm-up iteration comes first, so the
    one-time kernel attribute calls happen outside the capture."""
    numel = RAGGED
    W, cap = 4, 8 * 1024
    flats, views, offs = host_grads(numel, W, "f32")
    flat_dev, grads_dev = host_to_device_views(flats, numel, offs, "f32", DEV)
    members, locs = assign_buckets(numel, 4, cap)
    order = gen.straggler_order(members, p=0.5, seed=2)
    red = Reducer(numel, "f32", cap)
    set_kernel(red, kernel)
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    outs = [torch.full((n,), float("nan"), device=DEV) for n in numel]
    run_path(red, grads_dev, arena, outs, order=order, mode="mark_ready_many")   # warm-up
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            red.begin_iteration()
            red.mark_ready_many(order, side)
    torch.cuda.synchronize()
    for step in (1, 2):
        new_flats, new_views, _ = host_grads(numel, W, "f32", step=step)
        for r in range(W):
            flat_dev[r].copy_(torch.from_numpy(new_flats[r]).to(DEV))
        g.replay()
        torch.cuda.synchronize()
        want_arena, want_outs = reduce_buckets(new_views, members, locs, numel)
        assert bits_equal(arena.cpu().numpy(), want_arena), first_mismatch(arena.cpu().numpy(), want_arena)
        for v in range(len(numel)):
            assert bits_equal(outs[v].cpu().numpy(), want_outs[0][v])


def test_nosync_failed_step_changes_nothing():
    """A micro-step rejected for a NULL pointer leaves the block record as it
    was: a later adding step adds to every field (acc = g1 + g3), including
    the fields the rejected call had walked before the NULL."""
    from reduction_reducer_gb300 import InvalidArg
    numel = [100, 37, 4097]
    W = 2
    steps = [host_grads(numel, W, "f32", step=k) for k in range(3)]
    offs = steps[0][2]
    dev = [host_to_device_views(steps[k][0], numel, offs, "f32", DEV)[1] for k in range(3)]
    acc = [[torch.full((n,), float("nan"), device=DEV) for n in numel] for _ in range(W)]
    red = Reducer(numel, "f32", 1 << 20)
    red.bind(acc, torch.empty(red.arena_numel(), device=DEV), None)
    red.accumulate_nosync(acc, dev[0], first_step=True)
    bad = [[t.data_ptr() for t in rep] for rep in dev[1]]
    bad[1][1] = 0                                            # NULL gradient, replica 1, variable 1
    with pytest.raises(InvalidArg):
        red.accumulate_nosync(acc, bad, first_step=True)
    red.accumulate_nosync(acc, dev[2], first_step=False)
    torch.cuda.synchronize()
    for r in range(W):
        want = accumulate_steps([steps[0][1][r], steps[2][1][r]])
        for v in range(len(numel)):
            assert bits_equal(acc[r][v].cpu().numpy(), want[v]), (r, v)
    red.destroy()


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("coalesce", [1, 4096, 1 << 16, 1 << 40])
def test_coalesced_launches(coalesce, kernel):
    """DDP_OPT_COALESCE_ELEMS: the runs released by one mark_ready_many call
    merge into launches of at least that many elements; every element still
    equals the oracle, and the launch count drops accordingly (one launch
    for the whole call when nothing reaches the threshold)."""
    numel = shapes.numels(shapes.gpt2_medium(layers=2, vocab=3000, n_ctx=256))
    per_event = full_compare(numel, 8, "bf16", 0, order="reverse", mode="mark_ready_many", kernel=kernel,
                             options={_lib.OPT_COALESCE_ELEMS: 0})
    n = full_compare(numel, 8, "bf16", 0, order="reverse", mode="mark_ready_many", kernel=kernel,
                     options={_lib.OPT_COALESCE_ELEMS: coalesce})
    assert n <= per_event
    if coalesce == 1:
        assert n == per_event
    if coalesce == 1 << 40:
        assert n == 1
    # a straggler order parks buckets: merged runs still go out in index order
    full_compare(RAGGED, 4, "f32", 16 * 1024, order="straggler", mode="mark_ready_many", kernel=kernel,
                 options={_lib.OPT_COALESCE_ELEMS: coalesce}, iterations=2)


@pytest.mark.parametrize("kernel", ["ldg", "tma"])
def test_coalesced_launches_flushed_before_an_error(kernel):
    """A mark_ready_many call that fails at event i (a variable reported
    twice) still launches what events 0 .. i-1 released, although the
    coalescing threshold would have held those buckets back for a larger
    launch: their arena slices and copy-backs equal the oracle's, the rest
    of the arena is untouched."""
    from reduction_reducer_gb300 import AlreadyReady
    numel = RAGGED
    W, cap = 4, 16 * 1024
    flats, views, offs = host_grads(numel, W, "f32")
    members, locs = assign_buckets(numel, 4, cap)
    want_arena, want_outs = reduce_buckets(views, members, locs, numel)
    _, grads_dev = host_to_device_views(flats, numel, offs, "f32", DEV)
    red = Reducer(numel, "f32", cap)
    set_kernel(red, kernel)
    red.set_option(_lib.OPT_COALESCE_ELEMS, 1 << 40)          # nothing reaches it: one launch per call
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    outs = [torch.full((n,), float("nan"), device=DEV) for n in numel]
    red.bind(grads_dev, arena, outs)
    order = gen.reverse_order(len(numel))
    released = [b for b in range(len(members)) if all(v in order[:8] for v in members[b])]
    assert 0 < len(released) < len(members)
    red.begin_iteration()
    with pytest.raises(AlreadyReady):
        red.mark_ready_many(order[:8] + [order[3]] + order[8:])
    torch.cuda.synchronize()
    got = arena.cpu().numpy()
    lens = [sum(numel[v] for v in m) for m in members]
    starts = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    done = int(starts[len(released)])
    assert bits_equal(got[:done], want_arena[:done]), first_mismatch(got[:done], want_arena[:done])
    assert np.isnan(got[done:]).all()
    for b in released:
        for v in members[b]:
            assert bits_equal(outs[v].cpu().numpy(), want_outs[0][v]), v
    assert red.launch_count() == 1
    red.destroy()
