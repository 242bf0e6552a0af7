"""GPU parity of the communication-hook path against the oracle, bit for
bit -- the built-in hooks inside the fused bucket pass and through gather,
hook call and copy-back -- and of the hook contract: one call per bucket in
index order with the bucket's metadata."""

import numpy as np
import pytest
import torch

from oracle.buckets import assign_buckets
from oracle.hooks import gather_buckets, hook_bf16_compress, hook_mean, reduce_with_hook
from reduction_reducer_gb300 import HookError, InvalidArg, Reducer, _lib
from workloads import gen, shapes

from gpu_util import bits_equal, first_mismatch, host_grads, host_to_device_views

pytestmark = pytest.mark.gpu

DEV = "cuda"
MIB = 1 << 20
RAGGED = [0, 1, 2, 3, 5, 7, 8, 13, 64, 67, 100, 1000, 4095, 4097, 70001, 0, 9, 300007, 16, 31]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import os
    from reduction_reducer_gb300 import build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    _lib.load()
    torch.cuda.set_device(0)


def _setup(numel, W, dtype, cap, n_out, odd=False):
    flats, views, offs = host_grads(numel, W, dtype, odd=odd)
    _, grads_dev = host_to_device_views(flats, numel, offs, dtype, DEV)
    red = Reducer(numel, dtype, cap)
    N = red.arena_numel()
    arena = torch.full((N,), float("nan"), device=DEV)
    outs = [[torch.full((n,), float("nan"), device=DEV) for n in numel] for _ in range(max(n_out, 1))]
    go = None if n_out == 0 else (outs[0] if n_out == 1 else outs)
    red.bind(grads_dev, arena, go)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    rb = [torch.empty(max(N, 1), dtype=tdt, device=DEV) for _ in range(W)]
    return red, views, arena, outs, rb


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "gathered"])
@pytest.mark.parametrize("hook", ["mean", "bf16_compress"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("W,n_out", [(1, 1), (3, 1), (4, 4), (8, 0), (33, 1)])
def test_builtin_hooks(hook, dtype, W, n_out, fused):
    """Both routes of a built-in hook: inside the fused bucket pass (the
    default; the replica buffers stay as they were) and through gather, hook
    call and copy-back (the replica buffers hold each replica's buckets)."""
    numel = RAGGED
    cap = 16 * 1024
    red, views, arena, outs, rb = _setup(numel, W, dtype, cap, n_out, odd=(W == 3))
    for t in rb:
        t.view(torch.int16).fill_(0x7FC1)        # a NaN pattern (fp32 and bf16) no hook writes
    red.register_comm_hook(hook, rb)
    red.set_option(_lib.OPT_HOOK_FUSED, 1 if fused else 0)
    launches0 = red.launch_count()
    members, locs = assign_buckets(numel, 4 if dtype == "f32" else 2, cap)
    fn = hook_mean if hook == "mean" else hook_bf16_compress
    want_arena, want_outs, _ = reduce_with_hook(views, members, locs, numel, fn, n_out=max(n_out, 1))
    red.begin_iteration()
    red.mark_ready_many(gen.straggler_order(members, p=0.5, seed=1))
    torch.cuda.synchronize()
    got = arena.cpu().numpy()
    assert bits_equal(got, want_arena), first_mismatch(got, want_arena)
    for o in range(n_out):
        for v in range(len(numel)):
            assert bits_equal(outs[o][v].cpu().numpy(), want_outs[0][v]), (o, v)
    assert red.device_status() == 0
    if fused:
        # one launch per readiness event that releases buckets, nothing gathered
        assert red.launch_count() - launches0 <= len(members)
        for t in rb:
            assert bool((t.view(torch.int16) == 0x7FC1).all())
        return
    # the replica buffers hold each replica's gathered buckets
    bufs = gather_buckets(views, members, locs, numel)
    lens = [sum(numel[v] for v in m) for m in members]
    starts = np.concatenate([[0], np.cumsum(lens)])
    for r in range(W):
        host = rb[r].view(torch.int16).cpu().numpy().view(np.uint16) if dtype == "bf16" else rb[r].cpu().numpy()
        for b in range(len(members)):
            assert np.array_equal(host[starts[b]:starts[b + 1]].view(np.uint8), bufs[r][b].view(np.uint8))


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "gathered"])
@pytest.mark.parametrize("hook", ["mean", "bf16_compress"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_builtin_hooks_special_values(hook, dtype, fused):
    """±0, ±Inf, NaN, subnormals and ±3.4e38 (above the largest bf16, so the
    compression hook rounds it to ±Inf) at seeded positions: the hooks'
    device rounding and sums match the oracle bit for bit (NaN as a class)."""
    numel = RAGGED
    W, n_out, cap = 4, 1, 16 * 1024
    flats, views, offs = host_grads(numel, W, dtype, special=True)
    _, grads_dev = host_to_device_views(flats, numel, offs, dtype, DEV)
    red = Reducer(numel, dtype, cap)
    N = red.arena_numel()
    arena = torch.full((N,), float("nan"), device=DEV)
    outs = [torch.full((n,), float("nan"), device=DEV) for n in numel]
    red.bind(grads_dev, arena, outs)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    red.register_comm_hook(hook, [torch.empty(max(N, 1), dtype=tdt, device=DEV) for _ in range(W)])
    red.set_option(_lib.OPT_HOOK_FUSED, 1 if fused else 0)
    members, locs = assign_buckets(numel, 4 if dtype == "f32" else 2, cap)
    fn = hook_mean if hook == "mean" else hook_bf16_compress
    want_arena, want_outs, _ = reduce_with_hook(views, members, locs, numel, fn, n_out=n_out)
    red.begin_iteration()
    red.mark_ready_many(gen.reverse_order(len(numel)))
    torch.cuda.synchronize()
    got = arena.cpu().numpy()
    assert bits_equal(got, want_arena), first_mismatch(got, want_arena)
    assert np.isinf(want_arena).any() and np.isnan(want_arena).any()   # the special values reached the result
    for v in range(len(numel)):
        assert bits_equal(outs[v].cpu().numpy(), want_outs[0][v]), v
    assert red.device_status() == 0


def test_default_hook_equals_fused_pass():
    numel = shapes.numels(shapes.bert_large(layers=2, vocab=2048))
    W = 4
    flats, views, offs = host_grads(numel, W, "f32")
    _, grads_dev = host_to_device_views(flats, numel, offs, "f32", DEV)
    results = []
    for use_hook in (False, True):
        red = Reducer(numel, "f32", 2 * MIB)
        arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
        outs = [torch.full((n,), float("nan"), device=DEV) for n in numel]
        red.bind(grads_dev, arena, outs)
        if use_hook:
            red.register_comm_hook("mean", [torch.empty(red.arena_numel(), device=DEV) for _ in range(W)])
        red.begin_iteration()
        red.mark_ready_many(gen.reverse_order(len(numel)))
        torch.cuda.synchronize()
        results.append((arena.clone(), [o.clone() for o in outs]))
    assert torch.equal(results[0][0].view(torch.int32), results[1][0].view(torch.int32))
    for a, b in zip(results[0][1], results[1][1]):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_python_hook_sees_every_bucket_in_order():
    numel = RAGGED
    W, cap = 3, 16 * 1024
    red, views, arena, outs, rb = _setup(numel, W, "f32", cap, 1)
    members, locs = assign_buckets(numel, 4, cap)
    seen = []
    lib = _lib.load()

    def hook(bucket, stream):
        seen.append((bucket.index, bucket.num_buckets, bucket.is_last, bucket.W, bucket.numel,
                     [bucket.variables[i] for i in range(bucket.n_vars)],
                     [bucket.offsets[i] for i in range(bucket.n_vars)],
                     [bucket.lengths[i] for i in range(bucket.n_vars)]))
        return lib.ddp_hook_mean(None, bucket, stream)     # the user hook delegates the arithmetic

    red.register_comm_hook(hook, rb)
    red.begin_iteration()
    red.mark_ready_many(gen.straggler_order(members, p=0.5, seed=3))
    torch.cuda.synchronize()
    B = len(members)
    assert [s[0] for s in seen] == list(range(B))
    for b, (idx, nb, last, w, n, vs, of, ln) in enumerate(seen):
        assert (nb, last, w) == (B, b == B - 1, W)
        assert vs == members[b]
        assert of == [locs[v].offset for v in vs] and ln == [numel[v] for v in vs]
        assert n == sum(numel[v] for v in vs)
    want_arena, _, _ = reduce_with_hook(views, members, locs, numel, hook_mean)
    assert bits_equal(arena.cpu().numpy(), want_arena)


def test_hook_failure_and_registration_rules():
    numel = [64, 64]
    red, _, _, _, rb = _setup(numel, 2, "f32", 256, 1)
    red.register_comm_hook(lambda bucket, stream: 7, rb)
    red.begin_iteration()
    with pytest.raises(HookError):
        red.mark_ready_many([1, 0])
    red2, _, _, _, rb2 = _setup(numel, 2, "f32", 256, 1)
    red2.reduce_all()
    torch.cuda.synchronize()
    with pytest.raises(InvalidArg):
        red2.register_comm_hook("mean", rb2)            # after the first launch


@pytest.mark.parametrize("hook", ["mean", "bf16_compress"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("W,n_out", [(1, 0), (4, 0), (4, 1), (3, 3)])
def test_hooks_on_bucket_views(hook, dtype, W, n_out):
    """Gradients laid out as views of the bucket layout, no replica buffers:
    nothing is gathered, the hook reads the gradients in place, and the
    result matches the oracle bit for bit."""
    numel = RAGGED
    cap = 16 * 1024
    red = Reducer(numel, dtype, cap)
    _, boff = red.get_bucket_info()
    locs = red.get_locators()
    offs = [boff[b] + off for (b, _, off, _) in locs]
    total = boff[-1]
    flats, views, _ = host_grads(numel, W, dtype)
    # re-pack every replica's gradients in bucket order
    packed = []
    for r in range(W):
        f = np.zeros(total, dtype=flats[r].dtype)
        for v, n in enumerate(numel):
            f[offs[v]:offs[v] + n] = views[r][v].view(flats[r].dtype)
        packed.append(f)
    flat_dev, grads_dev = host_to_device_views(packed, numel, offs, dtype, DEV)
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    outs = [[torch.full((n,), float("nan"), device=DEV) for n in numel] for _ in range(max(n_out, 1))]
    red.bind(grads_dev, arena, None if n_out == 0 else (outs[0] if n_out == 1 else outs))
    seen = []
    lib = _lib.load()
    builtin = lib.ddp_hook_mean if hook == "mean" else lib.ddp_hook_bf16_compress

    def spy(bucket, stream):
        seen.append([bucket.replicas[r] for r in range(bucket.W)])
        return builtin(None, bucket, stream)

    red.register_comm_hook(spy, None)
    members, olocs = assign_buckets(numel, 4 if dtype == "f32" else 2, cap)
    fn = hook_mean if hook == "mean" else hook_bf16_compress
    want_arena, want_outs, _ = reduce_with_hook(views, members, olocs, numel, fn, n_out=max(n_out, 1))
    launches0 = red.launch_count()
    red.begin_iteration()
    red.mark_ready_many(gen.straggler_order(members, p=0.5, seed=2))
    torch.cuda.synchronize()
    got = arena.cpu().numpy()
    assert bits_equal(got, want_arena), first_mismatch(got, want_arena)
    for o in range(n_out):
        for v in range(len(numel)):
            assert bits_equal(outs[o][v].cpu().numpy(), want_outs[0][v]), (o, v)
    esz = 4 if dtype == "f32" else 2
    for b, ptrs in enumerate(seen):            # the hook saw the gradients themselves
        for r in range(W):
            assert ptrs[r] == flat_dev[r].data_ptr() + boff[b] * esz or boff[b + 1] == boff[b]
    # copy-back launches only (one per bucket with outputs), no gather
    assert red.launch_count() - launches0 == (len(members) if n_out else 0)


def test_hook_on_bucket_views_detects_a_broken_layout():
    numel = [100, 200, 300]
    W = 2
    red = Reducer(numel, "f32", 1 << 20)          # one bucket: push order 2, 1, 0
    _, boff = red.get_bucket_info()
    locs = red.get_locators()
    flat = [torch.zeros(boff[-1], device=DEV) for _ in range(W)]
    views = [[f[boff[b] + off:boff[b] + off + n] for (b, _, off, n) in locs] for f in flat]
    arena = torch.empty(red.arena_numel(), device=DEV)
    red.bind(views, arena, None)
    red.register_comm_hook("mean", None)
    red.set_option(_lib.OPT_HOOK_FUSED, 0)        # the hook-call route reads the views in place
    # rebinding in registration order breaks the view layout: the launch fails
    other = [torch.zeros(sum(numel), device=DEV) for _ in range(W)]
    offs = [0, 100, 300]
    red.bind([[f[o:o + n] for o, n in zip(offs, numel)] for f in other], arena, None)
    red.begin_iteration()
    with pytest.raises(InvalidArg):
        red.mark_ready_many([2, 1, 0])
