"""GPU parity of the fused last micro-step of a no_sync block against the
oracle, bit for bit.

The accumulated fields of the first K-1 micro-steps are bound as the
gradients; the last micro-step's gradients are bound with
``bind_last_step``; every reduction then averages fl32(acc_r + g_r) and
leaves the accumulated fields as they were.
"""

import pytest
import torch

from oracle.buckets import assign_buckets
from oracle.nosync import accumulate, accumulate_steps, reduce_last_step
from oracle.reduce import reduce_buckets
from reduction_reducer_gb300 import InvalidArg, Reducer, _lib
from workloads import gen, shapes

from gpu_util import bits_equal, first_mismatch, host_grads, host_to_device_views, layout

pytestmark = pytest.mark.gpu

DEV = "cuda"
MIB = 1 << 20
RAGGED = [0, 1, 2, 3, 5, 7, 8, 13, 64, 67, 100, 1000, 4095, 4097, 70001, 0, 9, 300007, 16, 31]
KERNEL = {"ldg": _lib.KERNEL_LDG, "tma": _lib.KERNEL_TMA, "auto": _lib.KERNEL_AUTO}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import os
    from reduction_reducer_gb300 import build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    _lib.load()
    torch.cuda.set_device(0)


def _drive(red, mode, order, stream=None):
    red.begin_iteration()
    if mode == "mark_ready":
        for v in order:
            red.mark_ready(v, stream)
    elif mode == "mark_ready_many":
        assert red.mark_ready_many(list(order), stream) == len(order)
    elif mode == "reduce_all":
        red.reduce_all(stream)
    elif mode == "reduce_bucket":
        for b in range(red.B):
            red.reduce_bucket(b, stream)
    else:
        raise ValueError(mode)
    torch.cuda.synchronize()


def _fields(numel, W, odd=False):
    offs, total = layout(numel, 64, odd)
    flat = [torch.full((total,), float("nan"), device=DEV) for _ in range(W)]
    return flat, [[f[o:o + n] for o, n in zip(offs, numel)] for f in flat]


@pytest.mark.parametrize("mode", ["mark_ready", "mark_ready_many", "reduce_all", "reduce_bucket"])
@pytest.mark.parametrize("kernel", ["ldg", "tma"])
@pytest.mark.parametrize("W", [1, 2, 3, 4, 5, 8, 16, 32])
def test_last_step_every_element(W, kernel, mode):
    numel = RAGGED
    K, cap = 3, 16 * 1024
    steps = [host_grads(numel, W, "f32", step=k, special=(W == 3)) for k in range(K)]
    offs = steps[0][2]
    acc_np = [accumulate_steps([steps[k][1][r] for k in range(K - 1)]) for r in range(W)]
    members, locs = assign_buckets(numel, 4, cap)
    n_out = W if W in (2, 4) else 1
    want_arena, want_outs = reduce_last_step(acc_np, steps[K - 1][1], members, locs, numel, n_out=n_out)

    dev = [host_to_device_views(steps[k][0], numel, offs, "f32", DEV)[1] for k in range(K)]
    acc_flat, acc = _fields(numel, W)
    red = Reducer(numel, "f32", cap)
    red.set_option(_lib.OPT_KERNEL, KERNEL[kernel])
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    outs = [[torch.full((n,), float("nan"), device=DEV) for n in numel] for _ in range(n_out)]
    red.bind(acc, arena, outs[0] if n_out == 1 else outs)
    for k in range(K - 1):
        red.accumulate_nosync(acc, dev[k], first_step=(k == 0))
    torch.cuda.synchronize()
    before = [f.clone() for f in acc_flat]
    red.bind_last_step(dev[K - 1])
    _drive(red, mode, gen.straggler_order(members, p=0.5, seed=W))
    assert red.device_status() == 0
    got = arena.cpu().numpy()
    assert bits_equal(got, want_arena), first_mismatch(got, want_arena)
    for o in range(n_out):
        for v in range(len(numel)):
            assert bits_equal(outs[o][v].cpu().numpy(), want_outs[0][v]), (o, v)
    for r in range(W):   # the accumulated fields are read, not written
        assert torch.equal(acc_flat[r].view(torch.int32), before[r].view(torch.int32)), r
    # unbound again: the next iteration averages the accumulated fields alone
    red.bind_last_step(None)
    _drive(red, "mark_ready_many", gen.reverse_order(len(numel)))
    plain_arena, _ = reduce_buckets(acc_np, members, locs, numel)
    assert bits_equal(arena.cpu().numpy(), plain_arena)
    red.destroy()


@pytest.mark.parametrize("kernel", ["ldg", "tma"])
def test_last_step_misaligned(kernel):
    """Last-step gradients at odd offsets beside 16-byte-aligned accumulated
    fields (and the reverse): the segments lose the vector path and take the
    scalar one; still bit-exact."""
    numel = RAGGED
    W, cap = 2, 64 * 1024
    members, locs = assign_buckets(numel, 4, cap)
    for acc_odd, last_odd in ((False, True), (True, False)):
        a_fl, a_np, a_off = host_grads(numel, W, "f32", step=0, odd=acc_odd, special=True)
        g_fl, g_np, g_off = host_grads(numel, W, "f32", step=1, odd=last_odd)
        want_arena, want_outs = reduce_last_step(a_np, g_np, members, locs, numel)
        _, acc = host_to_device_views(a_fl, numel, a_off, "f32", DEV)
        _, last = host_to_device_views(g_fl, numel, g_off, "f32", DEV)
        red = Reducer(numel, "f32", cap)
        red.set_option(_lib.OPT_KERNEL, KERNEL[kernel])
        arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
        outs = [torch.full((n,), float("nan"), device=DEV) for n in numel]
        red.bind(acc, arena, outs)
        red.bind_last_step(last)
        _drive(red, "mark_ready_many", gen.reverse_order(len(numel)))
        assert red.device_status() == 0
        assert bits_equal(arena.cpu().numpy(), want_arena), first_mismatch(arena.cpu().numpy(), want_arena)
        for v in range(len(numel)):
            assert bits_equal(outs[v].cpu().numpy(), want_outs[0][v]), v
        red.destroy()


def test_last_step_equals_unfused_block():
    """The fused reduction against accumulate-then-reduce through the same
    library, BERT-large with 2 layers, W = 4, library defaults."""
    numel = shapes.numels(shapes.bert_large(layers=2, vocab=2048))
    W, K, cap = 4, 4, 2 * MIB
    offs, total = gen.packed_offsets(numel, 64)
    steps = [[gen.draw_flat_torch(total, r, k, "f32", DEV) for r in range(W)] for k in range(K)]
    views = [[[f[o:o + n] for o, n in zip(offs, numel)] for f in sk] for sk in steps]
    results = []
    for fused in (False, True):
        acc_flat = [torch.empty(total, device=DEV) for _ in range(W)]
        acc = [[f[o:o + n] for o, n in zip(offs, numel)] for f in acc_flat]
        red = Reducer(numel, "f32", cap)
        arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
        out_flat = torch.full((total,), float("nan"), device=DEV)
        red.bind(acc, arena, [out_flat[o:o + n] for o, n in zip(offs, numel)])
        for k in range(K - 1 if fused else K):
            red.accumulate_nosync(acc, views[k], first_step=(k == 0))
        if fused:
            red.bind_last_step(views[K - 1])
        _drive(red, "mark_ready_many", gen.reverse_order(len(numel)))
        assert red.device_status() == 0
        results.append((arena.clone(), out_flat.clone()))
        red.destroy()
    assert torch.equal(results[0][0].view(torch.int32), results[1][0].view(torch.int32))
    assert torch.equal(results[0][1].view(torch.int32), results[1][1].view(torch.int32))


def test_last_step_rules_on_device():
    numel = [64, 100]
    W = 2
    acc_flat, acc = _fields(numel, W)
    last_flat, last = _fields(numel, W)
    red = Reducer(numel, "f32", 256)
    arena = torch.empty(red.arena_numel(), device=DEV)
    red.bind(acc, arena, None)
    red.bind_last_step(last)
    with pytest.raises(InvalidArg):
        red.set_option(_lib.OPT_FIND_UNUSED, 1)
    with pytest.raises(InvalidArg):
        red.register_comm_hook("mean", [torch.empty(red.arena_numel(), device=DEV) for _ in range(W)])
    red.begin_iteration()
    red.mark_ready(1)
    with pytest.raises(InvalidArg):     # inside an unfinished iteration
        red.bind_last_step(None)
    red.mark_ready(0)
    torch.cuda.synchronize()
    # rebinding the gradients drops the last step
    for f in acc_flat + last_flat:
        f.fill_(1.0)
    red.bind(acc, arena, None)
    _drive(red, "reduce_all", None)
    assert torch.equal(arena, torch.ones_like(arena))
    red.destroy()


def test_nosync_resnet50_last_step_full_size_every_element():
    """ResNet-50, W = 16, K = 8: seven accumulate micro-steps, then the
    eighth fused into the reduction; every element of the accumulated fields
    (left as the seventh step wrote them), the arena and the copy-back
    against the oracle."""
    from gpu_util import nosync_full_size_check
    numel = shapes.numels(shapes.resnet50())
    W, K = 16, 8
    offs, total = gen.packed_offsets(numel, 64)
    steps = [[gen.draw_flat_torch(total, r, k, "f32", DEV) for r in range(W)] for k in range(K)]
    views = [[[f[o:o + n] for o, n in zip(offs, numel)] for f in sk] for sk in steps]
    acc_flat = [torch.full((total,), float("nan"), device=DEV) for _ in range(W)]
    acc = [[f[o:o + n] for o, n in zip(offs, numel)] for f in acc_flat]
    red = Reducer(numel, "f32", 25 * MIB)
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    out_flat = torch.full((total,), float("nan"), device=DEV)
    red.bind(acc, arena, [out_flat[o:o + n] for o, n in zip(offs, numel)])
    for k in range(K - 1):
        red.accumulate_nosync(acc, views[k], first_step=(k == 0))
    red.bind_last_step(views[K - 1])
    _drive(red, "mark_ready_many", gen.reverse_order(len(numel)))
    assert red.device_status() == 0
    red.destroy()
    nosync_full_size_check(numel, offs, steps, acc_flat, arena, out_flat, K, True)
