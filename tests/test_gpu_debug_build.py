"""The bounds-checking build (-DDDP_DEBUG) on the GPU.

Every kernel of that build checks the ranges it walks and every bulk copy it
issues, and records the first failed check instead of touching memory out of
range.  These cases run the parity workloads through it: the results must
still equal the oracle bit for bit and the record must stay empty.  The
bounded-wait self-test makes a kernel's wait run out on purpose (a barrier
nothing completes) and checks that the wait ends with its status code and
that the device stays usable.
"""

import os

import numpy as np
import pytest
import torch

from oracle.buckets import assign_buckets
from oracle.hooks import hook_bf16_compress, hook_mean, reduce_with_hook
from oracle.nosync import accumulate_steps, reduce_last_step
from oracle.reduce import reduce_buckets
from oracle.unused import reduce_with_unused
from reduction_reducer_gb300 import Reducer, _lib, selftest_bounded_wait
from workloads import gen, shapes

from gpu_util import bits_equal, first_mismatch, host_grads, host_to_device_views

pytestmark = pytest.mark.gpu

DEV = "cuda"
MIB = 1 << 20
RAGGED = [0, 1, 2, 3, 5, 7, 8, 13, 64, 67, 100, 1000, 4095, 4097, 70001, 0, 9, 300007, 16, 31]
KERNEL = {"ldg": _lib.KERNEL_LDG, "tma": _lib.KERNEL_TMA}
DBG = _lib.DEBUG_LIB_PATH


@pytest.fixture(scope="module", autouse=True)
def _built():
    from reduction_reducer_gb300 import build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    if not os.path.exists(DBG):
        build.build_debug()
    _lib.load(DBG)
    torch.cuda.set_device(0)


def _clean(red):
    assert red.device_status() == 0
    assert red.debug_record() == (0, 0)


def _reduce_case(numel, W, dtype, cap, kernel, mode, odd=False, n_out=1):
    flats, views, offs = host_grads(numel, W, dtype, odd=odd, special=True)
    members, locs = assign_buckets(numel, 4 if dtype == "f32" else 2, cap)
    want_arena, want_outs = reduce_buckets(views, members, locs, numel, n_out=n_out)
    _, grads = host_to_device_views(flats, numel, offs, dtype, DEV)
    red = Reducer(numel, dtype, cap, lib_path=DBG)
    red.set_option(_lib.OPT_KERNEL, KERNEL[kernel])
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    outs = [[torch.full((n,), float("nan"), device=DEV) for n in numel] for _ in range(n_out)]
    red.bind(grads, arena, outs[0] if n_out == 1 else outs)
    red.begin_iteration()
    if mode == "mark_ready_many":
        red.mark_ready_many(gen.straggler_order(members, p=0.5, seed=W))
    else:
        red.reduce_all()
    torch.cuda.synchronize()
    _clean(red)
    assert bits_equal(arena.cpu().numpy(), want_arena), first_mismatch(arena.cpu().numpy(), want_arena)
    for o in range(n_out):
        for v in range(len(numel)):
            assert bits_equal(outs[o][v].cpu().numpy(), want_outs[0][v]), (o, v)
    red.destroy()


@pytest.mark.parametrize("kernel", ["ldg", "tma"])
@pytest.mark.parametrize("mode", ["mark_ready_many", "reduce_all"])
@pytest.mark.parametrize("W,dtype,odd", [(3, "f32", False), (4, "f32", True), (8, "bf16", False), (5, "bf16", True),
                                         (16, "f32", False), (256, "f32", True), (256, "bf16", False)])
def test_debug_build_reduce(W, dtype, odd, kernel, mode):
    _reduce_case(RAGGED, W, dtype, 16 * 1024, kernel, mode, odd=odd, n_out=W if W == 4 else 1)


@pytest.mark.parametrize("kernel", ["ldg", "tma"])
@pytest.mark.parametrize("cap_mib", [0, 1])
def test_debug_build_gpt2_reduced(kernel, cap_mib):
    numel = shapes.numels(shapes.gpt2_medium(layers=2, vocab=3000, n_ctx=256))
    _reduce_case(numel, 8, "bf16", cap_mib * MIB, kernel, "mark_ready_many")


@pytest.mark.parametrize("mode", ["mark_ready_many", "reduce_all"])
def test_debug_build_large_buckets(mode):
    """GPT-2-medium with 8 layers in 100 MiB buckets (54.6M and 98.7M bf16
    elements): the first bucket's bulk-copy launch gets eight resident
    waves (sized by its slices), the final one eight, and the single
    reduce_all launch 24."""
    numel = shapes.numels(shapes.gpt2_medium(layers=8))
    _reduce_case(numel, 8, "bf16", 100 * MIB, "tma", mode)


@pytest.mark.parametrize("kernel", ["ldg", "tma"])
def test_debug_build_nosync_and_last_step(kernel):
    numel = RAGGED
    W, K, cap = 16, 3, 16 * 1024
    steps = [host_grads(numel, W, "f32", step=k) for k in range(K)]
    offs = steps[0][2]
    acc_np = [accumulate_steps([steps[k][1][r] for k in range(K - 1)]) for r in range(W)]
    members, locs = assign_buckets(numel, 4, cap)
    want_arena, want_outs = reduce_last_step(acc_np, steps[K - 1][1], members, locs, numel)
    dev = [host_to_device_views(steps[k][0], numel, offs, "f32", DEV)[1] for k in range(K)]
    acc = [[torch.full((n,), float("nan"), device=DEV) for n in numel] for _ in range(W)]
    red = Reducer(numel, "f32", cap, lib_path=DBG)
    red.set_option(_lib.OPT_KERNEL, KERNEL[kernel])
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    outs = [torch.full((n,), float("nan"), device=DEV) for n in numel]
    red.bind(acc, arena, outs)
    for k in range(K - 1):
        red.accumulate_nosync(acc, dev[k], first_step=(k == 0))
    red.bind_last_step(dev[K - 1])
    red.begin_iteration()
    red.mark_ready_many(gen.reverse_order(len(numel)))
    torch.cuda.synchronize()
    _clean(red)
    for r in range(W):
        for v in range(len(numel)):
            assert bits_equal(acc[r][v].cpu().numpy(), acc_np[r][v]), (r, v)
    assert bits_equal(arena.cpu().numpy(), want_arena)
    for v in range(len(numel)):
        assert bits_equal(outs[v].cpu().numpy(), want_outs[0][v]), v
    red.destroy()


@pytest.mark.parametrize("kernel", ["ldg", "tma"])
def test_debug_build_unused_parameters(kernel):
    numel = RAGGED
    W, cap = 3, 16 * 1024
    rng = np.random.default_rng(17)
    used = rng.random((W, len(numel))) < 0.7
    used[:, 10] = True
    flats, views, offs = host_grads(numel, W, "f32")
    members, locs = assign_buckets(numel, 4, cap)
    want_arena, _ = reduce_with_unused(views, used.tolist(), members, locs, numel)
    _, grads = host_to_device_views(flats, numel, offs, "f32", DEV)
    red = Reducer(numel, "f32", cap, lib_path=DBG)
    red.set_option(_lib.OPT_KERNEL, KERNEL[kernel])
    red.set_option(_lib.OPT_FIND_UNUSED, 1)
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    red.bind(grads, arena, [torch.zeros(n, device=DEV) for n in numel])
    red.set_local_used(used.tolist())
    red.begin_iteration()
    g = used.any(axis=0)
    red.mark_ready_many([v for v in range(len(numel) - 1, -1, -1) if g[v]])
    torch.cuda.synchronize()
    _clean(red)
    assert bits_equal(arena.cpu().numpy(), want_arena), first_mismatch(arena.cpu().numpy(), want_arena)
    red.destroy()


@pytest.mark.parametrize("hook,fused", [("mean", 1), ("mean", 0), ("bf16_compress", 1)])
def test_debug_build_hooks(hook, fused):
    numel = RAGGED
    W, cap = 4, 16 * 1024
    flats, views, offs = host_grads(numel, W, "f32")
    members, locs = assign_buckets(numel, 4, cap)
    want_arena, want_outs, _ = reduce_with_hook(views, members, locs, numel,
                                                hook_mean if hook == "mean" else hook_bf16_compress)
    _, grads = host_to_device_views(flats, numel, offs, "f32", DEV)
    red = Reducer(numel, "f32", cap, lib_path=DBG)
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    outs = [torch.full((n,), float("nan"), device=DEV) for n in numel]
    red.bind(grads, arena, outs)
    red.register_comm_hook(hook, [torch.empty(red.arena_numel(), device=DEV) for _ in range(W)])
    red.set_option(_lib.OPT_HOOK_FUSED, fused)
    red.begin_iteration()
    red.mark_ready_many(gen.reverse_order(len(numel)))
    torch.cuda.synchronize()
    _clean(red)
    assert bits_equal(arena.cpu().numpy(), want_arena)
    for v in range(len(numel)):
        assert bits_equal(outs[v].cpu().numpy(), want_outs[0][v]), v
    red.destroy()


def test_debug_build_bert_large_bench_configuration():
    """The bench's own configuration (BERT-large W=4, library defaults,
    stored straggler order, one mark_ready_many call) through the checking
    build: no check fails on the full-size layout."""
    numel = shapes.numels(shapes.bert_large())
    path = os.path.join(os.path.dirname(__file__), "golden", "bert_large_ready_order.txt")
    order = [int(l) for l in open(path) if l.strip() and not l.startswith("#")]
    offs, total = gen.packed_offsets(numel, 64)
    W = 4
    flat = [gen.draw_flat_torch(total, r, 0, "f32", DEV) for r in range(W)]
    grads = [[f[o:o + n] for o, n in zip(offs, numel)] for f in flat]
    results = []
    for path_ in (_lib.LIB_PATH, DBG):
        red = Reducer(numel, "f32", 25 * MIB, lib_path=path_)
        arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
        out = torch.full((total,), float("nan"), device=DEV)
        red.bind(grads, arena, [out[o:o + n] for o, n in zip(offs, numel)])
        red.begin_iteration()
        red.mark_ready_many(order)
        torch.cuda.synchronize()
        _clean(red)
        results.append((arena.clone(), out.clone()))
        red.destroy()
    # the checking build computes the same bits as the release build
    assert torch.equal(results[0][0].view(torch.int32), results[1][0].view(torch.int32))
    assert torch.equal(results[0][1].view(torch.int32), results[1][1].view(torch.int32))


@pytest.mark.parametrize("lib_path", [_lib.LIB_PATH, DBG], ids=["release", "debug"])
def test_bounded_wait_gives_up_and_device_stays_usable(lib_path):
    """A wait on a barrier that nothing completes ends after its budget
    (~1 ms here) with the timeout code; the next reduction still matches the
    oracle."""
    assert selftest_bounded_wait(2_000_000, lib_path) == 3
    numel = [1000, 4097, 70001]
    flats, views, offs = host_grads(numel, 2, "f32")
    members, locs = assign_buckets(numel, 4, 16 * 1024)
    want_arena, _ = reduce_buckets(views, members, locs, numel)
    _, grads = host_to_device_views(flats, numel, offs, "f32", DEV)
    red = Reducer(numel, "f32", 16 * 1024, lib_path=lib_path)
    red.set_option(_lib.OPT_KERNEL, _lib.KERNEL_TMA)
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    red.bind(grads, arena, None)
    red.begin_iteration()
    red.reduce_all()
    torch.cuda.synchronize()
    _clean(red)
    assert bits_equal(arena.cpu().numpy(), want_arena)
    red.destroy()
