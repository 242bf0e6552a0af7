"""GPU parity of unused-parameter handling (find_unused_parameters and the
globally-unused bitmap) against the oracle, bit for bit.

A replica without a gradient contributes a zero-filled slice; variables
unused on every replica are marked ready at the first event and keep their
copy-back untouched (the guard words written before the run must survive);
under no_sync the local-use bits accumulate and a gradient field takes its
first gradient.
"""

import numpy as np
import pytest
import torch

from oracle.buckets import assign_buckets
from oracle.unused import accumulate_masked, globally_used, reduce_with_unused
from reduction_reducer_gb300 import AlreadyReady, Reducer, _lib
from workloads import gen, shapes

from gpu_util import bits_equal, first_mismatch, host_grads, host_to_device_views, layout

pytestmark = pytest.mark.gpu

DEV = "cuda"
GUARD = np.uint32(0x7FC0DEAD)
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


def _reducer(numel, dtype, cap, kernel):
    red = Reducer(numel, dtype, cap)
    red.set_option(_lib.OPT_KERNEL, {"tma": _lib.KERNEL_TMA, "ldg": _lib.KERNEL_LDG, "auto": _lib.KERNEL_AUTO}[kernel])
    red.set_option(_lib.OPT_FIND_UNUSED, 1)
    return red


def _guarded_outputs(numel, n_out):
    out_offs, out_total = layout(numel, 64)
    bufs, views = [], []
    for _ in range(n_out):
        flat = torch.from_numpy(np.full(out_total, GUARD, np.uint32).view(np.float32)).to(DEV)
        bufs.append(flat)
        views.append([flat[o:o + n] for o, n in zip(out_offs, numel)])
    return bufs, views, out_offs


def _used_pattern(rng, W, P, p=0.7):
    used = rng.random((W, P)) < p
    used[:, 3] = False                  # one variable unused on every replica
    used[0, 5] = False                  # one unused on replica 0 only
    used[:, 10] = True
    return used


def _check_outputs(bufs, out_offs, numel, want_outs, used):
    g = globally_used(used)
    for o, flat in enumerate(bufs):
        host = flat.cpu().numpy()
        for v, (off, n) in enumerate(zip(out_offs, numel)):
            got = host[off:off + n]
            if not g[v]:
                assert np.all(got.view(np.uint32) == GUARD), f"copy-back of unused variable {v} was written"
            else:
                assert bits_equal(got, want_outs[0][v]), (o, v, first_mismatch(got, want_outs[0][v]))


@pytest.mark.parametrize("kernel", ["ldg", "tma"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("W", [1, 2, 3, 4, 8, 64])
def test_unused_reduce(W, dtype, kernel):
    numel = RAGGED
    P = len(numel)
    rng = np.random.default_rng(W * 7 + (dtype == "bf16"))
    used = _used_pattern(rng, W, P)
    flats, views, offs = host_grads(numel, W, dtype, special=(W == 3))
    elem = 4 if dtype == "f32" else 2
    cap = 16 * 1024
    members, locs = assign_buckets(numel, elem, cap)
    n_out = W if W in (2, 4) else 1
    want_arena, want_outs = reduce_with_unused(views, used.tolist(), members, locs, numel, n_out=n_out)
    _, grads_dev = host_to_device_views(flats, numel, offs, dtype, DEV)
    red = _reducer(numel, dtype, cap, kernel)
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    bufs, out_views, out_offs = _guarded_outputs(numel, n_out)
    red.bind(grads_dev, arena, out_views[0] if n_out == 1 else out_views)
    red.set_local_used(used.tolist())
    red.begin_iteration()
    g = globally_used(used.tolist())
    order = [int(v) for v in rng.permutation(P) if g[v]]
    with pytest.raises(AlreadyReady):
        red.mark_ready(3)
    assert red.mark_ready_many(order) == len(order)
    torch.cuda.synchronize()
    assert red.device_status() == 0
    got = arena.cpu().numpy()
    assert bits_equal(got, want_arena), first_mismatch(got, want_arena)
    _check_outputs(bufs, out_offs, numel, want_outs, used.tolist())
    # the next iteration without new bits uses every replica again
    red.begin_iteration()
    red.mark_ready_many(list(range(P)))
    torch.cuda.synchronize()
    from oracle.reduce import reduce_buckets
    plain_arena, _ = reduce_buckets(views, members, locs, numel)
    assert bits_equal(arena.cpu().numpy(), plain_arena)


@pytest.mark.parametrize("kernel", ["ldg", "tma"])
def test_unused_with_nosync_bitmap(kernel):
    numel = RAGGED
    P, W, K = len(numel), 3, 3
    rng = np.random.default_rng(42)
    steps = [host_grads(numel, W, "f32", step=k) for k in range(K)]
    offs = steps[0][2]
    bits = [rng.random((W, P)) < 0.6 for _ in range(K)]
    for b in bits:
        b[:, 3] = False                                 # never used
    bits[1][:, 7] = True                                # used only from step 2 on
    bits[0][:, 7] = False
    # oracle: per replica, gradient fields fill on first use and add after
    acc_np, has = [], []
    for r in range(W):
        a, h = None, None
        for k in range(K):
            a, h = accumulate_masked(a, h, steps[k][1][r], bits[k][r].tolist(), first_step=(k == 0))
        acc_np.append(a)
        has.append(h)
    members, locs = assign_buckets(numel, 4, 16 * 1024)
    filled = [[a if a is not None else np.zeros(n, np.float32) for a, n in zip(acc_np[r], numel)] for r in range(W)]
    want_arena, want_outs = reduce_with_unused(filled, has, members, locs, numel)

    dev_steps = [host_to_device_views(steps[k][0], numel, offs, "f32", DEV)[1] for k in range(K)]
    acc_flat = [torch.full((offs[-1] + numel[-1] + 64,), float("nan"), device=DEV) for _ in range(W)]
    acc_dev = [[f[o:o + n] for o, n in zip(offs, numel)] for f in acc_flat]
    red = _reducer(numel, "f32", 16 * 1024, kernel)
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    bufs, out_views, out_offs = _guarded_outputs(numel, 1)
    red.bind(acc_dev, arena, out_views[0])
    for k in range(K):
        red.accumulate_nosync(acc_dev, dev_steps[k], first_step=(k == 0), used=bits[k].tolist())
    g = globally_used(has)
    red.begin_iteration()
    red.mark_ready_many([v for v in range(P - 1, -1, -1) if g[v]])
    torch.cuda.synchronize()
    assert red.device_status() == 0
    for r in range(W):
        for v in range(P):
            if has[r][v]:
                assert bits_equal(acc_dev[r][v].cpu().numpy(), acc_np[r][v]), (r, v)
            else:   # never filled in this block: untouched (still NaN)
                assert torch.isnan(acc_dev[r][v]).all()
    assert bits_equal(arena.cpu().numpy(), want_arena), first_mismatch(arena.cpu().numpy(), want_arena)
    _check_outputs(bufs, out_offs, numel, want_outs, has)


def test_unused_bert_large_full_size_every_element():
    """BERT-large W=4 in the bench's layout: the pooler unused on every
    replica, every fourth encoder layer's FFN unused on replica 1; every
    element of the arena and of the copy-back (untouched where the variable
    is unused everywhere) against the oracle."""
    numel = shapes.numels(shapes.bert_large())
    names = [n for n, _ in shapes.bert_large()]
    P, W = len(numel), 4
    used = np.ones((W, P), bool)
    for v, n in enumerate(names):
        if n.startswith("pooler"):
            used[:, v] = False
        if ".intermediate." in n or ".output.dense" in n:
            layer = int(n.split(".")[2])
            if layer % 4 == 0:
                used[1, v] = False
    offs, total = gen.packed_offsets(numel, 64)
    flat = [gen.draw_flat_torch(total, r, 0, "f32", DEV) for r in range(W)]
    grads = [[f[o:o + n] for o, n in zip(offs, numel)] for f in flat]
    red = Reducer(numel, "f32", 25 * MIB)
    red.set_option(_lib.OPT_FIND_UNUSED, 1)
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    out_flat = torch.from_numpy(np.full(total, GUARD, np.uint32).view(np.float32)).to(DEV)
    outs = [out_flat[o:o + n] for o, n in zip(offs, numel)]
    red.bind(grads, arena, outs)
    red.set_local_used(used.tolist())
    g = used.any(axis=0)
    red.begin_iteration()
    red.mark_ready_many([v for v in range(P - 1, -1, -1) if g[v]])
    torch.cuda.synchronize()
    assert red.device_status() == 0
    members, locs = assign_buckets(numel, 4, 25 * MIB)
    host = [f.cpu().numpy() for f in flat]
    want_arena, want_outs = reduce_with_unused([[h[o:o + n] for o, n in zip(offs, numel)] for h in host],
                                               used.tolist(), members, locs, numel)
    del host
    got = arena.cpu().numpy()
    assert bits_equal(got, want_arena), first_mismatch(got, want_arena)
    got = out_flat.cpu().numpy()
    for v in range(P):
        n = numel[v]
        if want_outs[0][v] is None:
            assert np.all(got[offs[v]:offs[v] + n].view(np.uint32) == GUARD), v
        else:
            assert bits_equal(got[offs[v]:offs[v] + n], want_outs[0][v]), (v, first_mismatch(got[offs[v]:offs[v] + n], want_outs[0][v]))
    assert not torch.isnan(arena).any()
    red.destroy()


@pytest.mark.parametrize("kernel", ["ldg", "tma", "auto"])
@pytest.mark.parametrize("per_event", [False, True])
def test_unused_more_segments_than_one_launch_holds(kernel, per_event):
    """9,000 small parameters in one bucket with unused tracking on: the
    replicas' local-use masks travel in the launch's parameter block, at
    most 3,840 segments per launch, so the bucket goes out as three chained
    launches; every element and every untouched copy-back against the
    oracle."""
    rng = np.random.default_rng(9000)
    P, W = 9000, 3
    numel = [int(x) for x in rng.integers(0, 41, size=P)]
    used = rng.random((W, P)) < 0.8
    used[:, ::97] = False                 # some unused on every replica
    flats, views, offs = host_grads(numel, W, "f32")
    cap = 64 * MIB
    members, locs = assign_buckets(numel, 4, cap)
    assert len(members) == 1
    want_arena, want_outs = reduce_with_unused(views, used.tolist(), members, locs, numel, n_out=1)
    _, grads_dev = host_to_device_views(flats, numel, offs, "f32", DEV)
    red = _reducer(numel, "f32", cap, kernel)
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    bufs, out_views, out_offs = _guarded_outputs(numel, 1)
    red.bind(grads_dev, arena, out_views[0])
    red.set_local_used(used.tolist())
    red.begin_iteration()
    g = globally_used(used.tolist())
    order = [int(v) for v in rng.permutation(P) if g[v]]
    if per_event:
        for v in order:
            red.mark_ready(v)
    else:
        assert red.mark_ready_many(order) == len(order)
    torch.cuda.synchronize()
    assert red.device_status() == 0
    assert red.launch_count() >= 3
    got = arena.cpu().numpy()
    assert bits_equal(got, want_arena), first_mismatch(got, want_arena)
    _check_outputs(bufs, out_offs, numel, want_outs, used.tolist())
    red.destroy()

