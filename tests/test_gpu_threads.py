"""Separate contexts driven from separate host threads at the same time.

A context is not thread-safe, but distinct contexts are independent: the
launch parameter blocks the host core fills are per thread and the
shared-memory attribute cache is locked.  Four threads, each with its own
context, stream and workload (different W, dtype, kernel, path), run several
iterations concurrently; every result must equal the oracle bit for bit.
"""

import threading

import numpy as np
import pytest
import torch

from oracle.buckets import assign_buckets
from oracle.nosync import accumulate_steps
from oracle.reduce import reduce_buckets
from oracle.unused import reduce_with_unused
from reduction_reducer_gb300 import Reducer, _lib
from workloads import gen

from gpu_util import bits_equal, first_mismatch, host_grads, host_to_device_views

pytestmark = pytest.mark.gpu

DEV = "cuda"
RAGGED = [0, 1, 2, 3, 5, 7, 8, 13, 64, 67, 100, 1000, 4095, 4097, 70001, 0, 9, 300007, 16, 31]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import os
    from reduction_reducer_gb300 import build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    _lib.load()
    torch.cuda.set_device(0)


def _plain(W, dtype, kernel, iters):
    numel = RAGGED
    cap = 16 * 1024
    flats, views, offs = host_grads(numel, W, dtype, special=True)
    members, locs = assign_buckets(numel, 4 if dtype == "f32" else 2, cap)
    want, _ = reduce_buckets(views, members, locs, numel)
    _, grads = host_to_device_views(flats, numel, offs, dtype, DEV)
    red = Reducer(numel, dtype, cap)
    red.set_option(_lib.OPT_KERNEL, kernel)
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    red.bind(grads, arena, [torch.zeros(n, device=DEV) for n in numel])
    order = gen.straggler_order(members, p=0.5, seed=W)

    def run(stream):
        for _ in range(iters):
            red.begin_iteration()
            red.mark_ready_many(order, stream)
    return red, run, lambda: (arena, want)


def _nosync(W, kernel, iters):
    numel = RAGGED
    K, cap = 3, 16 * 1024
    steps = [host_grads(numel, W, "f32", step=k) for k in range(K)]
    offs = steps[0][2]
    acc_np = [accumulate_steps([steps[k][1][r] for k in range(K)]) for r in range(W)]
    members, locs = assign_buckets(numel, 4, cap)
    want, _ = reduce_buckets(acc_np, members, locs, numel)
    dev = [host_to_device_views(steps[k][0], numel, offs, "f32", DEV)[1] for k in range(K)]
    acc = [[torch.empty(n, device=DEV) for n in numel] for _ in range(W)]
    red = Reducer(numel, "f32", cap)
    red.set_option(_lib.OPT_KERNEL, kernel)
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    red.bind(acc, arena, None)

    def run(stream):
        for _ in range(iters):
            for k in range(K):
                red.accumulate_nosync(acc, dev[k], first_step=(k == 0), stream=stream)
            red.begin_iteration()
            red.reduce_all(stream)
    return red, run, lambda: (arena, want)


def _unused(W, kernel, iters):
    numel = RAGGED
    cap = 16 * 1024
    rng = np.random.default_rng(W)
    used = rng.random((W, len(numel))) < 0.6
    used[:, 10] = True
    flats, views, offs = host_grads(numel, W, "f32")
    members, locs = assign_buckets(numel, 4, cap)
    want, _ = reduce_with_unused(views, used.tolist(), members, locs, numel)
    _, grads = host_to_device_views(flats, numel, offs, "f32", DEV)
    red = Reducer(numel, "f32", cap)
    red.set_option(_lib.OPT_KERNEL, kernel)
    red.set_option(_lib.OPT_FIND_UNUSED, 1)
    arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
    red.bind(grads, arena, None)
    g = used.any(axis=0)
    order = [v for v in range(len(numel) - 1, -1, -1) if g[v]]
    bits = red.bits(used.tolist())

    def run(stream):
        for _ in range(iters):
            red.set_local_used(bits)
            red.begin_iteration()
            red.mark_ready_many(order, stream)
    return red, run, lambda: (arena, want)


def test_four_contexts_on_four_threads():
    cases = [_plain(4, "f32", _lib.KERNEL_TMA, 6), _plain(8, "bf16", _lib.KERNEL_LDG, 6),
             _nosync(3, _lib.KERNEL_TMA, 3), _unused(5, _lib.KERNEL_LDG, 6)]
    torch.cuda.synchronize()
    errors = []
    start = threading.Barrier(len(cases))

    def worker(run):
        try:
            torch.cuda.set_device(0)
            stream = torch.cuda.Stream()
            start.wait()
            run(stream)
            stream.synchronize()
        except Exception as ex:      # noqa: BLE001 -- reported below
            errors.append(repr(ex))

    threads = [threading.Thread(target=worker, args=(run,), daemon=True) for _, run, _ in cases]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads)
    assert not errors, errors
    torch.cuda.synchronize()
    for red, _, result in cases:
        arena, want = result()
        got = arena.cpu().numpy()
        assert bits_equal(got, want), first_mismatch(got, want)
        assert red.device_status() == 0
        red.destroy()
