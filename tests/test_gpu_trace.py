"""The launch-trace build (-DDDP_TRACE): the same bits as the release build,
and per CTA four ordered %globaltimer stamps for every launch of the
bulk-copy bucket kernel (entry <= past the wait <= first stage <= last
stage)."""

import os

import numpy as np
import pytest
import torch

from reduction_reducer_gb300 import Reducer, _lib
from reduction_reducer_gb300.reducer import read_launch_trace
from workloads import gen, shapes

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from reduction_reducer_gb300 import build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    if not os.path.exists(_lib.TRACE_LIB_PATH):
        build.build_trace()
    torch.cuda.set_device(0)


def test_release_build_records_no_trace():
    _, _, seq = read_launch_trace(_lib.LIB_PATH)
    assert seq == -1


@pytest.mark.parametrize("mode", ["mark_ready", "mark_ready_many"])
def test_trace_build_stamps_and_bits(mode):
    numel = shapes.numels(shapes.bert_large(layers=2, vocab=4096))
    W, cap = 4, 1 << 20
    offs, total = gen.packed_offsets(numel, 64)
    flat = [gen.draw_flat_torch(total, r, 0, "f32", DEV) for r in range(W)]
    grads = [[f[o:o + n] for o, n in zip(offs, numel)] for f in flat]
    order = gen.reverse_order(len(numel))
    results = []
    for path in (_lib.LIB_PATH, _lib.TRACE_LIB_PATH):
        red = Reducer(numel, "f32", cap, lib_path=path)
        red.set_option(_lib.OPT_KERNEL, _lib.KERNEL_TMA)
        arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
        red.bind(grads, arena, None)
        _, _, seq0 = read_launch_trace(path)
        red.begin_iteration()
        if mode == "mark_ready":
            for v in order:
                red.mark_ready(v)
        else:
            red.mark_ready_many(order)
        torch.cuda.synchronize()
        buf, grid, seq1 = read_launch_trace(path)
        if path == _lib.TRACE_LIB_PATH:
            launches = red.launch_count()
            assert seq1 - seq0 == launches > 1
            for i in range(seq0, seq1):
                slot = i % _lib.TRACE_LAUNCHES
                t = buf[slot, :min(grid[slot], _lib.TRACE_CTAS)].astype(np.int64)
                busy = t[:, 2] > 0                      # CTAs with staged work (idle ones stop after the wait)
                assert np.all(t[:, 0] > 0) and np.all(t[:, 1] >= t[:, 0])
                assert np.all(t[busy, 2] >= t[busy, 1]) and np.all(t[busy, 3] >= t[busy, 2])
        results.append(arena.clone())
        red.destroy()
    assert torch.equal(results[0].view(torch.int32), results[1].view(torch.int32))
