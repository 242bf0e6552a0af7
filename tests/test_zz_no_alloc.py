"""The no-allocation entry point, checked against the ordinary one and
against the oracle.

``ddp_reduce_all_noalloc`` serves callers that may not call cudaMalloc (a
framework whose caching allocator owns the device memory budget, real-time
loops where an allocation and the device synchronisation it implies are not
allowed): its segment table lives in the library's static device scratch
instead of memory allocated by ddp_bind.  Here it must give bit for bit what
``ddp_reduce_all`` on a bound context gives, and what the CPU oracle computes
from the same inputs, on two calls in a row (the second with other inputs
and another layout, so nothing of the first call's table leaks into it), and
it must refuse a layout whose table does not fit the scratch.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test; it also passes on its own in a
fresh process.
"""

import numpy as np
import pytest
import torch

from oracle.buckets import assign_buckets
from oracle.reduce import reduce_buckets
from reduction_reducer_gb300 import InvalidArg, Reducer
from workloads import gen, shapes

pytestmark = pytest.mark.gpu

MIB = 1 << 20


@pytest.fixture(scope="module", autouse=True)
def _built():
    import os
    from reduction_reducer_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    _lib.load()
    torch.cuda.set_device(0)


def _case(numel, W, dtype, cap, n_out, seed_step):
    offs, total = gen.packed_offsets(numel, 64)
    flat = [gen.draw_flat_torch(total, r, seed_step, dtype, "cuda") for r in range(W)]
    grads = [[f[o:o + n] for o, n in zip(offs, numel)] for f in flat]
    red = Reducer(numel, dtype, cap)
    N = red.arena_numel()

    def outputs():
        arena = torch.full((N,), float("nan"), device="cuda")
        copies = [[torch.full((n,), float("nan"), device="cuda") for n in numel] for _ in range(n_out)]
        go = None if n_out == 0 else (copies[0] if n_out == 1 else copies)
        return arena, copies, go

    # the ordinary entry point: bind + reduce_all
    ref_arena, ref_copies, ref_go = outputs()
    red.bind(grads, ref_arena, ref_go)
    red.reduce_all()
    # the no-allocation entry point on the same inputs
    arena, copies, go = outputs()
    red.reduce_all_noalloc(grads, arena, go)
    torch.cuda.synchronize()
    assert torch.equal(arena.view(torch.int32), ref_arena.view(torch.int32))
    for o in range(n_out):
        for v in range(len(numel)):
            assert torch.equal(copies[o][v].view(torch.int32), ref_copies[o][v].view(torch.int32)), (o, v)
    assert not torch.isnan(arena).any()
    # and against the oracle on the same inputs, read back from the device
    host = [f.view(torch.int16).cpu().numpy().view(np.uint16) if dtype == "bf16" else f.cpu().numpy() for f in flat]
    members, locs = assign_buckets(numel, 4 if dtype == "f32" else 2, cap)
    want_arena, want_outs = reduce_buckets([[h[o:o + n] for o, n in zip(offs, numel)] for h in host],
                                           members, locs, numel)
    assert np.array_equal(arena.cpu().numpy().view(np.uint32), want_arena.view(np.uint32))
    for o in range(n_out):
        for v in range(len(numel)):
            assert np.array_equal(copies[o][v].cpu().numpy().view(np.uint32), want_outs[0][v].view(np.uint32)), (o, v)
    red.destroy()


def test_noalloc_matches_reduce_all_two_calls():
    # call 1: BERT-shaped (3 layers), W = 4 fp32, one copy-back
    _case(shapes.numels(shapes.bert_large(layers=3, vocab=4096)), 4, "f32", 2 * MIB, 1, seed_step=0)
    # call 2: other inputs, other layout: GPT-2-shaped bf16, W = 8, every replica's copy
    _case(shapes.numels(shapes.gpt2_medium(layers=2, vocab=3000, n_ctx=256)), 8, "bf16", 1 * MIB, 8, seed_step=1)


def test_noalloc_rejects_oversized_table():
    numel = [4] * 4000                      # 4000 segments x (8 + 8*16 + 8*16 + 4) bytes > 256 KiB
    red = Reducer(numel, "f32", 0)
    z = torch.zeros(16, device="cuda")
    grads = [[z[:4]] * len(numel) for _ in range(16)]
    arena = torch.zeros(red.arena_numel(), device="cuda")
    with pytest.raises(InvalidArg) as ei:
        red.reduce_all_noalloc(grads, arena, [[z[:4]] * len(numel) for _ in range(16)])
    assert "static scratch" in str(ei.value)
