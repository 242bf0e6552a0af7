"""The bucket all-reduce across ranks that each hold some of the replicas, on the CPU.

* the ownership plan (``ddp_shard_range``, host arithmetic of the library):
  the chunks of a flat range tile it in rank order, start 16-byte aligned
  for fp32 and bf16, are equal but for the last non-empty one, and differ
  from the ideal 1/G share by less than one alignment unit;
* the exchange (``reduction_reducer_gb300.sharded.ShardedAllReduce``) over
  ``gloo`` with world sizes 2 and 3: every rank holds one or two replicas of
  a ragged model, all-reduces its buckets in bucket-index order (all-to-alls
  of the raw chunks, the owner's mean in global replica order, all-gather),
  and must end with the oracle's unsharded mean over all the replicas, bit
  for bit.  The owner's arithmetic, a CUDA kernel in the library, is stood
  in for here by the oracle's mean (this test covers the plan and the
  exchange; the GPU tests cover the kernel).
"""

import os
import socket

import numpy as np
import pytest
import torch

from oracle.buckets import assign_buckets
from oracle.hooks import gather_buckets
from oracle.reduce import reduce_buckets, replica_mean
from workloads import gen


@pytest.fixture(scope="module")
def built():
    from reduction_reducer_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib.load()


@pytest.mark.parametrize("G", [1, 2, 3, 4, 5, 8, 16, 33, 64])
def test_chunks_tile_the_range(built, G):
    from reduction_reducer_gb300.sharded import shard_range
    for n in [0, 1, 2, 7, 8, 9, 15, 16, 17, 63, 64, 65, 100, 1000, 4097, 70001, 25 << 18, (1 << 31) + 37]:
        at = 0
        sizes = []
        for g in range(G):
            c, lo, hi = shard_range(n, G, g)
            assert c % 8 == 0 and (n == 0 or c > 0)
            assert lo == at and lo <= hi <= n                  # in rank order, no gap, no overlap
            assert lo % 8 == 0 or lo == n                      # 16-byte aligned starts
            assert n == 0 or c * G >= n                        # G chunks cover the range
            assert c - 8 < -(-n // G) <= c or n == 0           # the ideal share, rounded up to 8
            sizes.append(hi - lo)
            at = hi
        assert at == n
        nonempty = [s for s in sizes if s]
        assert all(s == c for s in nonempty[:-1])            # equal but for the last non-empty chunk


def test_bad_arguments(built):
    import ctypes as C
    from reduction_reducer_gb300 import InvalidArg
    from reduction_reducer_gb300.sharded import shard_range
    for args in [(-1, 2, 0), (10, 0, 0), (10, 2, 2), (10, 2, -1)]:
        with pytest.raises(InvalidArg):
            shard_range(*args)
    assert built.ddp_shard_range(10, 2, 1, None, None, None) == 0
    assert built.ddp_shard_mean(0, 0, None, None, 4, None) == -1      # G < 1
    assert built.ddp_shard_mean(65, 0, None, None, 4, None) == -1     # G > 64
    assert built.ddp_shard_mean(2, 7, None, None, 4, None) == -1      # dtype
    assert built.ddp_shard_mean(2, 0, None, None, 0, None) == 0       # nothing to do
    assert built.ddp_shard_mean(2, 0, (C.c_void_p * 2)(None, None), None, 4, None) == -1


RAGGED = [0, 1, 2, 3, 5, 7, 8, 13, 64, 67, 100, 1000, 4095, 4097, 7001, 0, 9, 30007, 16, 31]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _to_np(t, dtype):
    return t.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else t.numpy()


def _rank(rank, world, port, dtype, cap, Wl):
    import torch.distributed as dist
    from reduction_reducer_gb300.sharded import ShardedAllReduce
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elem = 4 if dtype == "f32" else 2
        members, locs = assign_buckets(RAGGED, elem, cap)
        # every replica's gradients (seeded per replica); rank g holds replicas
        # g*Wl ... g*Wl + Wl - 1
        offs, total = gen.packed_offsets(RAGGED, 1)
        grads = []
        for r in range(world * Wl):
            flat = gen.draw_flat_np(total, r, 0, dtype)
            grads.append([flat[o:o + n] for o, n in zip(offs, RAGGED)])
        want_arena, _ = reduce_buckets(grads, members, locs, RAGGED)
        mine = gather_buckets(grads[rank * Wl:(rank + 1) * Wl], members, locs, RAGGED)

        def oracle_mean(parts, out):
            out.copy_(torch.from_numpy(replica_mean([_to_np(p, dtype) for p in parts])))

        from reduction_reducer_gb300 import Reducer
        from reduction_reducer_gb300.sharded import verify_layout
        verify_layout(dist, Reducer(RAGGED, dtype, cap))            # the same layout on every rank
        reduce = ShardedAllReduce(dist, None, dtype, mean=oracle_mean)
        lens = [sum(RAGGED[v] for v in m) for m in members]
        starts = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        if world == 2 and cap == 0:      # buckets gathered straight into the output and through padding
            assert any(n and n % 16 == 0 for n in lens) and any(n % 16 for n in lens)
        for b in range(len(members)):            # bucket-index order on every rank
            local = [torch.from_numpy(m[b].view(np.int16)).view(torch.bfloat16) if dtype == "bf16"
                     else torch.from_numpy(m[b].copy()) for m in mine]
            out = torch.full((lens[b],), float("nan"))
            reduce(local[0] if Wl == 1 else local, out)
            got = out.numpy()
            want = want_arena[starts[b]:starts[b + 1]]
            assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (rank, b)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,dtype,cap,Wl", [(2, "f32", 16 * 1024, 1), (3, "bf16", 8 * 1024, 1), (3, "f32", 0, 1),
                                               (2, "f32", 0, 1), (2, "f32", 16 * 1024, 2), (3, "f32", 8 * 1024, 2),
                                               (3, "bf16", 0, 2)])
def test_sharded_allreduce_gloo_equals_unsharded_oracle(built, world, dtype, cap, Wl):
    import torch.multiprocessing as mp
    mp.start_processes(_rank, args=(world, _free_port(), dtype, cap, Wl), nprocs=world, join=True,
                       start_method="spawn")


def _rank_mismatch(rank, world, port):
    import torch.distributed as dist
    from reduction_reducer_gb300 import Reducer
    from reduction_reducer_gb300.sharded import verify_layout
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cap = 16 * 1024 if rank == 0 else 0                       # rank 1: one bucket per tensor
        with pytest.raises(RuntimeError, match="bucket count"):
            verify_layout(dist, Reducer(RAGGED, "f32", cap))
        numel = list(RAGGED)
        if rank == 1:
            numel[4], numel[5] = numel[5], numel[4]              # same sizes, other order: same count and arena
        with pytest.raises(RuntimeError, match="layout digest"):
            verify_layout(dist, Reducer(numel, "f32", 16 * 1024))
        red = Reducer(RAGGED, "f32", 16 * 1024)
        red.W = 1 + rank                  # as bound with one replica on rank 0 and two on rank 1
        with pytest.raises(RuntimeError, match="replicas per rank"):
            verify_layout(dist, red)
    finally:
        dist.destroy_process_group()


def test_layouts_that_differ_across_ranks_are_refused(built):
    """The construction check: a MIN and a MAX all-reduce of each rank's
    layout summary; every rank raises when one rank's buckets, or the number
    of replicas it holds, differ."""
    import torch.multiprocessing as mp
    mp.start_processes(_rank_mismatch, args=(2, _free_port()), nprocs=2, join=True, start_method="spawn")
