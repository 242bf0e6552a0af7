"""GPU side of the bucket all-reduce across ranks that each hold some of the replicas.

* ``ddp_shard_mean`` (the owner's mean of the replicas' chunks, in their
  order) against the oracle's mean, bit for bit, for up to 64 chunks, fp32
  and bf16, aligned and unaligned chunk pointers, ragged lengths, special
  values;
* the whole path through a reducer (Wl = 1 or 2 replicas per rank, the
  sharded hook) with a real NCCL process group: on this one-GPU machine the
  group has one rank, so the exchange is NCCL's all-to-all and all-gather
  with itself and the result is the mean of the rank's own replicas,
  against the oracle;
* the whole path with G = 2, 3 and 4 ranks as host threads on the one GPU
  (one or two replicas each).  Larger groups of processes run on the CPU
  over gloo (``tests/test_shard_plan.py``).
"""

import numpy as np
import pytest
import torch

from oracle.buckets import assign_buckets
from oracle.reduce import reduce_buckets, replica_mean
from reduction_reducer_gb300 import Reducer, _lib
from workloads import gen, shapes

from gpu_util import bits_equal, first_mismatch, host_grads, host_to_device_views

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import os
    from reduction_reducer_gb300 import build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    _lib.load()
    torch.cuda.set_device(0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("G", [1, 2, 3, 4, 8, 16, 33, 64])
def test_shard_mean_equals_oracle(G, dtype):
    from reduction_reducer_gb300.sharded import shard_mean
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    for n, shift in [(1, 0), (7, 0), (4096, 0), (70001, 0), (70001, 3), (300007, 1)]:
        # one receive buffer of G chunks, as the all-to-all leaves it; shift
        # moves every chunk off its 16-byte boundary
        chunk = -(-n // 8) * 8 + shift
        xs = [gen.draw_flat_np(n, c, 5, dtype) for c in range(G)]
        if dtype == "f32" and G >= 4 and n >= 8:       # signed zeros, infinities, NaN, a subnormal, overflow
            xs[1][:8] = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 2.0 ** -149, 3.4e38, -1.0], np.float32)
            xs[2][:8] = np.array([-0.0, -0.0, 1.0, np.inf, 1.0, 2.0 ** -149, 3.4e38, 1.0], np.float32)
        flat = np.zeros(G * chunk + shift, xs[0].dtype)
        for c in range(G):
            flat[shift + c * chunk:shift + c * chunk + n] = xs[c]
        dev = torch.from_numpy(flat.view(np.int16)).to(DEV).view(tdt) if dtype == "bf16" else torch.from_numpy(flat).to(DEV)
        parts = [dev[shift + c * chunk:shift + c * chunk + n] for c in range(G)]
        out = torch.full((n,), float("nan"), device=DEV)
        shard_mean(parts, out, dtype, int(torch.cuda.current_stream().cuda_stream))
        torch.cuda.synchronize()
        want = replica_mean(xs)
        got = out.cpu().numpy()
        assert bits_equal(got, want), (n, shift, first_mismatch(got, want))


@pytest.mark.parametrize("Wl", [1, 2])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_sharded_hook_nccl_single_rank(dtype, Wl):
    """A reducer with the sharded hook in a one-rank NCCL group: every bucket
    goes through the hook (all-to-all per replica, owner mean, all-gather)
    and the library's copy-back, in bucket order; the result is the oracle's
    mean of the rank's Wl replicas."""
    import torch.distributed as dist
    from reduction_reducer_gb300.sharded import sharded_hook
    numel = shapes.numels(shapes.bert_large(layers=2, vocab=2048))
    cap = 1 << 20
    store = dist.HashStore()
    dist.init_process_group("nccl", store=store, rank=0, world_size=1, device_id=torch.device(DEV, 0))
    try:
        flats, views, offs = host_grads(numel, Wl, dtype)
        _, grads_dev = host_to_device_views(flats, numel, offs, dtype, DEV)
        red = Reducer(numel, dtype, cap)
        arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
        outs = [torch.full((n,), float("nan"), device=DEV) for n in numel]
        red.bind(grads_dev, arena, outs)
        tdt = torch.float32 if dtype == "f32" else torch.bfloat16
        rbs = [torch.empty(red.arena_numel(), dtype=tdt, device=DEV) for _ in range(Wl)]
        red.register_comm_hook(sharded_hook(dist, rbs[0] if Wl == 1 else rbs, arena, dtype=dtype), rbs)
        s = torch.cuda.Stream()
        for _ in range(2):
            red.begin_iteration()
            red.mark_ready_many(gen.reverse_order(len(numel)), s)
        torch.cuda.synchronize()
        members, locs = assign_buckets(numel, 4 if dtype == "f32" else 2, cap)
        want_arena, want_outs = reduce_buckets(views, members, locs, numel)
        got = arena.cpu().numpy()
        assert bits_equal(got, want_arena), first_mismatch(got, want_arena)
        for v in range(len(numel)):
            assert bits_equal(outs[v].cpu().numpy(), want_outs[0][v]), v
        red.destroy()
    finally:
        dist.destroy_process_group()


class _ThreadGroup:
    """G ranks of one process, one host thread each, on this GPU: the two
    collectives the sharded all-reduce uses, exchanged through host-side
    slots between barriers (no kernel waits for another)."""

    def __init__(self, G):
        import threading
        self.G = G
        self.barrier = threading.Barrier(G, timeout=60)
        self.slots = [None] * G

    def member(self, rank):
        grp = self

        class _Dist:
            def get_world_size(self, group=None):
                return grp.G

            def get_rank(self, group=None):
                return rank

            def _publish(self, value):
                torch.cuda.synchronize()          # what this rank enqueued is done before others read it
                grp.slots[rank] = value
                grp.barrier.wait()

            def all_to_all_single(self, out, inp, output_split_sizes=None, input_split_sizes=None, group=None):
                self._publish(torch.split(inp, input_split_sizes))
                out.copy_(torch.cat([grp.slots[c][rank] for c in range(grp.G)]))
                torch.cuda.synchronize()
                grp.barrier.wait()                # slots are reused by the next collective

            def all_gather_into_tensor(self, out, inp, group=None):
                self._publish(inp)
                out.copy_(torch.cat([grp.slots[c] for c in range(grp.G)]))
                torch.cuda.synchronize()
                grp.barrier.wait()

            ReduceOp = torch.distributed.ReduceOp

            def all_reduce(self, t, op=None, group=None):
                self._publish(t.clone())
                stack = torch.stack([grp.slots[c] for c in range(grp.G)])
                t.copy_(stack.min(0).values if op == torch.distributed.ReduceOp.MIN else stack.max(0).values)
                grp.barrier.wait()
        return _Dist()


@pytest.mark.parametrize("G,dtype,cap,Wl", [(2, "f32", 1 << 20, 1), (3, "bf16", 1 << 19, 1), (4, "f32", 0, 1),
                                            (2, "f32", 1 << 20, 2), (3, "f32", 1 << 19, 2), (4, "bf16", 0, 2)])
def test_sharded_hook_thread_ranks_on_one_gpu(G, dtype, cap, Wl):
    """G ranks as host threads, each with its own reducer over its Wl
    replicas (rank g holds replicas g*Wl ... g*Wl + Wl - 1) and the sharded
    hook: every bucket goes through gather, the all-to-alls of raw chunks,
    the owner's mean (the library's kernel), the all-gather and the
    copy-back, in bucket order on every rank; every rank's arena and
    copied-back gradients equal the oracle's mean over the G*Wl replicas bit
    for bit."""
    import threading
    from reduction_reducer_gb300.sharded import sharded_hook, verify_layout
    numel = [0, 1, 2, 3, 5, 7, 8, 13, 64, 67, 100, 1000, 4095, 4097, 70001, 0, 9, 300007, 16, 31, 123457]
    flats, views, offs = host_grads(numel, G * Wl, dtype)
    members, locs = assign_buckets(numel, 4 if dtype == "f32" else 2, cap)
    want_arena, want_outs = reduce_buckets(views, members, locs, numel)
    grp = _ThreadGroup(G)
    results, errors = [None] * G, []

    def rank_main(r):
        try:
            torch.cuda.set_device(0)
            _, grads_dev = host_to_device_views(flats[r * Wl:(r + 1) * Wl], numel, offs, dtype, DEV)
            red = Reducer(numel, dtype, cap)
            arena = torch.full((red.arena_numel(),), float("nan"), device=DEV)
            outs = [torch.full((n,), float("nan"), device=DEV) for n in numel]
            red.bind(grads_dev, arena, outs)
            tdt = torch.float32 if dtype == "f32" else torch.bfloat16
            rbs = [torch.empty(max(red.arena_numel(), 1), dtype=tdt, device=DEV) for _ in range(Wl)]
            verify_layout(grp.member(r), red, device=DEV)
            red.register_comm_hook(sharded_hook(grp.member(r), rbs if Wl > 1 else rbs[0], arena, dtype=dtype), rbs)
            for _ in range(2):
                red.begin_iteration()
                red.mark_ready_many(gen.reverse_order(len(numel)))
            torch.cuda.synchronize()
            results[r] = (arena.cpu().numpy(), [o.cpu().numpy() for o in outs])
            red.destroy()
        except Exception as exc:      # noqa: BLE001 -- reported by the main thread
            errors.append((r, repr(exc)))
            grp.barrier.abort()

    threads = [threading.Thread(target=rank_main, args=(r,)) for r in range(G)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    for r in range(G):
        arena, outs = results[r]
        assert bits_equal(arena, want_arena), (r, first_mismatch(arena, want_arena))
        for v in range(len(numel)):
            assert bits_equal(outs[v], want_outs[0][v]), (r, v)
