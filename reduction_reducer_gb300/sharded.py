"""The bucket all-reduce across ranks that each hold one replica.

Each rank runs its own reducer (W = 1: its replica's gradients) with a
communication hook from this module.  The library calls the hook for every
launched bucket, in bucket-index order on every rank ("NCCL 专家课程 30",
section "Bucket 必须按序发起"), with the bucket's gradients gathered into a
flat buffer, and copies the hook's result back into the gradients.  The hook
performs the all-reduce as the pages describe it ("PyTorch Distributed
Training Internals", section "3. The All-Reduce Itself"): a reduce-scatter,
after which rank g owns the reduced values of chunk g of the bucket
(``ddp_shard_range``), then an all-gather of the chunks.

The reduce-scatter is exact: an all-to-all moves the replicas' raw values of
each chunk to its owner, and the owner sums them itself in rank order and
scales by fl32(1/G) (``ddp_shard_mean``, the library's kernel), so every rank
ends with the bits the one-GPU pass computes over the same G replicas.

Only plumbing lives here: the exchange runs through ``torch.distributed``
(NCCL between GPUs; any backend with all_to_all_single and
all_gather_into_tensor), the ownership plan and the arithmetic through the C
ABI.
"""

from __future__ import annotations

import ctypes as C

from . import _lib
from .reducer import DTYPES, _check_status, _ptr, _ptr_array


def verify_layout(dist, red, group=None, device=None):
    """Construction check across ranks ("PyTorch Distributed" paper summary:
    the sizes are compared across processes with a MIN and a MAX all-reduce
    before training starts): every rank of ``group`` must hold the same
    bucket layout -- parameter count, dtype, bucket count, arena size and the
    bucket offsets and members -- since the buckets' collectives must pair
    up in bucket order on every rank.  Raises RuntimeError naming what
    differs.  ``device``: where the all-reduced tensor lives (default: cuda
    for the NCCL backend, cpu otherwise)."""
    import hashlib
    import torch
    B, offs = red.get_bucket_info()
    locs = red.get_locators()
    h = hashlib.sha256()
    h.update(",".join(str(x) for x in offs).encode())
    h.update(";".join(f"{b}.{i}.{o}.{n}" for (b, i, o, n) in locs).encode())
    d = h.digest()
    fields = {"parameter count": red.P, "dtype": DTYPES[red.dtype], "bucket count": B, "arena size": int(offs[-1]),
              "layout digest (low)": int.from_bytes(d[:7], "little"),
              "layout digest (high)": int.from_bytes(d[7:14], "little")}
    if device is None:
        device = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    v = torch.tensor(list(fields.values()), dtype=torch.int64, device=device)
    lo, hi = v.clone(), v.clone()
    dist.all_reduce(lo, op=dist.ReduceOp.MIN, group=group)
    dist.all_reduce(hi, op=dist.ReduceOp.MAX, group=group)
    bad = [k for k, a, b in zip(fields, lo.tolist(), hi.tolist()) if a != b]
    if bad:
        raise RuntimeError("the ranks' bucket layouts differ in: " + ", ".join(bad))


def shard_range(n: int, G: int, g: int):
    """(chunk, lo, hi): rank g's part [lo, hi) of a flat range of n elements
    split in chunks of ``chunk`` elements (``ddp_shard_range``)."""
    lib = _lib.load()
    c, lo, hi = C.c_int64(), C.c_int64(), C.c_int64()
    _check_status(lib.ddp_shard_range(int(n), int(G), int(g), C.byref(c), C.byref(lo), C.byref(hi)), None)
    return c.value, lo.value, hi.value


def shard_mean(chunks, out, dtype: str, stream: int):
    """out[i] = rank-order fp32 mean of chunks[c][i] (device tensors or
    addresses, ``out.numel()`` values each) on ``stream``
    (``ddp_shard_mean``)."""
    lib = _lib.load()
    n = out.numel()
    arr = _ptr_array([_ptr(t) for t in chunks])
    _check_status(lib.ddp_shard_mean(len(chunks), DTYPES[dtype], arr, _ptr(out), n, stream), None)


class ShardedAllReduce:
    """The exact reduce-scatter + all-gather of one flat bucket over the
    ranks of ``group`` (every rank holds one replica).

    ``mean(chunks, out)`` is the owner's arithmetic; by default the
    library's ``ddp_shard_mean`` on the current CUDA stream.  Buffers for the
    exchange are allocated once per bucket size and reused.
    """

    def __init__(self, dist, group=None, dtype: str = "f32", mean=None):
        self.dist = dist
        self.group = group
        self.G = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        self.dtype = dtype
        self.mean = mean
        self._bufs = {}

    def _buf(self, key, n, dtype, like):
        t = self._bufs.get(key)
        if t is None or t.numel() < n or t.dtype != dtype or t.device != like.device:
            import torch
            t = torch.empty(n, dtype=dtype, device=like.device)
            self._bufs[key] = t
        return t[:n]

    def __call__(self, local, out):
        """local: this rank's bucket (1-D, gradient dtype); out: fp32 tensor
        of the same length that receives the mean over all ranks."""
        import torch
        n = local.numel()
        G = self.G
        plan = [shard_range(n, G, c) for c in range(G)]
        chunk, lo, hi = plan[self.rank]
        mine_n = hi - lo
        # reduce-scatter, exact: chunk c of the local bucket goes to rank c as
        # it is (uneven splits: the last non-empty chunk is shorter), and this
        # rank receives every replica's values of its own chunk, in rank order
        recv = self._buf("recv", G * mine_n, local.dtype, local)
        self.dist.all_to_all_single(recv, local, output_split_sizes=[mine_n] * G,
                                    input_split_sizes=[h - l for _, l, h in plan], group=self.group)
        mine = self._buf("mine", chunk, torch.float32, local)
        if mine_n > 0:
            parts = [recv[c * mine_n:(c + 1) * mine_n] for c in range(G)]   # replica c's values of my chunk
            if self.mean is not None:
                self.mean(parts, mine[:mine_n])
            else:
                shard_mean(parts, mine[:mine_n], self.dtype, int(torch.cuda.current_stream().cuda_stream))
        if chunk > mine_n:
            mine[mine_n:].zero_()            # padding of a short chunk: gathered, never used
        # all-gather of equal (padded) chunks; they tile [0, n) in rank order
        gathered = self._buf("gathered", G * chunk, torch.float32, local)
        self.dist.all_gather_into_tensor(gathered, mine, group=self.group)
        out.copy_(gathered[:n])


def sharded_hook(dist, replica_buffer, arena, group=None, dtype: str = "f32"):
    """A communication hook (for ``Reducer.register_comm_hook(hook,
    [replica_buffer])`` on a reducer bound with W = 1: this rank's replica)
    that all-reduces every bucket across the ranks of ``group`` with
    ``ShardedAllReduce``.  ``replica_buffer`` is the tensor the bucket's
    gradients lie in -- the registered replica buffer, or, when the hook was
    registered without one, the flat gradient tensor whose views in bucket
    order the reducer was bound to -- and ``arena`` the bucket arena the
    reducer reduces into.  The hook runs its exchange on the library's
    stream; a bucket of another replica count fails the launch (HookError)."""
    import torch
    reduce = ShardedAllReduce(dist, group, dtype)
    esz = replica_buffer.element_size()

    def hook(bucket, stream):
        if bucket.W != 1:
            return 1                          # one replica per rank: the others are the other ranks'
        n = int(bucket.numel)
        if n == 0:
            return 0
        at = (int(bucket.replicas[0]) - replica_buffer.data_ptr()) // esz
        res = (int(bucket.result) - arena.data_ptr()) // 4
        st = torch.cuda.ExternalStream(int(stream), device=arena.device) if stream else \
            torch.cuda.default_stream(arena.device)
        with torch.cuda.stream(st):
            reduce(replica_buffer[at:at + n], arena[res:res + n])
        return 0
    return hook
