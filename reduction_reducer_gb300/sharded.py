"""The bucket all-reduce across ranks that each hold some of the replicas.

Each rank runs its own reducer over the replicas it holds (Wl of them, the
same number on every rank; Wl = 1 when every rank holds one) with a
communication hook from this module.  The library calls the hook for every
launched bucket, in bucket-index order on every rank ("NCCL 专家课程 30",
section "Bucket 必须按序发起"), with the bucket's gradients gathered into
flat buffers, and copies the hook's result back into the gradients.  The
hook performs the all-reduce as the pages describe it ("PyTorch Distributed
Training Internals", section "3. The All-Reduce Itself"): a reduce-scatter,
after which rank g owns the reduced values of chunk g of the bucket
(``ddp_shard_range``), then an all-gather of the chunks.

The reduce-scatter is exact: all-to-alls move the replicas' raw values of
each chunk to its owner, and the owner sums them itself in global replica
order (rank g's replica r is replica g*Wl + r) and scales by fl32(1/W),
W = G*Wl (``ddp_shard_mean``, the library's kernel), so every rank ends with
the bits the one-GPU pass computes over the same W replicas.

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
    bucket offsets and members -- and, once bound, the same number of
    replicas, since the buckets' collectives must pair up in bucket order on
    every rank and carry equal shares (so call it at the same point on every
    rank: before ``bind`` everywhere or after it everywhere).  Raises
    RuntimeError naming what differs.  ``device``: where the all-reduced
    tensor lives (default: cuda for the NCCL backend, cpu otherwise)."""
    import hashlib
    import torch
    B, offs = red.get_bucket_info()
    locs = red.get_locators()
    h = hashlib.sha256()
    h.update(",".join(str(x) for x in offs).encode())
    h.update(";".join(f"{b}.{i}.{o}.{n}" for (b, i, o, n) in locs).encode())
    d = h.digest()
    fields = {"parameter count": red.P, "dtype": DTYPES[red.dtype], "bucket count": B, "arena size": int(offs[-1]),
              "replicas per rank": int(getattr(red, "W", 0)),
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
    """out[i] = fp32 mean of chunks[c][i] in the order of ``chunks`` (device
    tensors or addresses, ``out.numel()`` values each, at most 64 of them) on
    ``stream`` (``ddp_shard_mean``)."""
    lib = _lib.load()
    n = out.numel()
    arr = _ptr_array([_ptr(t) for t in chunks])
    _check_status(lib.ddp_shard_mean(len(chunks), DTYPES[dtype], arr, _ptr(out), n, stream), None)


class ShardedAllReduce:
    """The exact reduce-scatter + all-gather of one flat bucket over the
    ranks of ``group``, every rank holding the same number Wl of replicas
    (G*Wl <= 64).

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
        self._plans = {}

    def _plan(self, n):
        """Every rank's (chunk, lo, hi) for a bucket of n elements, cached
        per length (a layout has few distinct bucket lengths)."""
        p = self._plans.get(n)
        if p is None:
            p = [shard_range(n, self.G, c) for c in range(self.G)]
            self._plans[n] = p
        return p

    def _buf(self, key, n, dtype, like):
        t = self._bufs.get(key)
        if t is None or t.numel() < n or t.dtype != dtype or t.device != like.device:
            import torch
            t = torch.empty(n, dtype=dtype, device=like.device)
            self._bufs[key] = t
        return t[:n]

    def __call__(self, local, out):
        """local: this rank's bucket, one 1-D tensor of the gradient dtype
        (one replica per rank) or a list of the Wl replicas' buckets, each of
        the same length; out: fp32 tensor of that length that receives the
        mean over all G*Wl replicas in global replica order."""
        import torch
        reps = [local] if torch.is_tensor(local) else list(local)
        Wl = len(reps)
        G = self.G
        if Wl < 1 or G * Wl > 64:
            raise ValueError(f"{G} ranks x {Wl} replicas: between 1 and 64 replicas in all")
        n = reps[0].numel()
        if any(t.numel() != n for t in reps) or out.numel() != n:
            raise ValueError("the replicas' buckets and the output differ in length")
        plan = self._plan(n)
        chunk, lo, hi = plan[self.rank]
        mine_n = hi - lo
        splits = [h - l for _, l, h in plan]
        # reduce-scatter, exact: chunk c of each local replica's bucket goes to
        # rank c as it is (uneven splits: the last non-empty chunk is
        # shorter), and this rank receives every rank's values of its own
        # chunk, rank after rank; one all-to-all per local replica
        recv = []
        for r, t in enumerate(reps):
            buf = self._buf(("recv", r), G * mine_n, t.dtype, t)
            self.dist.all_to_all_single(buf, t, output_split_sizes=[mine_n] * G,
                                        input_split_sizes=splits, group=self.group)
            recv.append(buf)
        mine = self._buf("mine", chunk, torch.float32, reps[0])
        if mine_n > 0:
            # replica g*Wl + r is rank g's replica r: the one-GPU pass's order
            parts = [recv[r][g * mine_n:(g + 1) * mine_n] for g in range(G) for r in range(Wl)]
            if self.mean is not None:
                self.mean(parts, mine[:mine_n])
            else:
                shard_mean(parts, mine[:mine_n], self.dtype, int(torch.cuda.current_stream().cuda_stream))
        if chunk > mine_n:
            mine[mine_n:].zero_()            # padding of a short chunk: gathered, never used
        # all-gather of equal (padded) chunks; they tile [0, n) in rank order,
        # straight into the output when no chunk is padded
        if G * chunk == n and out.is_contiguous():
            self.dist.all_gather_into_tensor(out, mine, group=self.group)
        else:
            gathered = self._buf("gathered", G * chunk, torch.float32, reps[0])
            self.dist.all_gather_into_tensor(gathered, mine, group=self.group)
            out.copy_(gathered[:n])


def sharded_hook(dist, replica_buffers, arena, group=None, dtype: str = "f32"):
    """A communication hook (for ``Reducer.register_comm_hook(hook,
    replica_buffers)`` on a reducer bound with this rank's Wl replicas) that
    all-reduces every bucket across the ranks of ``group`` with
    ``ShardedAllReduce``.  ``replica_buffers``: the tensor (Wl = 1) or the Wl
    tensors the buckets' gradients lie in, replica by replica -- the
    registered replica buffers, or, when the hook was registered without
    them, the flat gradient tensors whose views in bucket order the reducer
    was bound to -- and ``arena`` the bucket arena the reducer reduces into.
    The hook runs its exchange on the library's stream; a bucket of another
    replica count fails the launch (HookError)."""
    import torch
    bufs = [replica_buffers] if torch.is_tensor(replica_buffers) else list(replica_buffers)
    reduce = ShardedAllReduce(dist, group, dtype)
    Wl = len(bufs)

    streams = {}

    def hook(bucket, stream):
        if bucket.W != Wl:
            return 1                          # every rank holds Wl replicas; the others are the other ranks'
        n = int(bucket.numel)
        if n == 0:
            return 0
        local = []
        for r, t in enumerate(bufs):
            at = (int(bucket.replicas[r]) - t.data_ptr()) // t.element_size()
            local.append(t[at:at + n])
        res = (int(bucket.result) - arena.data_ptr()) // 4
        key = int(stream or 0)
        st = streams.get(key)
        if st is None:
            st = torch.cuda.ExternalStream(key, device=arena.device) if key else torch.cuda.default_stream(arena.device)
            streams[key] = st
        with torch.cuda.stream(st):
            reduce(local, arena[res:res + n])
        return 0
    return hook
