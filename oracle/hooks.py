"""Oracle: bucket reduction through a communication hook.

Test infrastructure only; see the package docstring.

What the pages fix ("Distributed Data Parallel" notes, "Custom gradient
aggregation"; "NCCL 专家课程 30", section "从 Bucket 到 AllReduce Future"):

* a hook receives every ready bucket as a GradBucket -- its index, the
  number of buckets, whether it is the last, the flat bucket buffer and the
  per-parameter views (offsets, lengths) -- and produces the bucket's reduced
  value, which is copied back into the parameters' gradients;
* the default hook divides by the world size and all-reduces, so the result
  is the mean over the replicas; a hook owns its averaging ("forgetting to
  divide by the world size is a common silent bug").

Readings: each replica's bucket buffer is its gradients gathered into the
bucket layout (the copy into the bucket view); the built-in default hook
computes the same rank-order fp32 mean as the fused pass; the built-in
compression hook (the pages name gradient compression only as a future
direction) rounds each replica's bucket to bf16 (round to nearest even)
before that same mean, i.e. it averages what a bf16 wire would carry.
"""

from __future__ import annotations

import numpy as np

from .reduce import replica_mean, widen


def gather_buckets(grads, members, locators, numel):
    """Per replica, per bucket: the flat bucket buffer (the gradients copied
    into their views, in the gradient dtype)."""
    W = len(grads)
    out = []
    for r in range(W):
        per_bucket = []
        for b, vs in enumerate(members):
            n = sum(int(numel[v]) for v in vs)
            dt = grads[r][vs[0]].dtype if vs else np.float32
            buf = np.zeros(n, dtype=dt)
            for v in vs:
                lo = locators[v].offset
                buf[lo:lo + numel[v]] = grads[r][v]
            per_bucket.append(buf)
        out.append(per_bucket)
    return out


def f32_to_bf16_rne(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (as uint16 bits), round to nearest even; NaN stays NaN."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = ((u[nan] >> np.uint64(16)) | np.uint64(0x40)).astype(np.uint16)
    return r


def hook_mean(replica_buffers):
    """The default hook: rank-order fp32 mean of the replicas' buffers."""
    return replica_mean(replica_buffers)


def hook_bf16_compress(replica_buffers):
    """Compression hook: each replica's buffer rounded to bf16, then the mean."""
    return replica_mean([f32_to_bf16_rne(widen(x)) for x in replica_buffers])


def reduce_with_hook(grads, members, locators, numel, hook, n_out: int = 1):
    """Gather, hook per bucket in index order, copy-back.  Returns
    ``(arena, outs, calls)``; ``calls`` lists (index, num_buckets, is_last)."""
    bufs = gather_buckets(grads, members, locators, numel)
    B = len(members)
    lens = [sum(int(numel[v]) for v in vs) for vs in members]
    starts = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64) if B else np.zeros(1, np.int64)
    arena = np.full(int(starts[-1]), np.nan, dtype=np.float32)
    outs = [[None] * len(numel) for _ in range(n_out)]
    calls = []
    for b in range(B):
        result = hook([bufs[r][b] for r in range(len(grads))])
        calls.append((b, B, b == B - 1))
        arena[starts[b]:starts[b + 1]] = result
        for v in members[b]:
            lo = int(starts[b]) + locators[v].offset
            for o in range(n_out):
                outs[o][v] = arena[lo:lo + numel[v]].copy()
    return arena, outs, calls
