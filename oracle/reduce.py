"""Oracle: gather into buckets, W-way mean, copy-back.

Test infrastructure only; see the package docstring.

What the pages fix:

* the result every replica ends up with is the mean gradient
  g = (1/W) * sum_r g_r ("PyTorch Distributed Training Internals",
  section 3 "The All-Reduce Itself"; paper summary, "How gradient
  synchronization solves both problems");
* a ready gradient is copied into its bucket at its locator offset
  (``bucket.narrow(offset, numel).copy_(grad)``: paper summary, "The
  per-hook logic"); the whole bucket is reduced; the reduced values are
  copied back into every parameter's gradient, one batched copy per bucket
  ("Distributed Data Parallel" notes, "Backward pass");
* under ``gradient_as_bucket_view`` the gradient *is* the bucket view, so
  the copy-back disappears ("NCCL 专家课程 30", section
  "`gradient_as_bucket_view`").

The arithmetic, fixed as the plain definition with one summation order:
per element, widen each replica's value to fp32 (bf16 -> fp32 is exact),
then ``acc = x_0``; ``acc = fl32(acc + x_r)`` for r = 1 .. W-1 in rank order;
``out = fl32(acc * fl32(1/W))``.  Reading: the pages say fp32 buckets are
"averaged directly" and other dtypes "pre-divided and summed", and the
default hook divides before summing; for power-of-two W the two agree bit
for bit (scaling by 2^-k is exact barring underflow), and the multiply
after an in-order fp32 sum is the definition used here for every W.
Starting from ``x_0`` rather than ``0 + x_0`` keeps the sign of -0.0.
NumPy fp32 operations round to nearest-even and keep subnormals.

Emulation: the W replicas of one data-parallel group are W gradient sets
in one process; the reduced bucket and the copied-back gradients are the
values every replica would hold after the collective, so one output set
stands for all of them (``n_out=1``), or W identical copies are written
(``n_out=W``, the broadcast form used by the replicas-identical test).
"""

from __future__ import annotations

import numpy as np


def widen(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp32 exactly; fp32 passes through."""
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32)
    if x.dtype == np.float32:
        return x
    raise TypeError(f"unsupported gradient dtype {x.dtype}")


def inv_world(W: int) -> np.float32:
    """fl32(1/W): correctly rounded fp32 quotient."""
    return np.float32(1.0) / np.float32(W)


def replica_mean(xs) -> np.ndarray:
    """Mean of W equally long replica arrays, sequential fp32 sum then x 1/W."""
    W = len(xs)
    if W < 1:
        raise ValueError("need at least one replica")
    acc = np.array(widen(xs[0]), dtype=np.float32, copy=True)
    with np.errstate(invalid="ignore", over="ignore"):     # IEEE results, no warnings
        for r in range(1, W):
            acc = acc + widen(xs[r])
        return acc * inv_world(W)


def reduce_buckets(grads, members, locators, numel, buckets=None, n_out: int = 1):
    """Run the fused bucket pass over the given buckets (default: all).

    ``grads[r][v]``: replica r's gradient of variable v (1-D fp32 or bf16
    bits).  Returns ``(arena, outs)``:

    * ``arena`` -- fp32 flat buffer, the buckets back to back in index order,
      NaN where a bucket was not part of this pass;
    * ``outs[o][v]`` -- copied-back gradient of v for output copy o
      (``n_out`` copies; ``None`` for variables whose bucket was not reduced).
    """
    W = len(grads)
    B = len(members)
    lens = [sum(int(numel[v]) for v in vs) for vs in members]
    starts = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64) if B else np.zeros(1, np.int64)
    arena = np.full(int(starts[-1]), np.nan, dtype=np.float32)
    outs = [[None] * len(numel) for _ in range(n_out)]
    todo = range(B) if buckets is None else buckets
    for b in todo:
        for v in members[b]:                       # gather in push order
            loc = locators[v]
            mean = replica_mean([grads[r][v] for r in range(W)])
            lo = int(starts[b]) + loc.offset
            arena[lo:lo + loc.length] = mean        # bucket view of v
            for o in range(n_out):                  # copy-back
                outs[o][v] = arena[lo:lo + loc.length].copy()
    return arena, outs


def sgd_step(params, grads, lr: float):
    """p <- fl32(p - fl32(lr * g)), for the replicas-identical check."""
    lr32 = np.float32(lr)
    return [p - lr32 * g for p, g in zip(params, grads)]
