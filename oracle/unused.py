"""Oracle: unused parameters and the globally-unused bitmap.

Test infrastructure only; see the package docstring.

What the pages fix:

* with find_unused_parameters, each replica learns in its forward pass which
  parameters will receive no gradient; their bucket slices are zero-filled
  and they are treated as ready, so their buckets can still reduce ("Distributed
  Data Parallel" notes, "Forward pass" and "When a parameter never receives a
  gradient"); the reducer marks them ready when the first real hook fires
  ("NCCL 专家课程 30", section "Unused Parameter");
* a bitmap with one bit per parameter records local use; an OR all-reduce of
  the bitmaps tells which parameters were unused on every replica, and those
  keep their gradients untouched after the reduction (paper summary, "The
  solution: global unused parameter detection via bitmap AllReduce");
* under no_sync the bitmap is not reset between micro-steps: it accumulates
  by OR and serves the next communication (paper summary, "The conflict with
  unused parameter marking"); a gradient accumulates additively, and a
  parameter whose gradient field is still empty takes the first gradient it
  gets.

Readings (one GPU holds all W replicas, one ready order for all of them):

* a variable is reported ready when the replicas that use it have its
  gradient; variables unused on every replica are marked ready at the
  iteration's first event, in ascending index order, before that event;
* a replica's contribution to an unused parameter is +0.0 in the rank-order
  sum (the zero-filled slice), so the mean is over all W replicas;
* "untouched" means the copy-back of a globally unused parameter is not
  written; its bucket slice holds the reduced zeros;
* the first no_sync micro-step starts a new block: every gradient field is
  empty again.
"""

from __future__ import annotations

import numpy as np

from .readiness import ReadinessOracle
from .reduce import reduce_buckets


def globally_used(used):
    """used[r][v] -> per-variable OR over the replicas."""
    W = len(used)
    P = len(used[0]) if W else 0
    return [any(bool(used[r][v]) for r in range(W)) for v in range(P)]


def zero_filled(grads, used):
    """Each replica's inputs with its unused parameters replaced by zeros."""
    out = []
    for r, rep in enumerate(grads):
        out.append([g if used[r][v] else np.zeros_like(g) for v, g in enumerate(rep)])
    return out


def reduce_with_unused(grads, used, members, locators, numel, n_out: int = 1):
    """The bucket pass with unused parameters: returns ``(arena, outs)`` where
    ``outs[o][v]`` is None for a globally unused variable (left untouched)."""
    arena, outs = reduce_buckets(zero_filled(grads, used), members, locators, numel, n_out=n_out)
    g = globally_used(used)
    for o in range(n_out):
        for v in range(len(numel)):
            if not g[v]:
                outs[o][v] = None
    return arena, outs


class UnusedReadiness(ReadinessOracle):
    """The readiness state machine with globally unused variables marked
    ready at the iteration's first event."""

    def __init__(self, members, used):
        super().__init__(members)
        self.unused = [v for v, u in enumerate(globally_used(used)) if not u]
        self._marked = False

    def begin_iteration(self):
        super().begin_iteration()
        self._marked = False

    def _mark_unused(self):
        launched = []
        if not self._marked:
            self._marked = True
            for v in self.unused:
                launched += ReadinessOracle.mark_ready(self, v)
        return launched

    def mark_ready(self, v: int):
        self._ensure_started()
        launched = self._mark_unused()
        launched += super().mark_ready(v)
        return launched


def accumulate_masked(acc, has, g, used, first_step: bool):
    """One no_sync micro-step for one replica with its local-used bits.

    ``acc``/``has``: per-variable accumulators and "gradient field holds a
    value" flags (lists, updated and returned).  A used variable takes the
    gradient if its field is empty, otherwise adds it; an unused one is left
    alone.  ``first_step`` starts a new block (every field empty)."""
    P = len(g)
    if first_step or has is None:
        has = [False] * P
        acc = [None] * P if acc is None else list(acc)
    acc = list(acc)
    with np.errstate(invalid="ignore", over="ignore"):
        for v in range(P):
            if used[v]:
                acc[v] = np.array(g[v], dtype=np.float32, copy=True) if not has[v] else acc[v] + g[v]
                has[v] = True
    return acc, has
