"""Oracle: local gradient accumulation under ``no_sync``.

Test infrastructure only; see the package docstring.

What the pages fix ("PyTorch Distributed: Experiences on Accelerating Data
Parallel Training", Section 3.2.4 as summarised under "Gradient
Accumulation (no_sync)"; "Distributed Data Parallel" notes, "Gradient sync
you can turn off"):

* inside the context no bucket copy and no collective happens; each
  replica's gradient accumulates additively across backward passes;
* the first backward outside the context reduces the accumulated
  gradients (the same bucket pass as an ordinary iteration).

Readings: the first micro-step *assigns* its gradient (the gradient field
is empty before it, so ``acc = g_1`` exactly, keeping -0.0), every later one
does ``acc = fl32(acc + g_k)`` in step order; fp32 gradients only.  The
synchronizing backward that ends the block is one more micro-step whose
gradient accumulates into the same fields before its hooks hand them to the
bucket pass: each replica's reduced input is ``fl32(acc_r + g_r)``, formed
per replica and only then summed in rank order.
"""

from __future__ import annotations

import numpy as np

from .reduce import reduce_buckets


def accumulate(acc, g, first_step: bool):
    """One micro-step for one replica's list of per-variable arrays."""
    if first_step:
        return [np.array(x, dtype=np.float32, copy=True) for x in g]
    with np.errstate(invalid="ignore", over="ignore"):     # IEEE results, no warnings
        return [a + x for a, x in zip(acc, g)]


def accumulate_steps(steps):
    """``steps[k][v]`` -> accumulated per-variable arrays after all steps."""
    acc = None
    for k, g in enumerate(steps):
        acc = accumulate(acc, g, k == 0)
    return acc


def reduce_last_step(acc, g_last, members, locators, numel, n_out: int = 1):
    """The synchronizing micro-step: ``g_last`` accumulates into every
    replica's fields (``acc`` is not changed), then the ordinary bucket pass
    averages the sums.  Returns ``(arena, outs)`` as ``reduce_buckets``."""
    summed = [accumulate(a, g, first_step=False) for a, g in zip(acc, g_last)]
    return reduce_buckets(summed, members, locators, numel, n_out=n_out)
