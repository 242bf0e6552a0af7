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
does ``acc = fl32(acc + g_k)`` in step order; fp32 gradients only.
"""

from __future__ import annotations

import numpy as np


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
