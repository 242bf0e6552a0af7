"""Oracle: bucket rebuild from a traced ready order.

Test infrastructure only; see the package docstring.

What the pages fix ("NCCL 专家课程 30: DDP Reducer、Bucket 与计算通信重叠",
section "第一次迭代为何不同"; "PyTorch Distributed: Experiences on
Accelerating Data Parallel Training" summary, future-work paragraph on
dynamic bucket reordering):

* during an iteration the hooks record the variables in the order their
  gradients actually became ready;
* before the next forward pass the buckets are packed again, walking the
  variables in that recorded order, with two size limits: one for the
  first bucket and one for every later bucket;
* the packing rule is the construction-time one (whole tensors; close once
  the size reaches the limit); a rebuild with the observed order 11..0 of
  the course page's 12 equal tensors gives its layout table (1, 3 or 12
  buckets at caps of 64, 16 and 4 MiB) where the first iteration had one
  bucket holding the whole 48 MiB model.

Readings: the trace must list every variable exactly once (the recorded
order of a complete iteration); the first-bucket limit is a parameter (the
pages name it without a value); all replicas adopt one trace (the pages
have rank 0's indices synced to every rank; the one-GPU emulation has one
ready order to begin with).
"""

from __future__ import annotations

from .buckets import Locator


def rebuild_buckets(numel, elem_size: int, trace, first_cap_bytes: int, cap_bytes: int):
    """Pack the variables in ``trace`` order; returns ``(members, locators)``."""
    numel = [int(n) for n in numel]
    P = len(numel)
    if sorted(trace) != list(range(P)):
        raise ValueError("the trace must list every variable exactly once")
    if first_cap_bytes < 0 or cap_bytes < 0:
        raise ValueError("negative cap")
    members: list[list[int]] = []
    current: list[int] = []
    size = 0
    for v in trace:
        current.append(v)
        size += numel[v] * elem_size
        limit = first_cap_bytes if not members else cap_bytes
        if size >= limit:
            members.append(current)
            current, size = [], 0
    if current:
        members.append(current)
    locators: list[Locator | None] = [None] * P
    for b, vs in enumerate(members):
        offset = 0
        for intra, v in enumerate(vs):
            locators[v] = Locator(b, intra, offset, numel[v])
            offset += numel[v]
    return members, locators
