"""Oracle: assignment of parameters to gradient buckets (construction time).

Test infrastructure only; see the package docstring.

What the pages fix:

* Parameters are packed in the *reverse* of registration order
  ("PyTorch Distributed: Experiences on Accelerating Data Parallel
  Training", Section 3.2.2 as summarised under "Gradient Bucketing:
  Amortizing AllReduce Overhead", paragraph "Bucket construction";
  "Distributed Data Parallel" notes, "Internal Design", "Construction").
* Whole tensors are added one at a time; after adding a tensor's bytes
  (numel x element size) the bucket is closed as soon as its size has
  *reached or passed* the cap, so a tensor is never split and a bucket may
  exceed the cap ("NCCL 专家课程 30", section "`bucket_cap_mb` 不是张量切分器":
  an 8 MiB tensor under a 4 MiB cap gives an 8 MiB bucket).  The
  paper summary says "exceeds"; the reducer excerpt and the layout table of
  section "参数粒度实验" (48 x 1 MiB at cap 4 MiB -> 12 buckets of 4) fix
  the comparison as ``>=``.
* Each variable's locator holds its bucket index and its index inside the
  bucket, plus offset and length within the flat bucket ("NCCL 专家课程 30",
  section "Variable 到 Bucket"); the view of a variable is
  ``bucket.narrow(offset, numel)`` (paper summary, "The per-hook logic").

Readings where the pages are silent:

* intra-bucket index = push position; offset = sum of the lengths of the
  earlier members, in elements, with no padding inside a bucket;
* bucket 0 is the first bucket closed while walking the reverse order;
* bytes are counted with the element size of the gradient dtype;
* one cap for every bucket (no separate first-bucket cap);
* a non-empty remainder at the end of the walk forms the last bucket;
* zero-element tensors join the current bucket with length 0; negative
  sizes are rejected.
"""

from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Locator:
    bucket: int
    intra: int
    offset: int   # elements, within the bucket
    length: int   # elements


def assign_buckets(numel, elem_size: int, cap_bytes: int):
    """Greedy packing over the reversed parameter list.

    Returns ``(members, locators)``: ``members[b]`` is the list of variable
    indices of bucket b in push order, ``locators[v]`` the Locator of v.
    """
    numel = [int(n) for n in numel]
    if any(n < 0 for n in numel):
        raise ValueError("negative numel")
    if elem_size <= 0 or cap_bytes < 0:
        raise ValueError("bad element size or cap")
    members: list[list[int]] = []
    current: list[int] = []
    size = 0
    for v in range(len(numel) - 1, -1, -1):          # reverse registration order
        current.append(v)
        size += numel[v] * elem_size
        if size >= cap_bytes:                         # close once the cap is reached
            members.append(current)
            current, size = [], 0
    if current:
        members.append(current)

    locators: list[Locator | None] = [None] * len(numel)
    for b, vs in enumerate(members):
        offset = 0
        for intra, v in enumerate(vs):
            locators[v] = Locator(b, intra, offset, numel[v])
            offset += numel[v]
    return members, locators


def bucket_lengths(members, numel) -> list[int]:
    """Element count of every bucket."""
    return [sum(int(numel[v]) for v in vs) for vs in members]


def arena_offsets(members, numel) -> list[int]:
    """Start of every bucket when the buckets are laid out back to back in
    index order in one flat arena (B+1 entries; the last is the total)."""
    out = [0]
    for n in bucket_lengths(members, numel):
        out.append(out[-1] + n)
    return out
