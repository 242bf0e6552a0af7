"""Pins of the bucket-assignment oracle (no GPU).

The oracle's greedy walk is checked against facts that do not come from it:
a brute-force characterisation over every split of tiny lists, the
layout table printed on the NCCL/DDP course page, the 8 MiB-tensor example,
the per-gradient (cap 0) end point, and the Linear(10,10) example.
"""

import itertools
import os

import pytest

from oracle.buckets import arena_offsets, assign_buckets, bucket_lengths
from workloads import shapes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
MIB = 1 << 20


def _valid_splits(sizes_rev, cap):
    """Every split of the reversed list into consecutive non-empty groups
    such that (i) each group but the last reaches the cap and (ii) no group
    reaches the cap before its last member.  Exactly one split satisfies
    both: the reducer's "close as soon as the cap is reached" rule stated as
    properties of the result instead of as a walk.  (ii) concerns non-empty
    proper prefixes only; sizes are non-negative, so the largest of them,
    the group without its last member, decides."""
    n = len(sizes_rev)
    found = []
    for cuts in itertools.product([0, 1], repeat=max(n - 1, 0)):
        groups, cur = [], [0]
        for i in range(1, n):
            if cuts[i - 1]:
                groups.append(cur)
                cur = []
            cur.append(i)
        if n:
            groups.append(cur)
        ok = True
        for gi, g in enumerate(groups):
            total = sum(sizes_rev[i] for i in g)
            before_last = total - sizes_rev[g[-1]]
            if len(g) >= 2 and before_last >= cap:
                ok = False
            if gi < len(groups) - 1 and total < cap:
                ok = False
        if ok:
            found.append(groups)
    return found


@pytest.mark.parametrize("cap", [0, 1, 4, 12, 16, 40])
def test_bruteforce_unique_split(cap):
    elem = 4
    for n in range(0, 6):
        for numel in itertools.product([0, 1, 3, 4], repeat=n):
            members, locs = assign_buckets(numel, elem, cap)
            rev = list(range(n - 1, -1, -1))
            sizes_rev = [numel[v] * elem for v in rev]
            splits = _valid_splits(sizes_rev, cap)
            assert len(splits) == 1, (numel, cap, splits)
            expect = [[rev[i] for i in g] for g in splits[0]]
            assert members == expect, (numel, cap)
            # locators: index and prefix offsets inside each bucket
            for b, vs in enumerate(members):
                off = 0
                for intra, v in enumerate(vs):
                    assert (locs[v].bucket, locs[v].intra, locs[v].offset, locs[v].length) == (b, intra, off, numel[v])
                    off += numel[v]


def _golden_layouts():
    rows = []
    with open(os.path.join(GOLDEN, "bucket_layouts.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, cnt, mib, cap, nb, sizes = line.split()
            rows.append((name, int(cnt), int(mib), int(cap), int(nb), [int(s) for s in sizes.split(",")]))
    return rows


@pytest.mark.parametrize("row", _golden_layouts(), ids=lambda r: r[0])
def test_page_layout_table(row):
    name, cnt, mib, cap, nb, sizes = row
    numel = [mib * MIB // 4] * cnt
    members, _ = assign_buckets(numel, 4, cap * MIB)
    assert len(members) == nb
    assert [n * 4 // MIB for n in bucket_lengths(members, numel)] == sizes


def test_strict_greater_would_differ():
    # The table's 48 x 1 MiB at 4 MiB -> 12 buckets; a ">" close rule gives
    # buckets of 5 tensors.  Guards against the comparison being flipped.
    numel = [MIB // 4] * 48
    members, _ = assign_buckets(numel, 4, 4 * MIB)
    assert all(len(m) == 4 for m in members)


def test_large_tensor_never_split():
    numel = [2 * MIB // 4, 8 * MIB // 4]          # walked in reverse: 8 MiB first
    members, locs = assign_buckets(numel, 4, 4 * MIB)
    assert members == [[1], [0]]
    assert locs[1].length * 4 == 8 * MIB


def test_cap_zero_is_per_gradient():
    numel = [5, 0, 7, 1]
    members, _ = assign_buckets(numel, 4, 0)
    assert members == [[3], [2], [1], [0]]


def test_linear_example_layout():
    numel = shapes.numels(shapes.linear_10x10())     # weight 100, bias 10
    members, locs = assign_buckets(numel, 4, 25 * MIB)
    assert members == [[1, 0]]
    assert (locs[1].bucket, locs[1].intra, locs[1].offset, locs[1].length) == (0, 0, 0, 10)
    assert (locs[0].bucket, locs[0].intra, locs[0].offset, locs[0].length) == (0, 1, 10, 100)
    assert arena_offsets(members, numel) == [0, 110]


def test_empty_and_invalid():
    assert assign_buckets([], 4, 25 * MIB) == ([], [])
    with pytest.raises(ValueError):
        assign_buckets([3, -1], 4, 16)
    with pytest.raises(ValueError):
        assign_buckets([3], 4, -1)


def test_bf16_counts_two_bytes():
    numel = [MIB] * 4                                 # 2 MiB each in bf16, 4 MiB in fp32
    m16, _ = assign_buckets(numel, 2, 4 * MIB)
    m32, _ = assign_buckets(numel, 4, 4 * MIB)
    assert len(m16) == 2 and len(m32) == 4


def test_workload_layout_summary():
    """Bucket counts of the synthetic workloads (regression summary; the
    rules themselves are pinned above)."""
    def nb(fn, elem, cap_mib):
        return len(assign_buckets(shapes.numels(fn()), elem, cap_mib * MIB)[0])
    assert nb(shapes.resnet50, 4, 25) == 4
    assert nb(shapes.bert_large, 4, 25) == 37
    assert [nb(shapes.gpt2_medium, 2, c) for c in (0, 1, 5, 25, 100)] == [292, 98, 73, 20, 6]
