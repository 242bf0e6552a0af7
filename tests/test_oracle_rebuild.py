"""Pins of the bucket-rebuild oracle (no GPU)."""

import itertools
import os

import pytest

from oracle.buckets import assign_buckets, bucket_lengths
from oracle.rebuild import rebuild_buckets

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
MIB = 1 << 20
MAXSIZE = (1 << 63) - 1


def _valid_splits(sizes, first_cap, cap):
    """Every split of the traced list into consecutive groups such that each
    group but the last reaches its limit (first_cap for group 0, cap after)
    and no group reaches its limit before its last member.  Exactly one
    split qualifies: the packing rule stated as properties of the result."""
    n = len(sizes)
    out = []
    for cuts in itertools.product([0, 1], repeat=max(n - 1, 0)):
        groups, cur = [], [0] if n else []
        for i in range(1, n):
            if cuts[i - 1]:
                groups.append(cur)
                cur = []
            cur.append(i)
        if n:
            groups.append(cur)
        ok = True
        for gi, g in enumerate(groups):
            lim = first_cap if gi == 0 else cap
            tot = sum(sizes[i] for i in g)
            if len(g) >= 2 and tot - sizes[g[-1]] >= lim:
                ok = False
            if gi < len(groups) - 1 and tot < lim:
                ok = False
        if ok:
            out.append(groups)
    return out


@pytest.mark.parametrize("first_cap,cap", [(0, 0), (4, 12), (12, 4), (1, 40), (16, 16)])
def test_bruteforce_two_limits(first_cap, cap):
    for n in range(1, 6):
        values = [0, 1, 3, 4] if n <= 4 else [1, 4]
        for numel in itertools.product(values, repeat=n):
            for trace in itertools.permutations(range(n)):
                members, locs = rebuild_buckets(numel, 4, trace, first_cap, cap)
                sizes = [numel[v] * 4 for v in trace]
                splits = _valid_splits(sizes, first_cap, cap)
                assert len(splits) == 1
                assert members == [[trace[i] for i in g] for g in splits[0]]
                for b, vs in enumerate(members):
                    off = 0
                    for intra, v in enumerate(vs):
                        assert (locs[v].bucket, locs[v].intra, locs[v].offset) == (b, intra, off)
                        off += numel[v]


def test_reverse_trace_equal_caps_is_construction_layout():
    numel = [5, 0, 7, 1, 3, 9, 2]
    for cap in (0, 4, 12, 40, 1000):
        got = rebuild_buckets(numel, 4, list(range(6, -1, -1)), cap, cap)
        assert got == assign_buckets(numel, 4, cap)


def _golden():
    rows = []
    for line in open(os.path.join(GOLDEN, "rebuild_layouts.txt"), encoding="utf-8"):
        line = line.strip()
        if line and not line.startswith("#"):
            name, cnt, mib, fc, cap, sizes = line.split()
            rows.append((name, int(cnt), int(mib), int(fc), int(cap), [int(x) for x in sizes.split(",")]))
    return rows


@pytest.mark.parametrize("row", _golden(), ids=lambda r: r[0])
def test_page_rebuild_layouts(row):
    name, cnt, mib, fc, cap, sizes = row
    numel = [mib * MIB // 4] * cnt
    trace = list(range(cnt - 1, -1, -1))
    fcb = MAXSIZE if fc < 0 else fc * MIB
    cb = MAXSIZE if cap < 0 else cap * MIB
    members, _ = rebuild_buckets(numel, 4, trace, fcb, cb)
    assert [n * 4 // MIB for n in bucket_lengths(members, numel)] == sizes


def test_first_cap_only_shapes_bucket_zero():
    numel = [1] * 10
    members, _ = rebuild_buckets(numel, 1, list(range(10)), 2, 4)
    assert members == [[0, 1], [2, 3, 4, 5], [6, 7, 8, 9]]


def test_trace_order_decides_membership():
    numel = [4, 4, 4, 4]
    a, _ = rebuild_buckets(numel, 1, [3, 2, 1, 0], 8, 8)
    b, _ = rebuild_buckets(numel, 1, [0, 3, 1, 2], 8, 8)
    assert a == [[3, 2], [1, 0]] and b == [[0, 3], [1, 2]]


def test_trace_must_be_a_permutation():
    with pytest.raises(ValueError):
        rebuild_buckets([1, 1, 1], 4, [0, 1], 4, 4)
    with pytest.raises(ValueError):
        rebuild_buckets([1, 1, 1], 4, [0, 1, 1], 4, 4)
