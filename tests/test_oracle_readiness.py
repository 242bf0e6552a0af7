"""Pins of the readiness state-machine oracle (no GPU).

Checked against: a closed form of in-order launching over every
permutation of tiny parameter lists, the sequence diagram on the NCCL/DDP
course page (bucket 2 ready before bucket 1), the page's observed reverse
ready order, and the failure modes the pages name.
"""

import itertools
import os

import pytest

from oracle.buckets import assign_buckets
from oracle.readiness import (AlreadyReady, OutOfOrder, PriorReductionUnfinished,
                              ReadinessOracle, launch_events)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _closed_form(members, order):
    """Bucket b goes out at the event where the last of buckets 0..b
    completes: launch_at[b] = max_{j<=b} completion[j]."""
    pos = {v: t for t, v in enumerate(order)}
    completion = [max(pos[v] for v in vs) for vs in members]
    launch_at, m = [], -1
    for c in completion:
        m = max(m, c)
        launch_at.append(m)
    parked_after = []
    for t in range(len(order)):
        parked_after.append([b for b in range(len(members)) if completion[b] <= t < launch_at[b]])
    return launch_at, parked_after


LAYOUTS = [
    [1, 1, 1, 1, 1, 1, 1],      # caps below give 7, 4, 3, 2, 1 buckets
    [3, 0, 2, 5, 1, 4, 2],
    [1, 2, 3],
]


@pytest.mark.parametrize("numel", LAYOUTS)
@pytest.mark.parametrize("cap", [0, 2, 3, 6, 100])
def test_bruteforce_all_permutations(numel, cap):
    members, _ = assign_buckets(numel, 1, cap)
    P = len(numel)
    for order in itertools.permutations(range(P)):
        launch_at, trace = launch_events(members, order)
        expect_launch, expect_parked = _closed_form(members, order)
        assert launch_at == expect_launch, (order, members)
        for t, (v, b, pend, launched, parked) in enumerate(trace):
            assert v == order[t]
            assert launched == [bb for bb in range(len(members)) if expect_launch[bb] == t]
            assert parked == expect_parked[t]


def test_page_parking_sequence():
    rows = []
    with open(os.path.join(GOLDEN, "parking_sequence.txt"), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    members, _ = assign_buckets([1, 1, 1], 1, 1)
    sm = ReadinessOracle(members)
    sm.begin_iteration()
    for ev, v, b, launched, parked in rows:
        got = sm.mark_ready(int(v))
        assert sm.bucket_of[int(v)] == int(b)
        assert got == ([] if launched == "-" else [int(x) for x in launched.split(",")])
        assert sm.parked() == ([] if parked == "-" else [int(x) for x in parked.split(",")])


@pytest.mark.parametrize("cap_mib,launch_events_expected", [
    (4, list(range(12))),          # 12 buckets, each launched by its own tensor
    (16, [3, 7, 11]),              # 3 buckets of 4 tensors
    (64, [11]),                    # one 48 MiB bucket
])
def test_page_reverse_ready_order(cap_mib, launch_events_expected):
    # 12 independent 4 MiB tensors ready in the order 11, 10, ..., 0, as
    # observed on the NCCL/DDP course page ("Parameter Hook 如何安装").
    numel = [1 << 20] * 12
    members, _ = assign_buckets(numel, 4, cap_mib << 20)
    launch_at, trace = launch_events(members, list(range(11, -1, -1)))
    assert launch_at == launch_events_expected
    assert all(parked == [] for *_, parked in trace)


def test_errors():
    members, _ = assign_buckets([1, 1, 1], 1, 1)
    sm = ReadinessOracle(members)
    sm.begin_iteration()
    sm.mark_ready(2)
    with pytest.raises(AlreadyReady):
        sm.mark_ready(2)
    with pytest.raises(OutOfOrder):
        sm.launch_next(2)
    sm.mark_ready(1)
    # variable 0 never reports: the next iteration must refuse to start
    with pytest.raises(PriorReductionUnfinished):
        sm.begin_iteration()
    sm.abort_iteration()
    sm.begin_iteration()
    assert sm.launch_next(0) == [0]
    assert sm.launch_rest() == [1, 2]
    sm.begin_iteration()                    # previous one finished: fine


def test_explicit_launch_releases_parked():
    members, _ = assign_buckets([1, 1, 1], 1, 1)   # v -> bucket 2 - v
    sm = ReadinessOracle(members)
    sm.begin_iteration()
    assert sm.mark_ready(0) == []                   # bucket 2 parks
    assert sm.launch_next(0) == [0]
    assert sm.launch_next(1) == [1, 2]              # 1 goes, then parked 2
    sm.begin_iteration()
    sm.mark_ready(1)
    with pytest.raises(AlreadyReady):
        sm.mark_ready(1)
