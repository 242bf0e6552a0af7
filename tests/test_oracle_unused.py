"""Pins of the unused-parameter oracle (no GPU)."""

import itertools

import numpy as np

from oracle.buckets import assign_buckets
from oracle.readiness import launch_events
from oracle.reduce import reduce_buckets
from oracle.unused import (UnusedReadiness, accumulate_masked, globally_used,
                           reduce_with_unused)

F32 = np.float32


def test_all_used_is_the_plain_reduce():
    numel = [3, 5, 2]
    members, locs = assign_buckets(numel, 4, 16)
    rng = np.random.default_rng(0)
    grads = [[rng.standard_normal(n).astype(F32) for n in numel] for _ in range(4)]
    used = [[True] * 3 for _ in range(4)]
    a1, o1 = reduce_with_unused(grads, used, members, locs, numel)
    a2, o2 = reduce_buckets(grads, members, locs, numel)
    assert np.array_equal(a1, a2) and all(np.array_equal(x, y) for x, y in zip(o1[0], o2[0]))


def test_unused_replicas_contribute_zero_integer_exact():
    numel = [6, 4]
    members, locs = assign_buckets(numel, 4, 1 << 20)
    rng = np.random.default_rng(1)
    W = 4
    grads = [[rng.integers(-100, 100, size=n).astype(F32) for n in numel] for _ in range(W)]
    used = [[True, True], [False, True], [True, False], [False, False]]
    _, outs = reduce_with_unused(grads, used, members, locs, numel)
    for v in range(2):
        total = sum(grads[r][v].astype(np.int64) for r in range(W) if used[r][v])
        assert np.array_equal(outs[0][v], (total / W).astype(F32))      # mean over all W replicas


def test_globally_unused_left_untouched_and_bucket_zero():
    numel = [3, 2, 4]
    members, locs = assign_buckets(numel, 4, 1 << 20)
    grads = [[np.full(n, 7.0, F32) for n in numel] for _ in range(2)]
    used = [[True, False, True], [True, False, False]]
    arena, outs = reduce_with_unused(grads, used, members, locs, numel)
    assert globally_used(used) == [True, False, True]
    assert outs[0][1] is None
    lo = locs[1].offset
    assert np.array_equal(arena[lo:lo + 2], np.zeros(2, F32))
    assert np.array_equal(outs[0][2], np.full(4, 3.5, F32))            # (7 + 0) / 2


def test_zero_fill_is_positive_zero():
    # replica 0 holds -0.0, replica 1 does not use the parameter: -0 + +0 = +0
    numel = [1]
    members, locs = assign_buckets(numel, 4, 16)
    grads = [[np.array([-0.0], F32)], [np.array([5.0], F32)]]
    _, outs = reduce_with_unused(grads, [[True], [False]], members, locs, numel)
    assert outs[0][0][0] == 0 and not np.signbit(outs[0][0][0])


def test_unused_buckets_launch_at_first_event():
    """Course page ("Unused Parameter"): the unused indices are marked ready
    when the first real hook fires, so a bucket holding only unused
    parameters goes out then instead of hanging the iteration."""
    numel = [1, 1, 1, 1]
    members, _ = assign_buckets(numel, 1, 1)           # v -> bucket 3 - v
    used = [[True, True, False, True], [True, True, False, True]]
    sm = UnusedReadiness(members, used)
    sm.begin_iteration()
    # var 2 (bucket 1) is marked first and parks behind bucket 0; var 3
    # completes bucket 0, which goes out and takes the parked bucket 1 along
    assert sm.mark_ready(3) == [0, 1]
    assert sm.mark_ready(1) == [2]
    assert sm.mark_ready(0) == [3]
    # without the marking the iteration could never finish
    plain = UnusedReadiness(members, [[True] * 4, [True] * 4])
    plain.begin_iteration()
    plain.mark_ready(3), plain.mark_ready(1), plain.mark_ready(0)
    assert plain.next == 1


def test_unused_readiness_matches_closed_form():
    """Marking the globally unused variables ready first is the plain state
    machine run on the order (unused ascending) + (reported order)."""
    numel = [1, 2, 1, 3, 1]
    members, _ = assign_buckets(numel, 1, 2)
    for used_mask in itertools.product([True, False], repeat=5):
        used = [list(used_mask), [False] * 5]
        unused = [v for v in range(5) if not used_mask[v]]
        reported = [v for v in range(5) if used_mask[v]]
        for order in itertools.permutations(reported):
            if not order:
                continue
            sm = UnusedReadiness(members, used)
            sm.begin_iteration()
            got = []
            for v in order:
                got.append(sm.mark_ready(v))
            plain, _ = launch_events(members, unused + list(order))
            # every bucket goes out; the first event carries everything the
            # unused prefix released
            flat = [b for ev in got for b in ev]
            assert flat == list(range(len(members)))
            k = len(unused)
            assert got[0] == [b for b in range(len(members)) if plain[b] <= k]
            for i in range(1, len(order)):
                assert got[i] == [b for b in range(len(members)) if plain[b] == k + i]


def test_nosync_bitmap_accumulates_and_first_gradient_assigns():
    """A parameter unused in micro-step 1 but used in step 2 takes step 2's
    gradient (its field was empty); one unused in every step stays empty."""
    g1 = [np.array([1.0], F32), np.array([2.0], F32), np.array([3.0], F32)]
    g2 = [np.array([10.0], F32), np.array([20.0], F32), np.array([30.0], F32)]
    acc, has = accumulate_masked(None, None, g1, [True, False, False], first_step=True)
    acc, has = accumulate_masked(acc, has, g2, [True, True, False], first_step=False)
    assert acc[0][0] == 11.0 and acc[1][0] == 20.0 and acc[2] is None
    assert has == [True, True, False]
    # a new block forgets the old fields
    acc, has = accumulate_masked(acc, has, g1, [False, True, False], first_step=True)
    assert has == [False, True, False] and acc[1][0] == 2.0
