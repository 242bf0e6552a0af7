"""Pins of the no_sync accumulation oracle (no GPU)."""

import numpy as np

from oracle.buckets import assign_buckets
from oracle.nosync import accumulate, accumulate_steps, reduce_last_step
from oracle.reduce import reduce_buckets

F32 = np.float32


def test_integer_accumulation_exact_then_reduce():
    rng = np.random.default_rng(11)
    numel = [4, 9, 1]
    W, K = 4, 8
    steps = [[[rng.integers(-1000, 1000, size=n).astype(F32) for n in numel]
              for _ in range(K)] for _ in range(W)]
    accs = [accumulate_steps(steps[r]) for r in range(W)]
    for r in range(W):
        for v in range(len(numel)):
            assert np.array_equal(accs[r][v], sum(steps[r][k][v].astype(np.int64) for k in range(K)).astype(F32))
    members, locs = assign_buckets(numel, 4, 8)
    _, outs = reduce_buckets(accs, members, locs, numel)
    for v in range(len(numel)):
        total = sum(steps[r][k][v].astype(np.int64) for r in range(W) for k in range(K))
        assert np.array_equal(outs[0][v], (total / (W)).astype(F32))   # exact: |total| < 2^24, W = 4


def test_first_step_assigns():
    g = [np.array([-0.0, 1.5], F32)]
    acc = accumulate(None, g, first_step=True)
    assert np.signbit(acc[0][0]) and acc[0][1] == F32(1.5)
    assert acc[0] is not g[0]
    # one step only: identity
    assert np.array_equal(accumulate_steps([g])[0], g[0])


def test_in_step_order():
    # 1 + 2^-24 rounds to 1; order of the steps decides the result
    u = F32(2.0 ** -24)
    a = accumulate_steps([[np.array([1.0], F32)], [np.array([u], F32)], [np.array([u], F32)]])
    b = accumulate_steps([[np.array([u], F32)], [np.array([u], F32)], [np.array([1.0], F32)]])
    assert a[0][0] == F32(1.0)
    assert b[0][0] == F32(1.0) + F32(2.0 ** -23)


def test_last_step_integer_closed_form():
    # integer-valued gradients: every sum is exact, so the mean over replicas
    # of all K micro-steps is the integer total / W
    rng = np.random.default_rng(12)
    numel = [6, 0, 11, 2]
    W, K = 4, 5
    steps = [[[rng.integers(-500, 500, size=n).astype(F32) for n in numel] for _ in range(K)] for _ in range(W)]
    accs = [accumulate_steps(steps[r][:K - 1]) for r in range(W)]
    members, locs = assign_buckets(numel, 4, 16)
    arena, outs = reduce_last_step(accs, [steps[r][K - 1] for r in range(W)], members, locs, numel, n_out=2)
    for v, n in enumerate(numel):
        total = sum(steps[r][k][v].astype(np.int64) for r in range(W) for k in range(K))
        want = (total / W).astype(F32)
        assert np.array_equal(outs[0][v], want) and np.array_equal(outs[1][v], want)
    assert not np.isnan(arena).any()


def test_last_step_adds_per_replica_before_the_rank_sum():
    # W = 2, one element.  Per replica first: fl32(1 + u) = 1 (tie to even) and
    # fl32(u + u) = 2u, then 1 + 2u = 1 + 2^-23 exactly, times 1/2.  Summing the
    # accumulators first and the last-step gradients after would give 1/2.
    u = F32(2.0 ** -24)
    acc = [[np.array([1.0], F32)], [np.array([u], F32)]]
    g = [[np.array([u], F32)], [np.array([u], F32)]]
    members, locs = assign_buckets([1], 4, 0)
    _, outs = reduce_last_step(acc, g, members, locs, [1])
    assert outs[0][0][0] == F32((1.0 + 2.0 ** -23) / 2)
    assert outs[0][0][0] != F32(0.5)


def test_last_step_leaves_accumulators_and_keeps_signed_zero():
    acc = [[np.array([-0.0, 3.0], F32)]]
    g = [[np.array([-0.0, -3.0], F32)]]
    before = acc[0][0].copy()
    members, locs = assign_buckets([2], 4, 0)
    _, outs = reduce_last_step(acc, g, members, locs, [2])
    assert np.array_equal(acc[0][0].view(np.uint32), before.view(np.uint32))
    # W = 1: (-0) + (-0) = -0 and 3 + (-3) = +0, times 1
    assert np.signbit(outs[0][0][0]) and outs[0][0][1] == 0 and not np.signbit(outs[0][0][1])


def test_last_step_equals_the_unfused_block():
    rng = np.random.default_rng(13)
    numel = [5, 33, 1, 0, 70]
    W, K = 3, 4
    steps = [[[(rng.standard_normal(n) * 1e-3).astype(F32) for n in numel] for _ in range(K)] for _ in range(W)]
    members, locs = assign_buckets(numel, 4, 64)
    accs = [accumulate_steps(steps[r][:K - 1]) for r in range(W)]
    a1, o1 = reduce_last_step(accs, [steps[r][K - 1] for r in range(W)], members, locs, numel)
    a2, o2 = reduce_buckets([accumulate_steps(steps[r]) for r in range(W)], members, locs, numel)
    assert np.array_equal(a1.view(np.uint32), a2.view(np.uint32))
    assert all(np.array_equal(x.view(np.uint32), y.view(np.uint32)) for x, y in zip(o1[0], o2[0]))
