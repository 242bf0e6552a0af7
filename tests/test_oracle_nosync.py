"""Pins of the no_sync accumulation oracle (no GPU)."""

import numpy as np

from oracle.buckets import assign_buckets
from oracle.nosync import accumulate, accumulate_steps
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
