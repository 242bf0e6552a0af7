"""Pins of the bucket-reduce oracle (no GPU).

The oracle's mean is checked against exact rational arithmetic on
integer-valued gradients, hand-derived fp32 cases in which the summation
order decides the result, sign/subnormal special cases, the fp64 error
bound, the bf16 widening of known bit patterns, the Linear(10,10) full-batch
identity of the worked DDP example, and the replicas-identical invariant.
"""

from fractions import Fraction

import numpy as np
import pytest

from oracle.buckets import assign_buckets, arena_offsets
from oracle.reduce import reduce_buckets, replica_mean, sgd_step, widen
from workloads import gen, shapes

F32 = np.float32


@pytest.mark.parametrize("W", [1, 2, 3, 4, 5, 8, 16])
def test_integer_gradients_exact(W):
    rng = np.random.default_rng(W)
    xs = [rng.integers(-1024, 1025, size=257).astype(np.float32) for _ in range(W)]
    got = replica_mean(xs)
    inv = Fraction(float(F32(1) / F32(W)))          # fl32(1/W) as an exact rational
    for i in range(257):
        s = sum(int(x[i]) for x in xs)              # |s| <= 16 * 1024: exact in fp32
        exact = Fraction(s) * inv                   # <= 39 significant bits: exact in fp64
        want = F32(float(exact))                    # one rounding to fp32
        assert got[i] == want, (W, i)
    if W & (W - 1) == 0:                            # power of two: the true mean exactly
        for i in range(257):
            assert Fraction(float(got[i])) == Fraction(sum(int(x[i]) for x in xs), W)


def test_rank_order_is_sequential():
    # 1 + 2^-24 is a tie and rounds to 1 (even); the in-order sum loses both
    # small terms, a pairwise tree would keep them.
    u = F32(2.0 ** -24)
    xs = [np.array([1.0], F32), np.array([u], F32), np.array([u], F32), np.array([-1.0], F32)]
    assert replica_mean(xs)[0] == F32(0.0)
    # small terms first: 2^-23 + 1 = 1 + 2^-23 exactly, minus 1 -> 2^-23, x 1/4
    xs = [np.array([u], F32), np.array([u], F32), np.array([1.0], F32), np.array([-1.0], F32)]
    assert replica_mean(xs)[0] == F32(2.0 ** -25)


def test_signed_zero_and_subnormals():
    nz = np.array([-0.0], F32)
    out = replica_mean([nz, nz, nz, nz])
    assert out[0] == 0 and np.signbit(out[0])
    out = replica_mean([nz, np.array([0.0], F32)])
    assert out[0] == 0 and not np.signbit(out[0])
    tiny = np.array([2.0 ** -149], F32)               # smallest subnormal
    assert replica_mean([tiny])[0] == tiny[0]
    assert replica_mean([tiny, tiny])[0] == tiny[0]   # (2 * 2^-149) * 0.5, no flush
    assert replica_mean([tiny, tiny, tiny, tiny])[0] == tiny[0]


def test_special_values_propagate():
    inf = np.array([np.inf], F32)
    assert np.isposinf(replica_mean([inf, np.array([1.0], F32)])[0])
    assert np.isnan(replica_mean([inf, -inf])[0])
    assert np.isnan(replica_mean([np.array([np.nan], F32), np.array([1.0], F32)])[0])


@pytest.mark.parametrize("W", [2, 4, 8, 16])
def test_identical_replicas_return_input(W):
    # With at most 19 significant bits every partial sum k*x (k <= 16) is
    # exact, and x 1/W (a power of two) undoes the sum exactly.
    x = gen.draw_flat_np(1000, 0)
    m, e = np.frexp(x.astype(np.float64))
    x19 = np.ldexp(np.round(m * 2.0 ** 19) / 2.0 ** 19, e).astype(np.float32)
    assert np.array_equal(replica_mean([x19] * W), x19)
    # W = 2 needs no restriction: x + x = 2x exactly for any finite x.
    assert np.array_equal(replica_mean([x, x]), x)


@pytest.mark.parametrize("W", [2, 3, 8, 16])
def test_error_bound_vs_fp64(W):
    rng = np.random.default_rng(7)
    xs = [rng.standard_normal(5000).astype(F32) for _ in range(W)]
    got = replica_mean(xs).astype(np.float64)
    exact = sum(x.astype(np.float64) for x in xs) / W
    mag = sum(np.abs(x.astype(np.float64)) for x in xs) / W
    u = 2.0 ** -24
    assert np.all(np.abs(got - exact) <= (W + 1) * u * mag + 1e-45)


def test_bf16_widening_known_bits():
    bits = np.array([0x3F80, 0xC000, 0x0001, 0x7F80, 0x8000, 0x3E80], np.uint16)
    want = np.array([1.0, -2.0, 2.0 ** -133, np.inf, -0.0, 0.25], F32)
    got = widen(bits)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    # bf16 replicas are summed in fp32: 3 x bf16(1.0) + bf16(-2.0) -> 1/4
    out = replica_mean([bits[:1], bits[:1], bits[:1], bits[1:2]])
    assert out[0] == F32(0.25)


def test_gather_and_copy_back_layout():
    numel = [3, 0, 5, 2, 7]
    members, locs = assign_buckets(numel, 4, 16)
    rng = np.random.default_rng(3)
    W = 3
    grads = [[rng.integers(-50, 50, size=n).astype(F32) for n in numel] for _ in range(W)]
    arena, outs = reduce_buckets(grads, members, locs, numel)
    starts = arena_offsets(members, numel)
    assert not np.isnan(arena).any()
    for v, n in enumerate(numel):
        lo = starts[locs[v].bucket] + locs[v].offset
        want = replica_mean([grads[r][v] for r in range(W)])
        assert np.array_equal(arena[lo:lo + n], want)
        assert np.array_equal(outs[0][v], want)
    # a partial pass leaves other buckets untouched
    arena2, outs2 = reduce_buckets(grads, members, locs, numel, buckets=[1])
    b1 = slice(starts[1], starts[2])
    assert np.array_equal(arena2[b1], arena[b1])
    assert np.isnan(np.delete(arena2, np.arange(starts[1], starts[2]))).all()


def _full_batch_grads64(ex):
    x = np.concatenate([xi.astype(np.float64) for xi in ex["x"]])   # (W*n, 10)
    w = ex["weight"].astype(np.float64)
    b = ex["bias"].astype(np.float64)
    out = x @ w.T + b
    c = 2.0 / out.size
    dw = c * out.T @ x
    db = c * out.sum(axis=0)
    # magnitude for the fp32 error bound of the per-replica backward
    a = np.abs(x) @ np.abs(w).T + np.abs(b)
    mag_w = c * (np.abs(out) + a).T @ np.abs(x)
    mag_b = c * (np.abs(out) + a).sum(axis=0)
    return dw.reshape(-1), db, mag_w.reshape(-1), mag_b


def test_linear_example_mean_is_full_batch_gradient():
    """Worked example ("Distributed Data Parallel" notes, section
    "Example"): two replicas of Linear(10,10), randn(20,10) each, loss
    mean(out^2).  Since the full-batch loss over the 40 rows is the average
    of the two replicas' losses, the mean gradient is the full-batch one."""
    ex = gen.linear_example(W=2, n=20, seed=0)
    numel = shapes.numels(shapes.linear_10x10())
    members, locs = assign_buckets(numel, 4, 25 << 20)
    arena, outs = reduce_buckets(ex["grads"], members, locs, numel)
    dw, db, mag_w, mag_b = _full_batch_grads64(ex)
    u = 2.0 ** -24
    assert np.all(np.abs(outs[0][0] - dw) <= 64 * u * mag_w)
    assert np.all(np.abs(outs[0][1] - db) <= 64 * u * mag_b)
    # the same identity in fp64 holds to rounding
    g64 = []
    for xi in ex["x"]:
        x = xi.astype(np.float64)
        out = x @ ex["weight"].astype(np.float64).T + ex["bias"].astype(np.float64)
        c = 2.0 / out.size
        g64.append((c * out.T @ x).reshape(-1))
    assert np.allclose((g64[0] + g64[1]) / 2, dw, rtol=1e-12, atol=1e-15)
    # a dropped 1/W would be off by 2x
    assert not np.allclose(outs[0][0] * 2, dw, rtol=1e-3)


@pytest.mark.parametrize("W", [2, 4])
def test_replicas_identical_after_step(W):
    """After the reduce every replica holds the same gradient; starting from
    identical parameters (the rank-0 broadcast) the SGD step (lr 0.001, as
    in the worked example) leaves the replicas bitwise equal."""
    ex = gen.linear_example(W=W, n=20, seed=0)
    numel = shapes.numels(shapes.linear_10x10())
    members, locs = assign_buckets(numel, 4, 25 << 20)
    _, outs = reduce_buckets(ex["grads"], members, locs, numel, n_out=W)
    start = [ex["weight"].reshape(-1).copy(), ex["bias"].copy()]
    after = [sgd_step(start, outs[r], 0.001) for r in range(W)]
    for r in range(1, W):
        for a, b in zip(after[0], after[r]):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    # ... whereas stepping on the local (unreduced) gradients diverges
    local = [sgd_step(start, ex["grads"][r], 0.001) for r in range(W)]
    assert not np.array_equal(local[0][0], local[1][0])
