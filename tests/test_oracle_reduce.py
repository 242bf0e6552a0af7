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


def _f32_from_bits(u):
    return np.array([u], np.uint32).view(np.float32)


def test_sgd_step_hand_derived():
    """The SGD update p <- fl32(p - fl32(lr * g)) of the worked example (lr
    0.001, "Distributed Data Parallel" notes, "Example"), on values derived
    by hand; each case is chosen so that a flipped sign, a dropped or
    mis-scaled learning rate, or a missing product rounding changes the bits.

    fl32(0.001) = 0x3A83126F = 8589935 * 2^-33.
    (a) p = 1, g = 2^-10: lr*g = 8589935 * 2^-43 exactly (power-of-two
        scale); 1 - that lies 16.384 units of 2^-24 below 1, so the result
        is 1 - 16 * 2^-24 = 1 - 2^-20 = 0x3F7FFFF0.  p + lr*g would give
        1 + 2^-20 = 0x3F800008, dropping lr 1 - 2^-10 = 0x3F7FC000.
    (b) p = 2^-10, g = 3: lr*g = 25769805 * 2^-33 = 12884902.5 * 2^-32, a
        tie between mantissas 12884902 and 12884903; ties go to the even
        one, so fl32(lr*g) = 12884902 * 2^-32 = 0x3B449BA6, and
        p - it = (4194304 - 12884902) * 2^-32 = -8690598 * 2^-32, exact:
        0xBB049BA6.
    """
    got = sgd_step([np.array([1.0], F32)], [np.array([2.0 ** -10], F32)], 0.001)[0]
    assert got.view(np.uint32)[0] == 0x3F7FFFF0
    for wrong in (0x3F800008, 0x3F7FC000):
        assert got.view(np.uint32)[0] != wrong
    got = sgd_step([np.array([2.0 ** -10], F32)], [np.array([3.0], F32)], 0.001)[0]
    assert got.view(np.uint32)[0] == 0xBB049BA6
    # the product's rounding, checked on its own: fl32(0.001 * 3) is the even
    # neighbour of the tie
    assert (F32(0.001) * F32(3.0)).view(np.uint32) == 0x3B449BA6
    assert _f32_from_bits(0x3B449BA6)[0] == F32(12884902 * 2.0 ** -32)


def _round_f32(q: Fraction) -> np.float32:
    """Nearest fp32 to a rational in the normal range, ties to even, from
    integer arithmetic alone (exponent by comparison, scaled mantissa)."""
    if q == 0:
        return F32(0.0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = 0
    while a >= 2:
        a /= 2
        e += 1
    while a < 1:
        a *= 2
        e -= 1
    m = a * (1 << 23)                    # in [2^23, 2^24)
    lo = m.numerator // m.denominator
    rem = m - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return F32(sign * lo * 2.0 ** (e - 23))


def test_sgd_step_against_exact_rationals():
    """Seeded parameters and gradients of mixed magnitude: each result equals
    two correctly rounded steps of exact rational arithmetic -- the product
    lr*g rounded to fp32, then p minus it rounded to fp32."""
    rng = np.random.default_rng(7)
    p = (rng.standard_normal(400) * rng.choice([1e-3, 1.0, 30.0], 400)).astype(F32)
    g = (rng.standard_normal(400) * rng.choice([1e-6, 1e-3, 1.0], 400)).astype(F32)
    got = sgd_step([p], [g], 0.001)[0]
    lr = Fraction(float(F32(0.001)))
    for i in range(400):
        prod = _round_f32(lr * Fraction(float(g[i])))
        want = _round_f32(Fraction(float(p[i])) - Fraction(float(prod)))
        assert got[i].view(np.uint32) == want.view(np.uint32), (i, got[i], want)
