"""Pins of the communication-hook oracle (no GPU)."""

import numpy as np

from oracle.buckets import assign_buckets
from oracle.hooks import (f32_to_bf16_rne, gather_buckets, hook_bf16_compress, hook_mean,
                          reduce_with_hook)
from oracle.reduce import reduce_buckets, widen
from workloads import gen

F32 = np.float32


def _case(W=3, dtype="f32"):
    numel = [5, 0, 7, 3, 11]
    members, locs = assign_buckets(numel, 4, 24)
    rng = np.random.default_rng(4)
    grads = [[rng.standard_normal(n).astype(F32) for n in numel] for _ in range(W)]
    if dtype == "bf16":
        grads = [[f32_to_bf16_rne(g) for g in rep] for rep in grads]
    return numel, members, locs, grads


def test_gather_places_each_gradient_at_its_offset():
    numel, members, locs, grads = _case()
    bufs = gather_buckets(grads, members, locs, numel)
    for r in range(3):
        for v, n in enumerate(numel):
            b, lo = locs[v].bucket, locs[v].offset
            assert np.array_equal(bufs[r][b][lo:lo + n], grads[r][v])


def test_default_hook_is_the_fused_pass():
    for dtype in ("f32", "bf16"):
        numel, members, locs, grads = _case(dtype=dtype)
        a1, o1, calls = reduce_with_hook(grads, members, locs, numel, hook_mean)
        a2, o2 = reduce_buckets(grads, members, locs, numel)
        assert np.array_equal(a1.view(np.uint32), a2.view(np.uint32))
        assert all(np.array_equal(x, y) for x, y in zip(o1[0], o2[0]))
        B = len(members)
        assert calls == [(b, B, b == B - 1) for b in range(B)]


def test_bf16_compress_exact_on_bf16_values():
    # values already representable in bf16 are not changed by the compression
    numel, members, locs, grads = _case(dtype="bf16")
    wide = [[widen(g).copy() for g in rep] for rep in grads]
    a1, _, _ = reduce_with_hook(wide, members, locs, numel, hook_bf16_compress)
    a2, _ = reduce_buckets(grads, members, locs, numel)
    assert np.array_equal(a1.view(np.uint32), a2.view(np.uint32))


def test_bf16_rounding_known_cases():
    x = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 3.0], F32)
    assert list(f32_to_bf16_rne(x)) == [0x3F80, 0x3F82, 0xBF80, 0x4040]
    # mean of [1 + 2^-8] and [1 + 3 * 2^-8] after compression: (1 + (1 + 2^-6)) / 2
    out = hook_bf16_compress([x[:1], x[1:2]])
    assert out[0] == F32((1.0 + (1.0 + 2.0 ** -6)) / 2)
    assert hook_mean([x[:1], x[1:2]])[0] == F32(1.0 + 2.0 ** -7)


def test_workload_shapes_roundtrip():
    numel = [100, 10]
    members, locs = assign_buckets(numel, 4, 25 << 20)
    ex = gen.linear_example(W=2)
    arena, outs, calls = reduce_with_hook(ex["grads"], members, locs, numel, hook_mean)
    assert calls == [(0, 1, True)]
    assert not np.isnan(arena).any()


def test_bf16_rounding_matches_library_conversion():
    """f32 -> bf16 round to nearest even, pinned to a library routine (torch's
    CPU conversion) over 2^20 random bit patterns of every exponent, exact
    ties, the overflow edge (values above the largest bf16 round to Inf),
    subnormals, signed zeros, infinities and NaN (NaN compared as a class).
    The workloads' input generator rounds the same way."""
    import torch
    from workloads.gen import f32_to_bf16_bits
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 1 << 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    ties = (rng.integers(0, 1 << 16, size=4096, dtype=np.uint64).astype(np.uint32) << 16) | np.uint32(0x8000)
    edge = np.array([0x7F7F7FFF, 0x7F7F8000, 0x7F7F8001, 0x7F7FFFFF, 0xFF7FFFFF, 0x00000001, 0x80000001,
                     0x007FFFFF, 0x00008000, 0x00018000, 0x00000000, 0x80000000, 0x7F800000, 0xFF800000,
                     0x7FC00000, 0x7F800001, 0xFFFFFFFF], np.uint32)
    x = np.concatenate([bits, ties, edge]).view(np.float32)
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    for fn in (f32_to_bf16_rne, f32_to_bf16_bits):
        got = fn(x)
        assert np.array_equal(got[~nan], want[~nan])
        # NaN stays NaN: exponent all ones, non-zero mantissa
        assert np.all((got[nan] & 0x7F80) == 0x7F80) and np.all((got[nan] & 0x007F) != 0)
