"""Seeded synthetic inputs: per-replica gradients, ready orders, the Linear example.

Shared by the oracle-side tests and the GPU side; holds none of the
reducer's arithmetic (no bucketing, no readiness logic, no averaging).

Seeding convention (one rule for every workload):
  replica ``r`` at local step ``k`` draws its gradients from generator seed
  ``1000 * k + r``; single-step workloads use ``k = 0``.  Values are
  ``N(0, 1) * 1e-3`` in fp32; bf16 gradients are the round-to-nearest-even
  cast of that fp32 draw.

Two generators exist: NumPy's PCG64 (host, any size, used by CPU tests and
small GPU parity cases that copy host data to the device) and torch's CUDA
generator (device, used for the full-size workloads where host generation
would dominate).  They produce different streams; a test always compares
both sides on the *same* buffer contents.
"""

from __future__ import annotations

import random

import numpy as np

STD = np.float32(1e-3)


def seed_of(replica: int, step: int = 0) -> int:
    return 1000 * step + replica


# ---------------------------------------------------------------- dtype helpers

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16, returned as uint16 bit patterns.

    Input preparation only (the bf16 workloads store bf16 gradients).
    NaNs are kept quiet NaNs.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = ((u[nan] >> np.uint64(16)) | np.uint64(0x40)).astype(np.uint16)
    return r


# ---------------------------------------------------------------- layouts

def packed_offsets(numels, align: int = 1):
    """Element offsets of tensors packed in registration order into one flat
    buffer, each start rounded up to a multiple of ``align`` elements.
    Returns (offsets, total_elements)."""
    offs, cur = [], 0
    for n in numels:
        cur = -(-cur // align) * align
        offs.append(cur)
        cur += int(n)
    cur = -(-cur // align) * align
    return offs, cur


# ---------------------------------------------------------------- gradient draws (host)

def draw_flat_np(n: int, replica: int, step: int = 0, dtype: str = "f32") -> np.ndarray:
    """One replica's flat draw of ``n`` values (fp32 array, or uint16 bf16 bits)."""
    rng = np.random.default_rng(seed_of(replica, step))
    x = rng.standard_normal(n, dtype=np.float32) * STD
    if dtype == "f32":
        return x
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    raise ValueError(dtype)


def draw_grads_np(numels, W: int, step: int = 0, dtype: str = "f32", align: int = 1):
    """Per-replica gradients on the host.

    Returns ``(flats, views)``: ``flats[r]`` is replica r's flat buffer with
    tensors packed in registration order (``align``-element aligned starts),
    ``views[r][v]`` the 1-D view of tensor v inside it.
    """
    offs, total = packed_offsets(numels, align)
    flats, views = [], []
    for r in range(W):
        flat = draw_flat_np(total, r, step, dtype)
        flats.append(flat)
        views.append([flat[o:o + n] for o, n in zip(offs, numels)])
    return flats, views


# ---------------------------------------------------------------- gradient draws (device)

def draw_flat_torch(n: int, replica: int, step: int = 0, dtype: str = "f32", device="cuda", out=None):
    """One replica's flat draw generated directly on ``device`` with torch's
    generator for that device (fp32 ``randn * 1e-3``, bf16 = RNE cast)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed_of(replica, step))
    x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
    x.mul_(1e-3)
    if dtype == "bf16":
        x = x.to(torch.bfloat16)
    elif dtype != "f32":
        raise ValueError(dtype)
    if out is not None:
        out.copy_(x)
        return out
    return x


# ---------------------------------------------------------------- ready orders

def reverse_order(P: int) -> list[int]:
    """Exact reverse of registration order: P-1, ..., 0."""
    return list(range(P - 1, -1, -1))


def straggler_order(bucket_members, p: float = 0.25, seed: int = 0) -> list[int]:
    """Reverse order with seeded straggler moves across bucket boundaries.

    ``bucket_members[b]`` lists bucket b's variables in push order (an input:
    the layout itself is computed elsewhere).  For each boundary b -> b+1 in
    turn, with probability ``p`` (``random.Random(seed)``, one draw per
    boundary), bucket b's last-pushed member (its lowest variable index) is
    moved to just after bucket b+1's last-pushed member in the ready order,
    so bucket b+1 completes first and has to wait for bucket b.
    """
    P = sum(len(m) for m in bucket_members)
    order = reverse_order(P)
    rng = random.Random(seed)
    for b in range(len(bucket_members) - 1):
        draw = rng.random()
        if draw >= p or not bucket_members[b] or not bucket_members[b + 1]:
            continue
        v = bucket_members[b][-1]
        u = bucket_members[b + 1][-1]
        order.remove(v)
        order.insert(order.index(u) + 1, v)
    return order


# ---------------------------------------------------------------- the Linear(10,10) example

def linear_example(W: int = 2, n: int = 20, seed: int = 0):
    """Inputs and per-replica gradients of the worked DDP example.

    One ``Linear(10, 10)`` initialised from seed ``seed`` (uniform in
    +-1/sqrt(10), the default fan-in bound; every replica holds the same
    values, as after the rank-0 broadcast), replica r's input
    ``randn(n, 10)`` from seed ``seed + r``, loss ``mean(out**2)``.

    Returns a dict with ``weight`` (10x10), ``bias`` (10,), ``x`` (list of
    W arrays n x 10) and ``grads`` (list of W lists ``[dweight(100,),
    dbias(10,)]`` in registration order), all fp32.  The gradients are
    the model's backward pass (input preparation for the reducer).
    """
    rng = np.random.default_rng(seed)
    bound = np.float32(1.0 / np.sqrt(10.0))
    weight = rng.uniform(-bound, bound, size=(10, 10)).astype(np.float32)
    bias = rng.uniform(-bound, bound, size=(10,)).astype(np.float32)
    xs, grads = [], []
    for r in range(W):
        x = np.random.default_rng(seed + r).standard_normal((n, 10), dtype=np.float32)
        out = x @ weight.T + bias                      # (n, 10)
        gout = (np.float32(2.0) / np.float32(n * 10)) * out
        dw = (gout.T @ x).astype(np.float32)           # (10, 10)
        db = gout.sum(axis=0, dtype=np.float32)
        xs.append(x)
        grads.append([np.ascontiguousarray(dw).reshape(-1), np.ascontiguousarray(db)])
    return dict(weight=weight, bias=bias, x=xs, grads=grads)
