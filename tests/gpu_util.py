"""Helpers of the GPU parity tests: device buffers for the W replicas, the
run through the C ABI, and bitwise comparison with the oracle.

Replica gradients live in one flat device buffer per replica with the
parameters packed in registration order (``align`` elements between starts,
like separate allocations) or at deliberately odd offsets.
"""

from __future__ import annotations

import numpy as np
import torch

from oracle.buckets import assign_buckets
from oracle.nosync import accumulate, accumulate_steps
from oracle.reduce import reduce_buckets, replica_mean
from reduction_reducer_gb300 import Reducer
from workloads import gen

F32 = np.float32
TDT = {"f32": torch.float32, "bf16": torch.bfloat16}


def bits_equal(got: np.ndarray, want: np.ndarray) -> bool:
    """Bitwise equality of fp32 arrays, NaN compared as a class."""
    got = np.asarray(got, F32)
    want = np.asarray(want, F32)
    if got.shape != want.shape:
        return False
    if np.array_equal(got.view(np.uint32), want.view(np.uint32)):
        return True                          # every bit equal (the common case at full size)
    gn, wn = np.isnan(got), np.isnan(want)
    if not np.array_equal(gn, wn):
        return False
    return np.array_equal(got[~gn].view(np.uint32), want[~wn].view(np.uint32))


def first_mismatch(got, want):
    got = np.asarray(got, F32)
    want = np.asarray(want, F32)
    bad = ~((got.view(np.uint32) == want.view(np.uint32)) | (np.isnan(got) & np.isnan(want)))
    idx = np.flatnonzero(bad)
    return None if idx.size == 0 else (int(idx[0]), float(got[idx[0]]), float(want[idx[0]]), int(idx.size))


def to_host(t: torch.Tensor, dtype: str) -> np.ndarray:
    """A device buffer's contents on the host (bf16 as uint16 bit patterns)."""
    if dtype == "bf16":
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def check_every_element(numel, want_arena, want_outs, arena, out_flat, out_offs):
    """The whole bucket arena and every copied-back gradient against the
    oracle's, bit for bit."""
    got = arena.cpu().numpy()
    assert bits_equal(got, want_arena), first_mismatch(got, want_arena)
    del got
    host = out_flat.cpu().numpy()
    for v, (o, n) in enumerate(zip(out_offs, numel)):
        if n:
            assert bits_equal(host[o:o + n], want_outs[0][v]), (v, first_mismatch(host[o:o + n], want_outs[0][v]))


def host_to_device_views(flats_np, numel, offs, dtype, device):
    """Upload host flats (fp32 or bf16 bits) and return (flat tensors, views)."""
    flats, views = [], []
    for f in flats_np:
        if dtype == "bf16":
            t = torch.from_numpy(f.view(np.int16)).to(device).view(torch.bfloat16)
        else:
            t = torch.from_numpy(f).to(device)
        flats.append(t)
        views.append([t[o:o + n] for o, n in zip(offs, numel)])
    return flats, views


def layout(numel, align=64, odd=False):
    """Offsets of the parameters inside a replica's flat buffer."""
    if not odd:
        return gen.packed_offsets(numel, align)
    offs, cur = [], 0
    for i, n in enumerate(numel):
        cur += 1 + (i % 3)          # break every 16-byte phase
        offs.append(cur)
        cur += n
    return offs, cur + 3


def host_grads(numel, W, dtype, step=0, align=64, odd=False, special=False, seed_shift=0):
    """Host-drawn gradients: flats (per replica) and per-parameter numpy views."""
    offs, total = layout(numel, align, odd)
    flats = []
    for r in range(W):
        x = gen.draw_flat_np(total, r + seed_shift, step, "f32")
        if special:
            sv = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 2.0 ** -149, -2.0 ** -140,
                           3.4e38, -3.4e38, 1.0, 2.0 ** -24], F32)
            rng = np.random.default_rng(100 + r)
            pos = rng.choice(total, size=min(total, 4096), replace=False)
            x[pos] = sv[rng.integers(0, sv.size, size=pos.size)]
        flats.append(gen.f32_to_bf16_bits(x) if dtype == "bf16" else x)
    views = [[f[o:o + n] for o, n in zip(offs, numel)] for f in flats]
    return flats, views, offs


def run_path(red: Reducer, grads_dev, arena, outs, order=None, mode="mark_ready", stream=None):
    """Bind and run one iteration; mode: mark_ready | mark_ready_many |
    reduce_all | reduce_bucket."""
    red.bind(grads_dev, arena, outs)
    red.begin_iteration()
    if mode == "mark_ready":
        for v in order:
            red.mark_ready(v, stream)
    elif mode == "mark_ready_many":
        assert red.mark_ready_many(list(order), stream) == len(order)
    elif mode == "reduce_all":
        red.reduce_all(stream)
    elif mode == "reduce_bucket":
        for b in range(red.B):
            red.reduce_bucket(b, stream)
    else:
        raise ValueError(mode)
    torch.cuda.synchronize()


def sample_positions(numel, locs, starts, n_random=200_000, edge=40, seed=0):
    """Arena positions to check: random ones plus the first and last ``edge``
    elements of every parameter (heads, tails, segment boundaries)."""
    total = starts[-1]
    rng = np.random.default_rng(seed)
    pos = [rng.integers(0, total, size=min(n_random, total))] if total else []
    for v, n in enumerate(numel):
        if n == 0:
            continue
        lo = starts[locs[v].bucket] + locs[v].offset
        pos.append(np.arange(lo, lo + min(edge, n)))
        pos.append(np.arange(lo + max(0, n - edge), lo + n))
    if not pos:
        return np.zeros(0, np.int64)
    return np.unique(np.concatenate(pos)).astype(np.int64)


def arena_to_var(numel, locs, starts, pos):
    """Map arena positions to (variable, element index)."""
    # zero-length variables share their start with a neighbour: leave them out
    vs = np.array([v for v in range(len(numel)) if numel[v] > 0], np.int64)
    base = np.array([starts[locs[v].bucket] + locs[v].offset for v in vs], np.int64)
    order = np.argsort(base, kind="stable")
    k = np.searchsorted(base[order], pos, side="right") - 1
    var = vs[order[k]]
    j = pos - base[order[k]]
    assert np.all(j < np.array(numel, np.int64)[var]), "position outside its variable"
    return var, j


def sampled_check(numel, dtype, W, cap, flat_dev, offs, arena, outs, n_out, seed=0, n_random=200_000):
    """Oracle on sampled positions of a full-size run.  Inputs are read back
    from the replica buffers (written by the seeded generator, untouched by
    the kernels); the oracle computes the mean of exactly those values."""
    members, locs = assign_buckets(numel, 4 if dtype == "f32" else 2, cap)
    lens = [sum(numel[v] for v in m) for m in members]
    starts = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    pos = sample_positions(numel, locs, starts, n_random=n_random, seed=seed)
    var, j = arena_to_var(numel, locs, starts, pos)
    src_index = torch.from_numpy(np.array(offs, np.int64)[var] + j).to(flat_dev[0].device)
    xs = []
    for r in range(W):
        vals = flat_dev[r].index_select(0, src_index)
        if dtype == "bf16":
            xs.append(vals.view(torch.int16).cpu().numpy().view(np.uint16))
        else:
            xs.append(vals.cpu().numpy())
    want = replica_mean(xs)
    got_arena = arena.index_select(0, torch.from_numpy(pos).to(arena.device)).cpu().numpy()
    assert bits_equal(got_arena, want), first_mismatch(got_arena, want)
    for o in range(n_out):
        flat_out, out_offs = outs[o]
        got = flat_out.index_select(0, torch.from_numpy(np.array(out_offs, np.int64)[var] + j).to(arena.device))
        assert bits_equal(got.cpu().numpy(), want), first_mismatch(got.cpu().numpy(), want)
    return pos.size


def nosync_full_size_check(numel, offs, steps, acc_flat, arena, out_flat, K, fused_last, cap=25 << 20):
    """Every element of a no_sync block (K micro-steps, the last one fused
    into the reduction when ``fused_last``) against the oracle, one replica's
    steps on the host at a time: the accumulated fields the library left
    (after K, or K - 1 micro-steps when the last is fused: the reduction
    does not write them), then the arena and the copy-back."""
    members, locs = assign_buckets(numel, 4, cap)
    W = len(acc_flat)
    split = lambda h: [h[o:o + n] for o, n in zip(offs, numel)]
    reduced_inputs = []
    for r in range(W):
        per_step = [split(steps[k][r].cpu().numpy()) for k in range(K)]
        acc = accumulate_steps(per_step[:K - 1] if fused_last else per_step)
        got = split(acc_flat[r].cpu().numpy())
        for v in range(len(numel)):
            assert bits_equal(got[v], acc[v]), (r, v, first_mismatch(got[v], acc[v]))
        reduced_inputs.append(accumulate(acc, per_step[K - 1], first_step=False) if fused_last else acc)
        del per_step
    want_arena, want_outs = reduce_buckets(reduced_inputs, members, locs, numel)
    check_every_element(numel, want_arena, want_outs, arena, out_flat, offs)
