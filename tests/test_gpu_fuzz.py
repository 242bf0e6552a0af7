"""Seeded random combinations of the fused bucket pass against the oracle.

The fixed parity cases vary one thing at a time; these draw whole
configurations: parameter count and a size mix (empty tensors, odd small
sizes, sizes around the vector and tile widths, an occasional large one),
W (including widths without a compiled-in body), f32 or bf16, the cap
(per-gradient to one bucket), the output mode (as-view, one copy, W
copies), misaligned views, a random ready order, every launch mode and
every kernel choice, and (for the batched call) the launch-coalescing
threshold.  Each case is compared bit for bit with the oracle,
with guard words around the arena and every output (see full_compare).
"""

import numpy as np
import pytest

from test_gpu_parity import full_compare

pytestmark = pytest.mark.gpu

SIZES = [0, 1, 2, 3, 4, 5, 7, 8, 15, 16, 17, 31, 63, 64, 65, 255, 1023, 1024, 1025, 2047, 4095, 4096, 4097,
         8191, 8193, 65535, 65537, 100003]
CAPS = [0, 1024, 16 * 1024, 256 * 1024, 1 << 20, 64 << 20]
WS = [1, 2, 3, 4, 5, 7, 8, 9, 16, 33]
MODES = ["mark_ready", "mark_ready_many", "reduce_all", "reduce_bucket"]
KERNELS = ["ldg", "tma", "auto", "chained"]
# DDP_OPT_COALESCE_ELEMS of mark_ready_many: one launch per event, tiny to large merges, the whole call
COALESCE = [0, 1, 1000, 65536, 1 << 21, 1 << 40]


def draw_case(seed):
    rng = np.random.default_rng(10_000 + seed)
    P = int(rng.integers(1, 41))
    numel = [int(rng.choice(SIZES)) for _ in range(P)]
    if rng.random() < 0.25:
        numel[int(rng.integers(P))] = 1 << 20      # one large tensor: many tiles, many CTAs
    W = int(rng.choice(WS))
    dtype = "f32" if rng.random() < 0.5 else "bf16"
    cap = int(rng.choice(CAPS))
    n_out = int(rng.choice([0, 1, W]))
    case = dict(numel=numel, W=W, dtype=dtype, cap=cap, n_out=n_out, odd=bool(rng.random() < 0.3),
                mode=str(rng.choice(MODES)), kernel=str(rng.choice(KERNELS)))
    case["coalesce"] = int(rng.choice(COALESCE))
    return case


@pytest.mark.parametrize("seed", range(200))
def test_fuzz_bucket_pass(seed):
    c = draw_case(seed)
    from reduction_reducer_gb300 import _lib
    full_compare(c["numel"], c["W"], c["dtype"], c["cap"], order="random", n_out=c["n_out"], mode=c["mode"],
                 odd=c["odd"], kernel=c["kernel"], options={_lib.OPT_COALESCE_ELEMS: c["coalesce"]})


# ---------------------------------------------------------------- unused parameters

def draw_sizes(rng, P):
    numel = [int(rng.choice(SIZES)) for _ in range(P)]
    if rng.random() < 0.25:
        numel[int(rng.integers(P))] = 1 << 20
    return numel


@pytest.mark.parametrize("seed", range(60))
def test_fuzz_unused_parameters(seed):
    """Random local-use masks (some variables unused on every replica, whose
    copy-backs must stay untouched) over random layouts, W up to 64, driven
    in one mark_ready_many call or one mark_ready call per event."""
    import torch
    from oracle.buckets import assign_buckets
    from oracle.unused import globally_used, reduce_with_unused
    from gpu_util import bits_equal, first_mismatch, host_grads, host_to_device_views
    from test_gpu_unused import _check_outputs, _guarded_outputs, _reducer

    rng = np.random.default_rng(20_000 + seed)
    P = int(rng.integers(1, 31))
    numel = draw_sizes(rng, P)
    W = int(rng.choice([1, 2, 3, 4, 8, 16, 33, 64]))
    dtype = "f32" if rng.random() < 0.5 else "bf16"
    cap = int(rng.choice(CAPS))
    kernel = str(rng.choice(["ldg", "tma", "auto"]))
    per_event = bool(seed % 3 == 2)
    n_out = int(rng.choice([1, W]))
    used = rng.random((W, P)) < float(rng.choice([0.3, 0.7, 0.95]))
    if not used.any():              # with no gradient anywhere no ready event occurs and nothing is reduced
        used[0, int(rng.integers(P))] = True
    flats, views, offs = host_grads(numel, W, dtype, odd=bool(rng.random() < 0.3))
    members, locs = assign_buckets(numel, 4 if dtype == "f32" else 2, cap)
    want_arena, want_outs = reduce_with_unused(views, used.tolist(), members, locs, numel, n_out=n_out)
    _, grads_dev = host_to_device_views(flats, numel, offs, dtype, "cuda")
    red = _reducer(numel, dtype, cap, kernel)
    arena = torch.full((red.arena_numel(),), float("nan"), device="cuda")
    bufs, out_views, out_offs = _guarded_outputs(numel, n_out)
    red.bind(grads_dev, arena, out_views[0] if n_out == 1 else out_views)
    red.set_local_used(used.tolist())
    from reduction_reducer_gb300 import _lib
    red.set_option(_lib.OPT_COALESCE_ELEMS, int(rng.choice(COALESCE)))
    red.begin_iteration()
    g = globally_used(used.tolist())
    order = [int(v) for v in rng.permutation(P) if g[v]]
    if per_event:
        for v in order:
            red.mark_ready(v)
    else:
        assert red.mark_ready_many(order) == len(order)
    torch.cuda.synchronize()
    assert red.device_status() == 0
    got = arena.cpu().numpy()
    assert bits_equal(got, want_arena), first_mismatch(got, want_arena)
    _check_outputs(bufs, out_offs, numel, want_outs, used.tolist())
    red.destroy()


# ---------------------------------------------------------------- fused last micro-step

@pytest.mark.parametrize("seed", range(60))
def test_fuzz_fused_last_step(seed):
    """K-1 accumulate micro-steps, then the K-th fused into the reduction,
    over random layouts, W, K, launch modes and kernels; the accumulated
    fields must come out unchanged."""
    import torch
    from oracle.buckets import assign_buckets
    from oracle.nosync import accumulate_steps, reduce_last_step
    from reduction_reducer_gb300 import Reducer, _lib
    from gpu_util import bits_equal, first_mismatch, host_grads, host_to_device_views
    from test_gpu_last_step import KERNEL, _drive, _fields

    rng = np.random.default_rng(30_000 + seed)
    P = int(rng.integers(1, 31))
    numel = draw_sizes(rng, P)
    W = int(rng.choice([1, 2, 3, 4, 5, 8, 16, 33]))
    K = int(rng.integers(2, 5))
    cap = int(rng.choice(CAPS))
    kernel = str(rng.choice(["ldg", "tma", "auto"]))
    mode = str(rng.choice(MODES))
    n_out = int(rng.choice([0, 1, W]))
    steps = [host_grads(numel, W, "f32", step=k) for k in range(K)]
    offs = steps[0][2]
    acc_np = [accumulate_steps([steps[k][1][r] for k in range(K - 1)]) for r in range(W)]
    members, locs = assign_buckets(numel, 4, cap)
    want_arena, want_outs = reduce_last_step(acc_np, steps[K - 1][1], members, locs, numel, n_out=max(n_out, 1))

    dev = [host_to_device_views(steps[k][0], numel, offs, "f32", "cuda")[1] for k in range(K)]
    acc_flat, acc = _fields(numel, W, odd=bool(rng.random() < 0.3))
    red = Reducer(numel, "f32", cap)
    red.set_option(_lib.OPT_KERNEL, KERNEL[kernel])
    arena = torch.full((red.arena_numel(),), float("nan"), device="cuda")
    outs = [[torch.full((n,), float("nan"), device="cuda") for n in numel] for _ in range(max(n_out, 1))]
    red.bind(acc, arena, None if n_out == 0 else (outs[0] if n_out == 1 else outs))
    for k in range(K - 1):
        red.accumulate_nosync(acc, dev[k], first_step=(k == 0))
    torch.cuda.synchronize()
    before = [f.clone() for f in acc_flat]
    red.bind_last_step(dev[K - 1])
    order = [int(v) for v in rng.permutation(P)]
    red.set_option(_lib.OPT_COALESCE_ELEMS, int(rng.choice(COALESCE)))
    _drive(red, mode, order)
    assert red.device_status() == 0
    got = arena.cpu().numpy()
    assert bits_equal(got, want_arena), first_mismatch(got, want_arena)
    for o in range(n_out):
        for v in range(P):
            assert bits_equal(outs[o][v].cpu().numpy(), want_outs[0][v]), (o, v)
    for r in range(W):
        assert torch.equal(acc_flat[r].view(torch.int32), before[r].view(torch.int32)), r
    red.destroy()


# ---------------------------------------------------------------- communication hooks

@pytest.mark.parametrize("seed", range(40))
def test_fuzz_hooks(seed):
    """The built-in hooks (mean, bf16 compression), inside the fused pass
    (even seeds) or through gather, hook and copy-back (odd seeds), over
    random layouts, W up to 33, dtypes, output modes and kernel choices."""
    import torch
    from oracle.buckets import assign_buckets
    from oracle.hooks import hook_bf16_compress, hook_mean, reduce_with_hook
    from reduction_reducer_gb300 import Reducer, _lib
    from gpu_util import bits_equal, first_mismatch, host_grads, host_to_device_views

    rng = np.random.default_rng(40_000 + seed)
    P = int(rng.integers(1, 31))
    numel = draw_sizes(rng, P)
    W = int(rng.choice([1, 2, 3, 4, 8, 16, 33]))
    dtype = "f32" if rng.random() < 0.5 else "bf16"
    cap = int(rng.choice(CAPS))
    hook = str(rng.choice(["mean", "bf16_compress"]))
    n_out = int(rng.choice([0, 1, W]))
    kernel = str(rng.choice(["ldg", "tma", "auto"]))
    flats, views, offs = host_grads(numel, W, dtype, odd=bool(rng.random() < 0.3))
    _, grads_dev = host_to_device_views(flats, numel, offs, dtype, "cuda")
    red = Reducer(numel, dtype, cap)
    red.set_option(_lib.OPT_KERNEL, {"ldg": _lib.KERNEL_LDG, "tma": _lib.KERNEL_TMA, "auto": _lib.KERNEL_AUTO}[kernel])
    N = red.arena_numel()
    arena = torch.full((N,), float("nan"), device="cuda")
    outs = [[torch.full((n,), float("nan"), device="cuda") for n in numel] for _ in range(max(n_out, 1))]
    red.bind(grads_dev, arena, None if n_out == 0 else (outs[0] if n_out == 1 else outs))
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    red.register_comm_hook(hook, [torch.empty(max(N, 1), dtype=tdt, device="cuda") for _ in range(W)])
    red.set_option(_lib.OPT_HOOK_FUSED, 1 if seed % 2 == 0 else 0)
    red.set_option(_lib.OPT_COALESCE_ELEMS, int(rng.choice(COALESCE)))
    members, locs = assign_buckets(numel, 4 if dtype == "f32" else 2, cap)
    fn = hook_mean if hook == "mean" else hook_bf16_compress
    want_arena, want_outs, _ = reduce_with_hook(views, members, locs, numel, fn, n_out=max(n_out, 1))
    red.begin_iteration()
    assert red.mark_ready_many([int(v) for v in rng.permutation(P)]) == P
    torch.cuda.synchronize()
    assert red.device_status() == 0
    got = arena.cpu().numpy()
    assert bits_equal(got, want_arena), first_mismatch(got, want_arena)
    for o in range(n_out):
        for v in range(P):
            assert bits_equal(outs[o][v].cpu().numpy(), want_outs[0][v]), (o, v)
    red.destroy()


# ---------------------------------------------------------------- bucket rebuild

@pytest.mark.parametrize("seed", range(40))
def test_fuzz_rebuild(seed):
    """An iteration records a random ready order; the buckets are re-packed
    from it with random first and later caps; the next iteration must match
    the oracle on the rebuilt layout through the same binding."""
    import torch
    from oracle.rebuild import rebuild_buckets
    from oracle.reduce import reduce_buckets
    from reduction_reducer_gb300 import Reducer, _lib
    from gpu_util import bits_equal, first_mismatch, host_grads, host_to_device_views

    rng = np.random.default_rng(50_000 + seed)
    P = int(rng.integers(1, 31))
    numel = draw_sizes(rng, P)
    W = int(rng.choice([1, 2, 3, 4, 8, 16]))
    dtype = "f32" if rng.random() < 0.5 else "bf16"
    elem = 4 if dtype == "f32" else 2
    kernel = str(rng.choice(["ldg", "tma", "auto"]))
    flats, views, offs = host_grads(numel, W, dtype, odd=bool(rng.random() < 0.3))
    _, grads_dev = host_to_device_views(flats, numel, offs, dtype, "cuda")
    red = Reducer(numel, dtype, int(rng.choice(CAPS)))
    red.set_option(_lib.OPT_KERNEL, {"ldg": _lib.KERNEL_LDG, "tma": _lib.KERNEL_TMA, "auto": _lib.KERNEL_AUTO}[kernel])
    arena = torch.full((red.arena_numel(),), float("nan"), device="cuda")
    outs = [torch.full((n,), float("nan"), device="cuda") for n in numel]
    red.bind(grads_dev, arena, outs)
    order = [int(v) for v in rng.permutation(P)]
    red.begin_iteration()
    red.mark_ready_many(order)
    torch.cuda.synchronize()
    assert red.get_ready_trace() == order
    first_cap, cap = int(rng.choice(CAPS)), int(rng.choice(CAPS))
    red.rebuild_buckets(None, first_cap, cap)
    arena.fill_(float("nan"))
    order2 = [int(v) for v in rng.permutation(P)]
    red.set_option(_lib.OPT_COALESCE_ELEMS, int(rng.choice(COALESCE)))
    red.begin_iteration()
    red.mark_ready_many(order2)
    torch.cuda.synchronize()
    members, locs = rebuild_buckets(numel, elem, order, first_cap, cap)
    want_arena, want_outs = reduce_buckets(views, members, locs, numel)
    assert red.B == len(members)
    assert red.device_status() == 0
    got = arena.cpu().numpy()
    assert bits_equal(got, want_arena), first_mismatch(got, want_arena)
    for v in range(P):
        assert bits_equal(outs[v].cpu().numpy(), want_outs[0][v]), v
    red.destroy()
