"""Benchmark of the DDP Reducer gradient path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one reducer iteration of the BERT-large-shaped workload (391
fp32 tensors, 335,141,888 elements, W = 4 replicas resident in HBM, 25 MiB
buckets -> 37 buckets): ``begin_iteration`` then ``mark_ready`` for every
parameter in the stored straggler ready order; each released bucket range
is one fused launch (gather of the W replicas' per-parameter gradients,
fp32 rank-order sum, x 1/W, bucket write, copy-back).  The bucket build is
construction time and is not in the step.

Metric: algorithmic HBM bytes per step / time, in GB/s, where the bytes are
W*N*4 (replica reads) + N*4 (bucket write) + N*4 (copy-back write); gradient
elements per second are W*N / time.  Inputs (5.4 GB read per step) exceed
the 129 MB L2, so no flush is needed between steps.

Prints ONE JSON line on rank 0.  Under torchrun (N > 1) every rank runs its
own independent replica of the workload (the W replicas of one emulation
live on one GPU and need no collective: "replicas only"); value = total
bytes over ranks / max time over ranks.  The same run then times the
bucket all-reduce split across the N ranks (one replica per rank, NCCL) as
``per_config["bert_large_sharded_allreduce"]``; ``--sharded`` times that
alone as the main line (``--replicas-per-rank`` replicas on each rank).

``--impl reference`` times the CPU oracle (the plain NumPy restatement of the
same path) on a bounded sample of the same workload on the host cores.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from workloads import gen, shapes  # noqa: E402

MIB = 1 << 20
METRIC = "fused bucket-reduce HBM GB/s and % of GB300 peak; gradient elems/s at W replicas"
KERNEL_SRCS = [os.path.join(ROOT, "reduction_reducer_gb300", "csrc", f)
               for f in ("ddp_kernels_tma.cu", "ddp_device.cuh")]
ORDER_FILE = os.path.join(ROOT, "tests", "golden", "bert_large_ready_order.txt")
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
NOMINAL_HBM_GBS = 8000.0


# ---------------------------------------------------------------- helpers

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_hash() -> str:
    """Hash of the dominant kernel's sources, to tell whether the committed
    ncu traffic figure still describes the kernel that runs."""
    h = hashlib.sha256()
    for path in KERNEL_SRCS:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_order(path=ORDER_FILE):
    with open(path) as f:
        return [int(l) for l in f if l.strip() and not l.startswith("#")]


def view_bytes(W, N, s_in, n_out=1):
    return W * N * s_in + N * 4 + n_out * N * 4


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 100 ms with host
    arrival times, so samples can be matched to the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id=None):
        self.samples = []
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "100"]
        if bus_id:
            cmd += ["-i", bus_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                self.samples.append((time.time(), float(parts[0]), float(parts[1]), parts[3:7]))
            except ValueError:
                continue

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        inside = [s for s in self.samples if t0 <= s[0] <= t1 + 0.1]
        window = "timed region"
        if not inside:
            inside = [s for s in self.samples if t0 - 1.0 <= s[0] <= t1 + 1.0]
            window = "timed region +-1 s (region shorter than the 100 ms sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "no samples"}
        reasons = sorted({names[i] for s in inside for i, v in enumerate(s[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": max(s[2] for s in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


# ---------------------------------------------------------------- workloads on the device

class Workload:
    """Device buffers, reducer and step function of one configuration."""

    def __init__(self, name, torch, device, cap_mib=25, n_out=1, driver="hooks", layout="params", layers=None,
                 lib_path=None):
        from reduction_reducer_gb300 import Reducer
        self.torch = torch
        spec = shapes.WORKLOADS[name]
        self.name = name
        self.W = spec["W"]
        self.dtype = spec["dtype"]
        self.s_in = 4 if self.dtype == "f32" else 2
        self.layers = layers
        self.numel = shapes.numels(spec["shapes"]() if layers is None else spec["shapes"](layers=layers))
        self.P = len(self.numel)
        self.N = sum(self.numel)
        self.cap = cap_mib * MIB
        self.n_out = n_out
        self.driver = driver
        self.red = Reducer(self.numel, self.dtype, self.cap, **({"lib_path": lib_path} if lib_path else {}))
        self.B = self.red.B
        if layout == "params":          # per-parameter tensors, registration order
            offs, total = gen.packed_offsets(self.numel, 64)
        else:                           # replicas laid out as their buckets (as-view)
            _, boff = self.red.get_bucket_info()
            locs = self.red.get_locators()
            offs = [boff[b] + off for (b, _, off, _) in locs]
            total = boff[-1]
        self.offs, self.total = offs, total
        self.flat = [gen.draw_flat_torch(total, r, 0, self.dtype, device) for r in range(self.W)]
        self.grads = [[f[o:o + n] for o, n in zip(offs, self.numel)] for f in self.flat]
        self.arena = torch.empty(self.red.arena_numel(), dtype=torch.float32, device=device)
        if n_out:
            out_offs, out_total = gen.packed_offsets(self.numel, 64)
            self.out_flat = torch.empty(out_total, dtype=torch.float32, device=device)
            outs = [self.out_flat[o:o + n] for o, n in zip(out_offs, self.numel)]
        else:
            self.out_flat, outs = None, None
        self.red.bind(self.grads, self.arena, outs)
        if spec["order"] == "straggler" and name == "bert_large" and cap_mib == 25 and layers is None:
            self.order = read_order()
        else:
            self.order = gen.reverse_order(self.P)
        self.bytes = view_bytes(self.W, self.N, self.s_in, n_out)
        import ctypes
        self._order_c = (ctypes.c_int32 * len(self.order))(*self.order)

    def step(self, stream):
        red = self.red
        if self.driver == "hooks":          # the ready order reported in one call
            red.begin_iteration()
            red.mark_ready_many(self._order_c, stream)
        elif self.driver == "events":       # one mark_ready call per event
            red.begin_iteration()
            for v in self.order:
                red.mark_ready(v, stream)
        else:
            red.reduce_all(stream)

    def free(self):
        self.red.destroy()
        self.flat = self.grads = self.arena = self.out_flat = None


def max_over_ranks(value: float, dist, device) -> float:
    """Largest value over the process group (the slowest rank's time)."""
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def time_steps(torch, stream, fn, steps, warmup, dist=None):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    ms = start.elapsed_time(end)
    if dist:
        ms = max_over_ranks(ms, dist, "cuda")
        dist.barrier()
    return ms, t0, t1


def kernel_name(wl) -> str:
    """The bucket kernel a workload's iteration launches: the context's
    choice, except that with the automatic choice one mark_ready call per
    event (calls not chained) launches the bulk-copy kernel."""
    from reduction_reducer_gb300 import _lib
    k = wl.red.get_option(_lib.OPT_QUERY_KERNEL)
    t = "float" if wl.dtype == "f32" else "uint16_t"
    tma, ldg = f"bucket_reduce_tma_kernel<{t}, {wl.W}>", f"bucket_reduce_kernel<{t}, {wl.W}>"
    if k == _lib.KERNEL_TMA:
        return tma
    if (wl.driver == "events" and wl.red.get_option(_lib.OPT_KERNEL) == _lib.KERNEL_AUTO
            and not wl.red.get_option(_lib.OPT_CHAINED)):
        return tma
    return ldg


def traffic_for(kernel_key, alg_bytes_per_launch):
    """DRAM bytes per launch from the committed ncu summary: the measured
    ratio of DRAM bytes to algorithmic bytes on the captured case, scaled to
    this launch's algorithmic bytes; None when the kernel source changed
    since the capture."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            d = json.load(f)
    except Exception:
        return None
    e = d.get(kernel_key)
    if not e or e.get("kernel_sha") != kernel_hash():
        return None
    return e["dram_bytes_per_algorithmic_byte"] * alg_bytes_per_launch


# ---------------------------------------------------------------- CPU oracle timing

def oracle_sample_model(name="bert_large", cap_mib=25, n_buckets=3):
    """Host inputs of a CPU-oracle sample: the tensors of the first
    ``n_buckets`` buckets of a configuration's layout, as a model of their
    own (their reverse walk closes the same buckets, so the oracle does the
    sample's work and allocates an arena of the sample's size, not the whole
    model's), with seeded N(0, 1e-3) draws per replica in the
    configuration's dtype."""
    from oracle.buckets import assign_buckets
    spec = shapes.WORKLOADS[name]
    full = shapes.numels(spec["shapes"]())
    W, dtype = spec["W"], spec["dtype"]
    s_in = 4 if dtype == "f32" else 2
    members, _ = assign_buckets(full, s_in, cap_mib * MIB)
    n_buckets = min(n_buckets, len(members))
    vars_ = sorted(v for b in range(n_buckets) for v in members[b])
    numel = [full[v] for v in vars_]
    sub_members, locs = assign_buckets(numel, s_in, cap_mib * MIB)
    assert [sorted(vars_[i] for i in m) for m in sub_members] == [sorted(members[b]) for b in range(n_buckets)]
    offs, total = gen.packed_offsets(numel)
    grads = []
    for r in range(W):
        flat = gen.draw_flat_np(total, r, 0, dtype)
        grads.append([flat[o:o + n] for o, n in zip(offs, numel)])
    n_el = sum(numel)
    desc = (f"buckets 0..{n_buckets - 1} of the {name} {cap_mib} MiB layout ({len(vars_)} tensors, {n_el} elements, "
            f"W={W}, {dtype})")
    return dict(numel=numel, W=W, s_in=s_in, members=sub_members, locs=locs, grads=grads, n_el=n_el, desc=desc)


def oracle_sample_inputs(max_buckets: int = 3):
    """The BERT-large sample of ``cpu_baseline`` and the reference arm."""
    return oracle_sample_model("bert_large", 25, max_buckets)


def _time_until(fn, target_s):
    fn()                                   # untimed first call (page faults of fresh memory)
    reps, t = 0, 0.0
    while t < target_s:
        t0 = time.perf_counter()
        fn()
        t += time.perf_counter() - t0
        reps += 1
    return reps, t


def oracle_sample_gbs(target_s: float, max_buckets: int = 3, inputs=None):
    """Time the CPU oracle on the sample, repeating until ``target_s`` of
    oracle work; input generation is outside the timing."""
    from oracle.reduce import reduce_buckets
    d = inputs or oracle_sample_inputs(max_buckets)
    reps, t = _time_until(lambda: reduce_buckets(d["grads"], d["members"], d["locs"], d["numel"]), target_s)
    gbs = view_bytes(d["W"], d["n_el"], d["s_in"]) * reps / t / 1e9
    sample = f"{d['desc']} x {reps} repetitions, {t:.1f} s of oracle work"
    return gbs, sample, t


def cpu_threads_used():
    return 1   # NumPy elementwise ufuncs run on the calling thread


def oracle_config_sample(name, cap_mib, target_s=2.0):
    """The CPU oracle timed on one configuration's own layout: its first
    bucket (seeded draws, the configuration's W and dtype), reduced
    repeatedly until ``target_s`` of oracle work; same byte formula as the
    GPU line.  For the no_sync configuration the adding micro-step is timed
    on the same bucket (12 bytes per replica element)."""
    from oracle.nosync import accumulate
    from oracle.reduce import reduce_buckets
    d = oracle_sample_model(name, cap_mib, 1)
    W, n_el = d["W"], d["n_el"]
    reps, t = _time_until(lambda: reduce_buckets(d["grads"], d["members"], d["locs"], d["numel"]), target_s)
    out = {"gbs": round(view_bytes(W, n_el, d["s_in"]) * reps / t / 1e9, 3), "us_per_reduce": round(1e6 * t / reps, 1),
           "cores": cpu_threads_used(), "kind": "oracle",
           "sample": f"{d['desc']} x {reps} repetitions, {t:.1f} s of oracle work"}
    if shapes.WORKLOADS[name].get("K"):
        acc = [[x.copy() for x in g] for g in d["grads"]]
        reps_a, t_a = _time_until(lambda: [accumulate(acc[r], d["grads"][r], first_step=False) for r in range(W)],
                                  target_s)
        out["accumulate_gbs"] = round(3 * W * n_el * 4 * reps_a / t_a / 1e9, 3)
    return out


def add_cpu_oracle(per_config, target_s=2.0):
    """A bounded CPU-oracle sample beside each configuration's GPU line."""
    for key, name, cap in (("linear_w2", "linear", 25), ("resnet50_w8", "resnet50", 25),
                           ("bert_large_reduce_all", "bert_large", 25),
                           *((f"gpt2_medium_w8_bf16_cap{c}", "gpt2_medium", c) for c in (0, 1, 5, 25, 100)),
                           ("nosync_resnet50_w16_k8", "nosync_resnet50", 25)):
        if key in per_config:
            per_config[key]["cpu_oracle"] = oracle_config_sample(name, cap, target_s)


# ---------------------------------------------------------------- arms

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    per_step = []
    inputs = oracle_sample_inputs(max_buckets=2)
    for i in range(args.warmup + args.steps):
        gbs, sample, t = oracle_sample_gbs(args.ref_step_s, inputs=inputs)
        if i >= args.warmup:
            per_step.append((gbs, t))
    total_t = sum(t for _, t in per_step)
    value = statistics.median(g for g, _ in per_step)
    numel = shapes.numels(shapes.bert_large())
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1000 * total_t / max(1, len(per_step)), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "bert_large", "W": 4, "P": len(numel), "N": sum(numel), "cap_mib": 25,
                   "mode": "copy-back (n_out=1)", "sample": "bounded sample, see cpu_baseline"},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": cpu_threads_used(),
                         "kind": "oracle", "sample": sample,
                         "host_cpus": os.cpu_count(), "affinity": len(os.sched_getaffinity(0))},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_nosync_only(args):
    """The no_sync workload alone (ResNet-50, W=16, K micro-steps + reduce):
    a compact case for profiling the accumulate kernel."""
    import torch
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=device)
    res = nosync_config(torch, device, stream, args.steps, args.warmup, None, K=args.nosync_k, kernel=args.kernel)
    print(json.dumps({"workload": f"nosync_resnet50_w16_k{args.nosync_k}", **res}), flush=True)
    return 0


def run_gpt2_only(args):
    """The GPT-2-medium workload alone (W=8 bf16 at --cap-mib, reverse ready
    order, one mark_ready_many call per step): a compact case for profiling
    the per-gradient (cap 0) and small-bucket launches."""
    import torch
    from reduction_reducer_gb300 import _lib
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=device)
    wl = Workload("gpt2_medium", torch, device, args.cap_mib, n_out=1, driver=args.driver, layers=args.layers)
    if args.kernel != "auto":
        wl.red.set_option(_lib.OPT_KERNEL, KERNEL_FLAG[args.kernel])
    with torch.cuda.stream(stream):
        ms, _, _ = time_steps(torch, stream, lambda: wl.step(stream), args.steps, args.warmup)
    t = ms / args.steps
    name = "gpt2_medium" if args.layers is None else f"gpt2_medium_{args.layers}layers"
    print(json.dumps({"workload": f"{name}_w8_bf16_cap{args.cap_mib}", "gbs": round(wl.bytes / (t * 1e-3) / 1e9, 1),
                      "ms_per_step": round(t, 4), "buckets": wl.B, "kernel": kernel_name(wl)}), flush=True)
    wl.free()
    return 0


def sharded_timing(torch, dist, device, rank, world, Wl, steps, warmup):
    """Time the bucket all-reduce across the ranks of the default process
    group, every rank holding Wl replicas of BERT-large (25 MiB buckets,
    stored straggler order): per bucket, in bucket-index order, gather into
    the bucket buffers, all-to-alls of the raw chunks, the owner's mean in
    replica order, all-gather, copy-back.  Bytes per rank and step: Wl*N*4
    read + 2*N*4 written (the fused pass's algorithmic bytes at W = Wl)."""
    from reduction_reducer_gb300 import Reducer
    from reduction_reducer_gb300.sharded import sharded_hook, verify_layout
    stream = torch.cuda.Stream(device=device)
    numel = shapes.numels(shapes.bert_large())
    offs, total = gen.packed_offsets(numel, 64)
    flats = [gen.draw_flat_torch(total, rank * Wl + r, 0, "f32", device) for r in range(Wl)]
    grads = [[f[o:o + n] for o, n in zip(offs, numel)] for f in flats]
    red = Reducer(numel, "f32", 25 * MIB)
    arena = torch.empty(red.arena_numel(), device=device)
    out_flat = torch.empty(total, device=device)
    red.bind(grads, arena, [out_flat[o:o + n] for o, n in zip(offs, numel)])
    rbs = [torch.empty(red.arena_numel(), device=device) for _ in range(Wl)]
    verify_layout(dist, red)                      # every rank must pair the same buckets
    red.register_comm_hook(sharded_hook(dist, rbs, arena, dtype="f32"), rbs)
    order = read_order()

    def step():
        red.begin_iteration()
        red.mark_ready_many(order, stream)

    with torch.cuda.stream(stream):
        ms, _, _ = time_steps(torch, stream, step, steps, warmup, dist if world > 1 else None)
    N = sum(numel)
    per_rank = Wl * N * 4 + 2 * N * 4
    t = ms / steps
    B = red.B
    red.destroy()
    del flats, grads, arena, out_flat, rbs
    torch.cuda.empty_cache()
    return {"gbs": round(per_rank * world / (t * 1e-3) / 1e9, 1), "ms_per_step": round(t, 4), "ranks": world,
            "replicas_per_rank": Wl, "W": world * Wl, "P": len(numel), "N": N, "buckets": B,
            "bytes_per_rank_step": per_rank,
            "note": f"bucket all-reduce across {world} NCCL rank(s), {Wl} replica(s) each: all-to-all of raw "
                    "chunks, owner mean, all-gather, in bucket order; gbs = bytes of all ranks / slowest rank"}


def run_sharded(args):
    """The bucket all-reduce across ranks that each hold Wl replicas
    (--replicas-per-rank, default one; one rank per GPU under torchrun,
    NCCL), timed by ``sharded_timing``; value = the bytes of all ranks / the
    slowest rank's time (weak scaling: per-rank work is fixed)."""
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1 or "MASTER_ADDR" in os.environ:
        dist.init_process_group("nccl", device_id=device)
    else:
        dist.init_process_group("nccl", store=dist.HashStore(), rank=0, world_size=1, device_id=device)
    r = sharded_timing(torch, dist, device, rank, world, args.replicas_per_rank, args.steps, args.warmup)
    if rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": r["gbs"], "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": f"synthetic (seeded N(0,1e-3) gradients generated on the device, {r['replicas_per_rank']} "
                    "replica(s) per rank)",
            "config": {"workload": "bert_large", "W": r["W"], "replicas_per_rank": r["replicas_per_rank"],
                       "P": r["P"], "N": r["N"], "cap_mib": 25, "buckets": r["buckets"], "mode": "copy-back (n_out=1)",
                       "parallelism": f"sharded all-reduce x{world} (all-to-all of raw chunks, owner mean, all-gather)",
                       "bytes_per_rank_step": r["bytes_per_rank_step"]}}), flush=True)
    dist.destroy_process_group()
    return 0


def run_mix_rates(args):
    """Roofline context: the streaming rate GB300's HBM gives plain torch
    kernels by read:write mix (4 GiB fp32 buffers, best of 20 with CUDA
    events), beside the fused pass on the BERT-large shapes for W = 1 .. 32
    replicas (one mark_ready_many call, reverse order, library defaults).
    The pass at W replicas reads W and writes 2 units per element: at W = 4
    it has the 2:1 mix of torch.add."""
    import torch
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)

    def best_ms(fn, reps=20, warm=3):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(b))
        return best

    n = 1 << 30
    x = torch.empty(n, device=dev).normal_()
    y = torch.empty(n, device=dev).normal_()
    z = torch.empty(n, device=dev)
    out = {}
    for name, fn, nbytes in (("torch copy_ (1 read : 1 write)", lambda: z.copy_(x), 8 * n),
                             ("torch add (2 reads : 1 write)", lambda: torch.add(x, y, out=z), 12 * n),
                             ("torch fill_ (write only)", lambda: z.fill_(1.0), 4 * n),
                             ("torch sum (read only)", lambda: x.sum(), 4 * n)):
        ms = best_ms(fn)
        out[name] = {"gbs": round(nbytes / (ms * 1e-3) / 1e9, 1), "ms": round(ms, 3)}
    del x, y, z
    torch.cuda.empty_cache()
    stream = torch.cuda.Stream(device=dev)
    for W, r in replica_sweep(torch, dev, stream, (1, 2, 4, 8, 16, 32), args.steps, args.warmup).items():
        out[f"fused pass, BERT-large shapes, W={W} ({W} reads : 2 writes)"] = r
    print(json.dumps({"mix_rates": out}), flush=True)
    return 0


def replica_sweep(torch, dev, stream, Ws, steps, warmup, dist=None):
    """The fused pass on the BERT-large shapes (fp32, 25 MiB buckets, reverse
    order, library defaults, one mark_ready_many call, one copy-back) for
    each replica count in Ws: {W: {"gbs", "ms"}} of its algorithmic bytes
    (W reads and 2 writes per element)."""
    from reduction_reducer_gb300 import Reducer
    numel = shapes.numels(shapes.bert_large())
    offs, total = gen.packed_offsets(numel, 64)
    order = gen.reverse_order(len(numel))
    N = sum(numel)
    out = {}
    for W in Ws:
        flat = [gen.draw_flat_torch(total, r, 0, "f32", dev) for r in range(W)]
        grads = [[f[o:o + k] for o, k in zip(offs, numel)] for f in flat]
        red = Reducer(numel, "f32", 25 * MIB)
        arena = torch.empty(red.arena_numel(), device=dev)
        res = torch.empty(total, device=dev)
        red.bind(grads, arena, [res[o:o + k] for o, k in zip(offs, numel)])

        def step():
            red.begin_iteration()
            red.mark_ready_many(order, stream)
        with torch.cuda.stream(stream):
            ms, _, _ = time_steps(torch, stream, step, steps, warmup, dist)
        t = ms / steps
        out[W] = {"gbs": round(view_bytes(W, N, 4) / (t * 1e-3) / 1e9, 1), "ms": round(t, 4)}
        red.destroy()
        del flat, grads, arena, res
        torch.cuda.empty_cache()
    return out


def run_trace(args):
    """Launch boundaries of one BERT-large iteration taken apart, from the
    trace build's per-CTA %globaltimer stamps (libddpreducer_trace.so, built
    here when missing): for every pair of consecutive launches A -> B, with
    one mark_ready call per event (B waits for A) and in one mark_ready_many
    call (B chained after A).  Stamps: t0 CTA entry, t1 past the wait (past
    the trigger when chained), t2 first stage consumed, t3 last stage
    consumed.  Per pair: A's tail (last t3 - 90th percentile of A's t3: the
    time its last tenth of CTAs takes to finish), B's release (first t1 of
    B - last t3 of A), B's first data after its release, and the gap between
    A's last and B's first consumed stage (negative: they overlap)."""
    import torch
    from reduction_reducer_gb300 import _lib, build
    from reduction_reducer_gb300.reducer import read_launch_trace
    if not os.path.exists(_lib.TRACE_LIB_PATH):
        build.build_trace()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(device=dev)
    wl = Workload("bert_large", torch, dev, 25, n_out=1, driver="events", layers=args.layers,
                  lib_path=_lib.TRACE_LIB_PATH)
    out = {}
    for drv in ("events", "hooks"):
        wl.driver = drv
        with torch.cuda.stream(stream):
            ms, _, _ = time_steps(torch, stream, lambda: wl.step(stream), 10, 3)
            torch.cuda.synchronize()
            _, _, seq0 = read_launch_trace()
            wl.step(stream)
            torch.cuda.synchronize()
        buf, grid, seq1 = read_launch_trace()
        n = seq1 - seq0
        if n > _lib.TRACE_LAUNCHES:
            raise RuntimeError("more launches in one iteration than trace slots")
        spans = []
        for i in range(seq0, seq1):
            slot = i % _lib.TRACE_LAUNCHES
            t = buf[slot, :min(grid[slot], _lib.TRACE_CTAS)].astype(np.int64)
            busy = t[:, 3] > 0                        # CTAs that consumed staged work (0: none)
            first = t[t[:, 2] > 0, 2]
            spans.append({"entry0": int(t[:, 0].min()), "release0": int(t[:, 1].min()),
                          "first0": int(first.min()), "end_p90": int(np.percentile(t[busy, 3], 90)),
                          "end": int(t[busy, 3].max()), "ctas": int(t.shape[0])})
        pairs = list(zip(spans[:-1], spans[1:]))
        med = lambda xs: round(float(np.median(xs)) / 1e3, 2)
        stamps = np.unique(buf[buf > 0])
        res = int(np.diff(stamps).min()) if stamps.size > 1 else None
        out[drv] = {"launches": n, "ms_per_step_untraced_timing": round(ms / 10, 4),
                    "median_us": {"A_last_tenth_of_ctas": med([a["end"] - a["end_p90"] for a, _ in pairs]),
                                  "B_release_after_A_end": med([b["release0"] - a["end"] for a, b in pairs]),
                                  "B_first_data_after_release": med([b["first0"] - b["release0"] for _, b in pairs]),
                                  "gap_A_last_to_B_first_stage": med([b["first0"] - a["end"] for a, b in pairs]),
                                  "launch_span": med([s["end"] - s["first0"] for s in spans])},
                    "timer_resolution_ns": res,
                    "step_span_us": round((spans[-1]["end"] - spans[0]["entry0"]) / 1e3, 1)}
    wl.free()
    print(json.dumps({"trace": out, "workload": "bert_large" + (f"_{args.layers}layers" if args.layers else ""),
                      "kernel": "bucket_reduce_tma_kernel (trace build)"}), flush=True)
    return 0


def run_ours(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    device = torch.device("cuda", torch.cuda.current_device())
    peak, peak_kind = peaks()
    bus = None
    try:
        bus = torch.cuda.get_device_properties(device).pci_bus_id
    except Exception:
        pass
    sampler = ClockSampler(bus) if rank == 0 else None
    stream = torch.cuda.Stream(device=device)

    wl = Workload("bert_large", torch, device, 25, n_out=1, driver=args.driver, layers=args.layers)
    hook_bufs = profiling_setup(torch, device, wl.red, args, wl.W)
    if args.unused:
        apply_unused(wl)
    with torch.cuda.stream(stream):
        l0 = wl.red.launch_count()
        ms, t0, t1 = time_steps(torch, stream, lambda: wl.step(stream), args.steps, args.warmup, dist)
        launches = wl.red.launch_count() - l0
    # the launch count per step is fixed by the ready order; l0 was taken
    # before the warm-up steps
    per_step_launches = launches / (args.steps + args.warmup)
    timed_launches = int(round(per_step_launches * args.steps))
    ms_step = ms / args.steps
    gbs = wl.bytes / (ms_step * 1e-3) / 1e9
    value = gbs * world
    elems = wl.W * wl.N / (ms_step * 1e-3)

    # roofline of the dominant kernel (bucket_reduce): the timed stream holds
    # only its launches, back to back, so bytes / region time bounds the
    # per-launch achieved bandwidth from below.
    roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
            "frac": round(gbs / peak, 4),
            "traffic": traffic_for("bucket_reduce", wl.bytes / max(per_step_launches, 1)),
            "peak_kind": f"{peak_kind} (copy bandwidth, MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
            "kernel": kernel_name(wl), "launches_per_step": round(per_step_launches, 2),
            "bytes_per_launch_avg": int(wl.bytes / max(per_step_launches, 1)),
            "duration_source": "CUDA events over the timed region / launches (PDL back-to-back)",
            "frac_of_nominal_8TBps": round(gbs / NOMINAL_HBM_GBS, 4)}
    if roof["traffic"] is not None:
        roof["traffic"] = int(roof["traffic"])

    extra = {}
    if not args.no_extra:
        extra = extra_configs(torch, device, stream, args, dist, keep=wl)
    if dist is not None and not args.no_extra:
        # the same workload's bucket all-reduce split across the ranks (one
        # replica per rank), beside the per-rank emulation timed above
        extra["bert_large_sharded_allreduce"] = sharded_timing(
            torch, dist, device, rank, world, 1, max(3, min(args.steps, 20)), max(3, args.warmup))

    e2e = None
    if not args.no_e2e:
        try:
            e2e = measure_e2e(torch, wl, stream, max(1, min(args.steps, args.e2e_steps)), dist)
        except (RuntimeError, MemoryError) as exc:   # e.g. pinned host memory exhausted with many ranks
            e2e = {"value": None, "unit": "GB/s", "error": f"{type(exc).__name__}: {str(exc)[:200]}"}
            torch.cuda.synchronize()
    wl.free()
    torch.cuda.empty_cache()

    clocks = sampler.summary(t0, t1) if sampler else None
    if sampler:
        sampler.stop()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        gbs_cpu, sample, _ = oracle_sample_gbs(args.cpu_s)
        cpu = {"value": round(gbs_cpu, 3), "unit": "GB/s", "cores": cpu_threads_used(), "kind": "oracle",
               "sample": sample, "host_cpus": os.cpu_count(), "affinity": len(os.sched_getaffinity(0))}
        if extra:
            add_cpu_oracle(extra, args.cpu_config_s)

    if dist:
        dist.barrier()
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded N(0,1e-3) gradients generated on the device)",
            "config": {"workload": "bert_large" if args.layers is None else f"bert_large_{args.layers}layers",
                       "W": wl.W, "P": wl.P, "N": wl.N, "cap_mib": 25,
                       "buckets": wl.B, "mode": "copy-back (n_out=1)",
                       "driver": {"hooks": "begin_iteration + mark_ready_many (one call, every ready event in order)",
                                  "events": "begin_iteration + one mark_ready call per ready event",
                                  "all": "one reduce_all launch per step"}[args.driver]
                                 + (", stored straggler ready order" if args.layers is None and args.driver != "all"
                                    else ", reverse order" if args.driver != "all" else ""),
                       "bytes_per_step": wl.bytes,
                       "l2": (f"no flush: each step streams {wl.bytes / 1e9:.1f} GB, inputs "
                              f"{wl.W * wl.N * wl.s_in / 1e9:.1f} GB > 129 MB L2"),
                       "parallelism": f"replicas only x{world}",
                       **({"profiling": {"kernel": args.kernel, "hook": args.hook, "hook_route": args.hook_route,
                                         "unused": args.unused}}
                          if args.kernel != "auto" or args.hook != "none" or args.unused else {})},
            "pct_of_nominal_8TBps": round(100 * gbs / NOMINAL_HBM_GBS, 2), "pct_of_measured_copy_bw": round(100 * gbs / peak, 2),
            "grad_elems_per_s": round(elems * world, 1),
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": timed_launches * world,
            "clocks": clocks, "per_config": extra,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def measure_e2e(torch, wl, stream, steps, dist, n_h2d=2, n_d2h=1):
    """Same metric through the public API with host buffers.  Every step
    copies the W replicas' gradients from pinned host memory and reads the
    averaged gradients back to pinned host memory, pipelined per bucket the
    way DDP overlaps communication with the backward pass: bucket b's slices
    go up on a copy stream, its ready events are reported as soon as they
    have landed (one mark_ready_many call per bucket), and its averaged
    slice comes back on a second copy stream while later buckets are still
    in flight."""
    import ctypes
    ok = 1
    try:
        host_in = [torch.empty(f.numel(), dtype=f.dtype, pin_memory=True) for f in wl.flat]
        host_out = torch.empty(wl.out_flat.numel(), dtype=torch.float32, pin_memory=True)
    except (RuntimeError, MemoryError):
        ok = 0
    if dist:                     # every rank goes on, or none does (no rank left waiting in a collective)
        flag = torch.tensor([ok], dtype=torch.int32, device=stream.device)
        dist.all_reduce(flag, op=dist.ReduceOp.MIN)
        ok = int(flag.item())
    if not ok:
        raise RuntimeError("pinned host buffers for the end-to-end measurement could not be allocated on every rank")
    for h, f in zip(host_in, wl.flat):
        h.copy_(f)
    # several copy streams: one copy engine alone does not fill the host link
    h2d_streams = [torch.cuda.Stream(device=stream.device) for _ in range(n_h2d)]
    d2h_streams = [torch.cuda.Stream(device=stream.device) for _ in range(n_d2h)]
    out_offs, _ = gen.packed_offsets(wl.numel, 64)
    buckets = []
    for members in wl.red.get_members():
        lo_v, hi_v = min(members), max(members)
        lo, hi = wl.offs[lo_v], wl.offs[hi_v] + wl.numel[hi_v]          # replica slice (registration order)
        olo, ohi = out_offs[lo_v], out_offs[hi_v] + wl.numel[hi_v]      # copy-back slice
        vars_c = (ctypes.c_int32 * len(members))(*members)
        buckets.append((lo, hi, olo, ohi, vars_c, len(members)))
    h2d = sum((hi - lo) * f.element_size() for (lo, hi, *_) in buckets for f in wl.flat)
    d2h = sum((ohi - olo) * 4 for (_, _, olo, ohi, *_) in buckets)
    ev_in = [[torch.cuda.Event() for _ in h2d_streams] for _ in buckets]
    ev_red = [torch.cuda.Event() for _ in buckets]
    red = wl.red

    def one():
        begin = torch.cuda.Event()
        begin.record(stream)
        for hs in h2d_streams:
            hs.wait_event(begin)
        for b, (lo, hi, *_rest) in enumerate(buckets):
            for r, (h, f) in enumerate(zip(host_in, wl.flat)):
                with torch.cuda.stream(h2d_streams[r % n_h2d]):
                    f[lo:hi].copy_(h[lo:hi], non_blocking=True)
            for i, hs in enumerate(h2d_streams):
                ev_in[b][i].record(hs)
        red.begin_iteration()
        for b, (lo, hi, olo, ohi, vars_c, n) in enumerate(buckets):
            for ev in ev_in[b]:
                stream.wait_event(ev)
            red.mark_ready_many(vars_c, stream)
            ev_red[b].record(stream)
            ds = d2h_streams[b % n_d2h]
            ds.wait_event(ev_red[b])
            with torch.cuda.stream(ds):
                host_out[olo:ohi].copy_(wl.out_flat[olo:ohi], non_blocking=True)
        for ds in d2h_streams:
            done = torch.cuda.Event()
            done.record(ds)
            stream.wait_event(done)

    # per-step events: the host link is shared with the machine's other
    # work, so the step time is reported as the median with its spread
    with torch.cuda.stream(stream):
        one()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        ev[0].record(stream)
        for i in range(steps):
            one()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    if dist:
        per = [max_over_ranks(t, dist, "cuda") for t in per]
    ms_step = statistics.median(per)

    # The host link itself, measured the same minute: one whole-buffer copy
    # each way (pinned memory, best of 3).  The step cannot beat the slower
    # direction's bytes over its rate.
    def link(copy, nbytes):
        best = None
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            with torch.cuda.stream(stream):
                copy()
            e1.record(stream)
            e1.synchronize()
            t = e0.elapsed_time(e1)
            best = t if best is None else min(best, t)
        return nbytes / (best * 1e-3) / 1e9
    up = link(lambda: wl.flat[0].copy_(host_in[0], non_blocking=True), host_in[0].numel() * host_in[0].element_size())
    down = link(lambda: host_out.copy_(wl.out_flat, non_blocking=True), host_out.numel() * 4)
    bound_s = max(h2d / (up * 1e9), d2h / (down * 1e9))
    bound = wl.bytes / bound_s / 1e9
    serial = wl.bytes / (ms_step * 1e-3) / 1e9

    # Consecutive steps overlapped, as a training loop streaming batches
    # would: bucket b's next upload waits only for this step's reduction of
    # bucket b (its inputs are then free), and bucket b's next reduction for
    # this step's download of bucket b (its outputs are then free), so the
    # host link never idles between steps.  Every step still uploads all of
    # its inputs and downloads its result.
    ev_d2h = [torch.cuda.Event() for _ in buckets]

    def pipelined(start=None):
        for b, (lo, hi, *_rest) in enumerate(buckets):
            for hs in h2d_streams:
                hs.wait_event(start if start is not None else ev_red[b])
            for r, (h, f) in enumerate(zip(host_in, wl.flat)):
                with torch.cuda.stream(h2d_streams[r % n_h2d]):
                    f[lo:hi].copy_(h[lo:hi], non_blocking=True)
            for i, hs in enumerate(h2d_streams):
                ev_in[b][i].record(hs)
        red.begin_iteration()
        for b, (lo, hi, olo, ohi, vars_c, n) in enumerate(buckets):
            for ev in ev_in[b]:
                stream.wait_event(ev)
            stream.wait_event(ev_d2h[b])
            red.mark_ready_many(vars_c, stream)
            ev_red[b].record(stream)
            ds = d2h_streams[b % n_d2h]
            ds.wait_event(ev_red[b])
            with torch.cuda.stream(ds):
                host_out[olo:ohi].copy_(wl.out_flat[olo:ohi], non_blocking=True)
            ev_d2h[b].record(ds)

    with torch.cuda.stream(stream):
        for b in range(len(buckets)):                # recorded once before the first wait on them
            ev_d2h[b].record(d2h_streams[b % n_d2h])
        pipelined()                                  # warm-up step
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        # each step's completion (its last download) is marked on a stream of
        # its own that only waits and records, so the marks order nothing
        marker = torch.cuda.Stream(device=stream.device)
        t0 = torch.cuda.Event(enable_timing=True)
        done = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        t0.record(stream)
        for i in range(steps):
            pipelined(t0 if i == 0 else None)
            for ds in d2h_streams:
                ev = torch.cuda.Event()
                ev.record(ds)
                marker.wait_event(ev)
            done[i].record(marker)
        torch.cuda.synchronize()
    # steady-state period: median interval between consecutive completions
    # (a step delayed by other traffic on the host link does not skew it)
    intervals = [done[i - 1].elapsed_time(done[i]) for i in range(1, steps)] or [t0.elapsed_time(done[0])]
    ms_pipe = statistics.median(intervals)
    ms_mean = t0.elapsed_time(done[-1]) / steps
    if dist:
        ms_pipe = max_over_ranks(ms_pipe, dist, "cuda")
        ms_mean = max_over_ranks(ms_mean, dist, "cuda")
    pipe = wl.bytes / (ms_pipe * 1e-3) / 1e9
    return {"value": round(serial, 2), "unit": "GB/s", "steps": steps,
            "ms_per_step": round(ms_step, 3), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "step_ms": {"median": round(ms_step, 3), "min": round(min(per), 3), "mean": round(sum(per) / steps, 3),
                        "max": round(max(per), 3)},
            "h2d_gbs": round(h2d / (ms_step * 1e-3) / 1e9, 1),
            "host_link": {"h2d_gbs": round(up, 1), "d2h_gbs": round(down, 1), "bound_gbs": round(bound, 1),
                          "frac_of_bound": round(serial / bound, 3),
                          "note": "one pinned whole-buffer copy each way, best of 3, same run; bound = step "
                                  "bytes / max(h2d bytes / h2d rate, d2h bytes / d2h rate)"},
            "pipelined": {"value": round(pipe, 2), "ms_per_step": round(ms_pipe, 3),
                          "step_ms": {"median_interval": round(ms_pipe, 3), "min_interval": round(min(intervals), 3),
                                      "max_interval": round(max(intervals), 3),
                                      "mean_incl_first_and_tail": round(ms_mean, 3)},
                          "note": "consecutive steps overlapped bucket by bucket (bucket b's next upload waits for "
                                  "this step's reduction of b, its next reduction for this step's download of b); "
                                  "median interval between the completions of consecutive steps"},
            "note": ("algorithmic bytes of the step / median time of a step that copies the replicas' gradients "
                     "host->device per bucket, reduces each bucket as it lands (mark_ready_many per bucket) "
                     f"and copies its averaged gradients back; pinned host buffers, {n_h2d} host->device and "
                     f"{n_d2h} device->host copy streams")}


def extra_configs(torch, device, stream, args, dist, keep):
    """The other configurations, each timed the same way (GB/s of its own
    algorithmic bytes)."""
    out = {}
    steps, warm = max(5, min(args.steps, 50)), max(3, args.warmup)

    def timed(wl, key, note):
        with torch.cuda.stream(stream):
            ms, _, _ = time_steps(torch, stream, lambda: wl.step(stream), steps, warm, dist)
        t = ms / steps
        gbs = wl.bytes / (t * 1e-3) / 1e9
        peak, _ = peaks()
        out[key] = {"gbs": round(gbs, 1), "ms_per_step": round(t, 4),
                    "pct_of_nominal_8TBps": round(100 * gbs / NOMINAL_HBM_GBS, 2), "pct_of_measured_copy_bw": round(100 * gbs / peak, 2),
                    "bytes_per_step": wl.bytes, "buckets": wl.B, "W": wl.W, "kernel": kernel_name(wl),
                    "grad_elems_per_s": round(wl.W * wl.N / (t * 1e-3), 1), "note": note}

    # Linear(10,10), W=2: one bucket of 110 elements, launch latency rather
    # than bandwidth (reported in microseconds per iteration)
    wl = Workload("linear", torch, device, 25, n_out=1, driver="events")
    timed(wl, "linear_w2", "Linear(10,10), W=2, one mark_ready call per event; latency-bound (one launch)")
    out["linear_w2"]["us_per_step"] = round(out["linear_w2"]["ms_per_step"] * 1e3, 2)
    # the same iteration's GPU latency without the host calls in between: 100
    # iterations (begin_iteration + two mark_ready calls each) captured in one
    # CUDA graph, replayed
    with torch.cuda.stream(stream):
        wl.step(stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for _ in range(100):
                wl.step(stream)
    reps = max(3, steps // 20)
    with torch.cuda.stream(stream):
        ms, _, _ = time_steps(torch, stream, g.replay, reps, warm, dist)
    out["linear_w2_graph"] = {"us_per_step": round(ms * 1e3 / (reps * 100), 2), "W": wl.W, "buckets": wl.B,
                              "kernel": kernel_name(wl),
                              "note": "Linear(10,10), W=2: 100 iterations of one mark_ready call per event captured "
                                      "in one CUDA graph and replayed (GPU latency of a one-launch iteration)"}
    del g
    wl.free()
    # BERT-large, one launch over all buckets (kernel alone)
    keep.driver = "all"
    timed(keep, "bert_large_reduce_all", "one reduce_all launch per step")
    # BERT-large, one Python mark_ready call per ready event: each launch waits
    # for the previous one (foreign work could sit between calls)
    keep.driver = "events"
    timed(keep, "bert_large_event_calls", "one mark_ready call per event (launches wait for their predecessor)")
    # the same with calls chained (DDP_OPT_CHAINED: the caller guarantees that
    # nothing else runs on the stream during the iteration)
    from reduction_reducer_gb300 import _lib
    keep.red.set_option(_lib.OPT_CHAINED, 1)
    timed(keep, "bert_large_event_calls_chained",
          "one mark_ready call per event, DDP_OPT_CHAINED = 1 (each launch follows its predecessor at once)")
    keep.red.set_option(_lib.OPT_CHAINED, 0)
    keep.driver = "hooks"
    # BERT-large after a rebuild from the recorded (straggler) ready order,
    # first bucket capped at 1 MiB
    import time as _time
    t0 = _time.perf_counter()
    keep.red.rebuild_buckets(None, 1 << 20, 25 << 20)
    rebuild_ms = (_time.perf_counter() - t0) * 1e3
    keep._order_c = (__import__("ctypes").c_int32 * len(keep.order))(*keep.order)
    timed(keep, "bert_large_rebuilt", "after ddp_rebuild_buckets from the recorded order (first cap 1 MiB)")
    out["bert_large_rebuilt"]["rebuild_host_ms"] = round(rebuild_ms, 3)
    out["bert_large_rebuilt"]["buckets"] = keep.red.B
    keep.red.rebuild_buckets(list(range(keep.P - 1, -1, -1)), 25 << 20, 25 << 20)   # back to the construction layout
    # BERT-large with unused parameters: pooler unused everywhere, the FFN of
    # every fourth layer unused on replica 1
    unused_config(keep, timed, out)
    # BERT-large through the built-in mean hook: gather + hook + copy-back
    hook_config(torch, device, keep, timed, out)
    # BERT-large as-view: replicas laid out as buckets, no copy-back
    wl = Workload("bert_large", torch, device, 25, n_out=0, driver="hooks", layout="buckets")
    timed(wl, "bert_large_as_view", "gradient_as_bucket_view: W*N*4 + N*4 bytes")
    wl.free()
    torch.cuda.empty_cache()
    wl = Workload("resnet50", torch, device, 25, n_out=1, driver="hooks")
    timed(wl, "resnet50_w8", "ResNet-50 W=8 fp32, reverse order")
    wl.free()
    torch.cuda.empty_cache()
    for cap in (0, 1, 5, 25, 100):
        wl = Workload("gpt2_medium", torch, device, cap, n_out=1, driver="hooks")
        timed(wl, f"gpt2_medium_w8_bf16_cap{cap}", f"GPT-2-medium bf16 W=8, cap {cap} MiB")
        if cap == 0:
            # the same per-gradient buckets with one launch per releasing event
            wl.red.set_option(_lib.OPT_COALESCE_ELEMS, 0)
            timed(wl, "gpt2_medium_w8_bf16_cap0_launch_per_event",
                  "GPT-2-medium bf16 W=8, cap 0, DDP_OPT_COALESCE_ELEMS = 0: one launch per releasing event")
        if cap in (0, 25):
            # one mark_ready call per event, as a backward pass reports its hooks:
            # per-gradient buckets against 25 MiB ones (the pages' bucketing experiment)
            wl.driver = "events"
            timed(wl, f"gpt2_medium_w8_bf16_cap{cap}_event_calls",
                  f"GPT-2-medium bf16 W=8, cap {cap} MiB, one mark_ready call per event (launches wait for their "
                  "predecessor)")
            wl.red.set_option(_lib.OPT_CHAINED, 1)
            timed(wl, f"gpt2_medium_w8_bf16_cap{cap}_event_calls_chained",
                  f"GPT-2-medium bf16 W=8, cap {cap} MiB, one mark_ready call per event, DDP_OPT_CHAINED = 1")
        wl.free()
        torch.cuda.empty_cache()
    out["nosync_resnet50_w16_k8"] = nosync_config(torch, device, stream, steps, warm, dist)
    # the replica count on the BERT-large shapes (reverse order; the headline
    # iteration is W = 4 with the stored straggler order)
    sweep = replica_sweep(torch, device, stream, (1, 2, 4, 8, 16, 32), min(steps, 30), warm, dist)
    for W, r in sweep.items():
        out[f"bert_large_shapes_w{W}"] = {
            "gbs": r["gbs"], "ms_per_step": r["ms"], "W": W,
            "pct_of_w8": round(100 * r["gbs"] / sweep[8]["gbs"], 1),
            "note": f"BERT-large shapes, W={W} fp32 ({W} reads : 2 writes per element), reverse order, one "
                    "mark_ready_many call"}
    # whole iterations captured in a CUDA graph (launch-bound layouts)
    for name, cap in (("gpt2_medium", 0), ("bert_large", 25)):
        wl = Workload(name, torch, device, cap, n_out=1, driver="hooks")
        graph_config(torch, wl, stream, steps, warm, dist, out, f"{name}_cap{cap}_graph")
        wl.free()
        torch.cuda.empty_cache()
    return out


def graph_config(torch, wl, stream, steps, warm, dist, out, key):
    """One iteration (begin_iteration + mark_ready_many) captured into a CUDA
    graph after a warm-up iteration, replayed as the step."""
    with torch.cuda.stream(stream):
        wl.step(stream)                          # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            wl.step(stream)
    launches = wl.red.launch_count()
    with torch.cuda.stream(stream):
        ms, _, _ = time_steps(torch, stream, g.replay, steps, warm, dist)
    t = ms / steps
    out[key] = {"gbs": round(wl.bytes / (t * 1e-3) / 1e9, 1), "ms_per_step": round(t, 4), "bytes_per_step": wl.bytes,
                "buckets": wl.B, "W": wl.W, "kernel": kernel_name(wl),
                "note": "iteration captured in a CUDA graph (PDL-chained launches), replayed per step"}
    del g


def hook_config(torch, device, keep, timed, out):
    """The communication-hook path on BERT-large W=4.  A registered built-in
    hook runs inside the fused bucket pass by default (mean, and the bf16
    compression hook); the gather, hook call and copy-back route is timed
    beside it, reported against the fused pass's algorithmic bytes (what the
    iteration must move) and against the bytes its three passes move."""
    from reduction_reducer_gb300 import _lib
    for hook in ("mean", "bf16_compress"):
        wl = Workload("bert_large", torch, device, 25, n_out=1, driver="hooks")
        rb = [torch.empty(wl.red.arena_numel(), dtype=torch.float32, device=device) for _ in range(wl.W)]
        wl.red.register_comm_hook(hook, rb)
        timed(wl, f"bert_large_hook_{hook}", f"register_comm_hook('{hook}'): the hook's arithmetic inside the fused "
              "bucket pass (nothing gathered), W*N*4 + 2*N*4 bytes")
        wl.free()
        del rb
        torch.cuda.empty_cache()
    wl = Workload("bert_large", torch, device, 25, n_out=1, driver="hooks")
    rb = [torch.empty(wl.red.arena_numel(), dtype=torch.float32, device=device) for _ in range(wl.W)]
    wl.red.register_comm_hook("mean", rb)
    wl.red.set_option(_lib.OPT_HOOK_FUSED, 0)
    timed(wl, "bert_large_hook_mean_gathered", "register_comm_hook('mean') with DDP_OPT_HOOK_FUSED = 0: gather + "
          "hook call + copy-back per bucket; gbs uses the fused pass's algorithmic bytes")
    moved = 2 * wl.W * wl.N * 4 + wl.W * wl.N * 4 + wl.N * 4 + 2 * wl.N * 4
    out["bert_large_hook_mean_gathered"]["bytes_moved_per_step"] = moved
    out["bert_large_hook_mean_gathered"]["moved_gbs"] = round(
        moved / (out["bert_large_hook_mean_gathered"]["ms_per_step"] * 1e-3) / 1e9, 1)
    wl.free()
    del rb
    torch.cuda.empty_cache()
    # the hook-call route on gradients that are views of the bucket layout:
    # the hook reads them in place, nothing is gathered and nothing copied back
    wl = Workload("bert_large", torch, device, 25, n_out=0, driver="hooks", layout="buckets")
    wl.red.register_comm_hook("mean", None)
    wl.red.set_option(_lib.OPT_HOOK_FUSED, 0)
    timed(wl, "bert_large_hook_mean_as_view", "register_comm_hook('mean', replica_buffers=None) on bucket views, "
          "hook-call route: the hook's mean per bucket, W*N*4 + N*4 bytes")
    wl.free()
    torch.cuda.empty_cache()


def apply_unused(wl):
    """Make ``wl.step`` an iteration with unused parameters (find_unused): on
    BERT-large the pooler is unused on every replica and the FFN of every
    fourth layer on replica 1; ``wl.bytes`` becomes the replica reads that
    happen + bucket writes + copy-backs actually written.  Returns a function
    that restores the plain iteration."""
    import ctypes
    from reduction_reducer_gb300 import _lib
    names = [n for n, _ in (shapes.bert_large() if wl.layers is None else shapes.bert_large(layers=wl.layers))]
    used = [[True] * wl.P for _ in range(wl.W)]
    for v, n in enumerate(names):
        if n.startswith("pooler"):
            for r in range(wl.W):
                used[r][v] = False
        if (".intermediate." in n or ".output.dense" in n) and int(n.split(".")[2]) % 4 == 0:
            used[1][v] = False
    gused = [any(used[r][v] for r in range(wl.W)) for v in range(wl.P)]
    wl.red.set_option(_lib.OPT_FIND_UNUSED, 1)
    order = [v for v in wl.order if gused[v]]
    order_c = (ctypes.c_int32 * len(order))(*order)
    saved_step, saved_bytes = wl.step, wl.bytes
    used_c = wl.red.bits(used)                     # marshalled once

    def step(stream):
        wl.red.set_local_used(used_c)
        wl.red.begin_iteration()
        wl.red.mark_ready_many(order_c, stream)
    wl.step = step
    wl.bytes = (sum(wl.numel[v] * wl.s_in for r in range(wl.W) for v in range(wl.P) if used[r][v])
                + wl.N * 4 + sum(wl.numel[v] * 4 for v in range(wl.P) if gused[v]))

    def restore():
        wl.step, wl.bytes = saved_step, saved_bytes
        wl.red.set_option(_lib.OPT_FIND_UNUSED, 0)
    return restore


def unused_config(wl, timed, out):
    """find_unused_parameters on BERT-large (see apply_unused), timed as a
    configuration line."""
    restore = apply_unused(wl)
    timed(wl, "bert_large_find_unused", "find_unused: pooler unused on every replica, every 4th FFN unused "
          "on replica 1; bytes count only the reads and copy-backs that happen")
    restore()


KERNEL_FLAG = {"auto": 2, "ldg": 0, "tma": 1}


def profiling_setup(torch, device, red, args, W):
    """Profiling cases only: force a kernel (--kernel) and route the buckets
    through a built-in hook (--hook).  Returns the replica buffers it
    allocated (kept alive by the caller)."""
    from reduction_reducer_gb300 import _lib
    if getattr(args, "kernel", "auto") != "auto":
        red.set_option(_lib.OPT_KERNEL, KERNEL_FLAG[args.kernel])
    if getattr(args, "hook", "none") == "none":
        return None
    tdt = torch.float32 if red.dtype == "f32" else torch.bfloat16
    bufs = [torch.empty(max(red.arena_numel(), 1), dtype=tdt, device=device) for _ in range(W)]
    red.register_comm_hook(args.hook, bufs)
    red.set_option(_lib.OPT_HOOK_FUSED, 1 if args.hook_route == "fused" else 0)
    return bufs


def nosync_config(torch, device, stream, steps, warm, dist, K=8, kernel="auto"):
    from reduction_reducer_gb300 import Reducer, _lib
    numel = shapes.numels(shapes.resnet50())
    W = 16
    N = sum(numel)
    offs, total = gen.packed_offsets(numel, 64)
    fresh = [[gen.draw_flat_torch(total, r, k, "f32", device) for r in range(W)] for k in range(K)]
    fresh_v = [[[f[o:o + n] for o, n in zip(offs, numel)] for f in fk] for fk in fresh]
    acc_flat = [torch.empty(total, device=device) for _ in range(W)]
    acc = [[f[o:o + n] for o, n in zip(offs, numel)] for f in acc_flat]
    red = Reducer(numel, "f32", 25 * MIB)
    if kernel != "auto":
        red.set_option(_lib.OPT_KERNEL, KERNEL_FLAG[kernel])
    arena = torch.empty(red.arena_numel(), device=device)
    out_flat = torch.empty(total, device=device)
    red.bind(acc, arena, [out_flat[o:o + n] for o, n in zip(offs, numel)])
    import ctypes
    order = gen.reverse_order(len(numel))
    order_c = (ctypes.c_int32 * len(order))(*order)
    acc_p = red.pointers(acc)                       # marshalled once, reused every call
    fresh_p = [red.pointers(fv) for fv in fresh_v]

    def cycle():
        for k in range(K):
            red.accumulate_nosync(acc_p, fresh_p[k], first_step=(k == 0), stream=stream)
        red.begin_iteration()
        red.mark_ready_many(order_c, stream)

    def acc_only():
        red.accumulate_nosync(acc_p, fresh_p[1 % K], first_step=False, stream=stream)

    # the last micro-step fused into the reduction: K - 1 accumulate launches,
    # then one pass over (acc_r, g_r) pairs; the last step's gradient buffers
    # are bound once, as a training loop would
    def cycle_fused():
        for k in range(K - 1):
            red.accumulate_nosync(acc_p, fresh_p[k], first_step=(k == 0), stream=stream)
        red.begin_iteration()
        red.mark_ready_many(order_c, stream)

    def last_only():
        red.begin_iteration()
        red.mark_ready_many(order_c, stream)

    with torch.cuda.stream(stream):
        ms, _, _ = time_steps(torch, stream, cycle, steps, warm, dist)
        ms_acc, _, _ = time_steps(torch, stream, acc_only, steps, warm, dist)
        red.bind_last_step(fresh_p[K - 1])
        ms_f, _, _ = time_steps(torch, stream, cycle_fused, steps, warm, dist)
        ms_last, _, _ = time_steps(torch, stream, last_only, steps, warm, dist)
    t, t_f = ms / steps, ms_f / steps
    cycle_bytes = 2 * W * N * 4 + (K - 1) * 3 * W * N * 4 + view_bytes(W, N, 4)
    last_bytes = 2 * W * N * 4 + 2 * N * 4       # read acc_r and g_r, write bucket and copy-back
    fused_bytes = 2 * W * N * 4 + (K - 2) * 3 * W * N * 4 + last_bytes
    res = {"gbs": round(cycle_bytes / (t * 1e-3) / 1e9, 1), "ms_per_cycle": round(t, 4),
           "bytes_per_cycle": cycle_bytes, "W": W, "K": K,
           "accumulate_gbs": round(3 * W * N * 4 / (ms_acc / steps * 1e-3) / 1e9, 1),
           "accumulate_ms": round(ms_acc / steps, 4),
           "fused_last_step": {"gbs": round(fused_bytes / (t_f * 1e-3) / 1e9, 1), "ms_per_cycle": round(t_f, 4),
                               "bytes_per_cycle": fused_bytes,
                               "reduce_gbs": round(last_bytes / (ms_last / steps * 1e-3) / 1e9, 1),
                               "reduce_ms": round(ms_last / steps, 4), "reduce_bytes": last_bytes,
                               "note": "K-1 accumulate micro-steps + the K-th fused into the reduction"},
           "kernel": ("bulk copy" if red.get_option(10) == 1 else "register streaming"),
           "note": "K accumulate micro-steps (first one a copy) + one reduce (mark_ready_many)"}
    red.destroy()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--layers", type=int, default=None, help="fewer layers of BERT or GPT-2 (profiling cases)")
    ap.add_argument("--workload", default="bert_large", choices=["bert_large", "nosync_resnet50", "gpt2_medium"],
                    help="nosync_resnet50 / gpt2_medium: that workload alone (profiling cases)")
    ap.add_argument("--cap-mib", type=int, default=0, help="bucket cap of --workload gpt2_medium")
    ap.add_argument("--nosync-k", type=int, default=8, help="micro-steps of --workload nosync_resnet50")
    ap.add_argument("--driver", default="hooks", choices=["hooks", "events", "all"])
    ap.add_argument("--kernel", default="auto", choices=["auto", "ldg", "tma"],
                    help="profiling cases: force the bucket-reduce/accumulate kernel")
    ap.add_argument("--unused", action="store_true",
                    help="profiling cases: the main workload with unused parameters (find_unused)")
    ap.add_argument("--hook", default="none", choices=["none", "mean", "bf16_compress"],
                    help="profiling cases: reduce the main workload through a built-in hook")
    ap.add_argument("--hook-route", default="fused", choices=["fused", "gathered"],
                    help="profiling cases: --hook inside the fused pass or through gather + hook call + copy-back")
    ap.add_argument("--sharded", action="store_true",
                    help="the bucket all-reduce across ranks (NCCL; reduce-scatter as all-to-alls of raw chunks "
                         "+ owner mean, then all-gather)")
    ap.add_argument("--replicas-per-rank", type=int, default=1,
                    help="--sharded: replicas each rank holds (the same on every rank)")
    ap.add_argument("--trace", action="store_true",
                    help="launch boundaries of one BERT-large iteration from the trace build's per-CTA timestamps")
    ap.add_argument("--mix-rates", action="store_true",
                    help="roofline context: torch streaming rates by read:write mix and the fused pass for W = 1 .. 32")
    ap.add_argument("--cpu-s", type=float, default=10.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--cpu-config-s", type=float, default=2.0,
                    help="seconds of oracle work per configuration (per_config cpu_oracle)")
    ap.add_argument("--ref-step-s", type=float, default=2.0, help="oracle seconds per reference step")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.sharded:
        return run_sharded(args)
    if args.mix_rates:
        return run_mix_rates(args)
    if args.trace:
        return run_trace(args)
    if args.workload == "nosync_resnet50":
        return run_nosync_only(args)
    if args.workload == "gpt2_medium":
        return run_gpt2_only(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
