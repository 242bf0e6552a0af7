"""Host-side checks of the C-ABI library (no GPU, no compute call).

* the library loads and exports every function include/ddp_reducer.h declares;
* the C++ bucket builder reproduces the oracle's locators bit for bit on
  every workload and on brute-force tiny lists;
* the C++ readiness state machine (dry-run: state only, nothing launched)
  reproduces the oracle's launches and parked sets on every permutation of
  tiny lists and on the stored BERT-large straggler order;
* error codes of the failure cases the pages name.
"""

import itertools
import os
import re

import numpy as np
import pytest

from oracle.buckets import assign_buckets
from oracle.readiness import ReadinessOracle
from workloads import gen, shapes

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def lib():
    from reduction_reducer_gb300 import _lib
    if not os.path.exists(_lib.LIB_PATH):
        from reduction_reducer_gb300 import build
        build.build()
    return _lib.load()


def header_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"^\s*(?:const\s+)?[\w\*\s]+?\b(ddp_\w+)\s*\(", text, flags=re.M))
    return names


def test_exports_every_declared_symbol(lib):
    from reduction_reducer_gb300 import _lib
    declared = header_functions()
    assert {"ddp_build_buckets", "ddp_mark_ready", "ddp_reduce_bucket", "ddp_reduce_all",
            "ddp_accumulate_nosync"} <= declared
    for name in declared:
        assert hasattr(lib, name), name
    assert declared <= set(_lib.SIGNATURES), declared - set(_lib.SIGNATURES)


def _make(numel, dtype="f32", cap=25 << 20):
    from reduction_reducer_gb300 import Reducer
    return Reducer(numel, dtype, cap)


WORKLOAD_CASES = [
    ("linear", shapes.linear_10x10, "f32", 25),
    ("resnet50", shapes.resnet50, "f32", 25),
    ("bert_large", shapes.bert_large, "f32", 25),
] + [(f"gpt2_medium_cap{c}", shapes.gpt2_medium, "bf16", c) for c in (0, 1, 5, 25, 100)]


@pytest.mark.parametrize("name,fn,dtype,cap_mib", WORKLOAD_CASES, ids=[c[0] for c in WORKLOAD_CASES])
def test_locators_match_oracle_on_workloads(lib, name, fn, dtype, cap_mib):
    numel = shapes.numels(fn())
    red = _make(numel, dtype, cap_mib << 20)
    members, locs = assign_buckets(numel, 4 if dtype == "f32" else 2, cap_mib << 20)
    assert red.B == len(members)
    got = red.get_locators()
    assert got == [(l.bucket, l.intra, l.offset, l.length) for l in locs]
    B, offs = red.get_bucket_info()
    lens = [sum(numel[v] for v in m) for m in members]
    assert offs == [sum(lens[:b]) for b in range(B + 1)]


def test_locators_match_oracle_bruteforce(lib):
    for n in range(0, 5):
        for numel in itertools.product([0, 1, 3, 4], repeat=n):
            for cap in (0, 1, 4, 12, 16, 40):
                red = _make(list(numel), "f32", cap)
                _, locs = assign_buckets(numel, 4, cap)
                assert red.get_locators() == [(l.bucket, l.intra, l.offset, l.length) for l in locs], (numel, cap)
                red.destroy()


def _run_dry(red, order):
    red.set_dry_run(True)
    red.begin_iteration()
    trace = []
    for v in order:
        launched = red.mark_ready(v)
        trace.append((launched, red.get_progress()[1]))
    return trace


def _oracle_trace(members, order):
    sm = ReadinessOracle(members)
    sm.begin_iteration()
    out = []
    for v in order:
        launched = sm.mark_ready(v)
        out.append((launched, sm.parked()))
    return out


@pytest.mark.parametrize("numel,cap", [([1] * 6, 2), ([3, 0, 2, 5, 1, 4], 3), ([1] * 6, 0), ([2, 2, 2], 100)])
def test_state_machine_matches_oracle_all_permutations(lib, numel, cap):
    members, _ = assign_buckets(numel, 1, cap)
    red = _make(numel, "f32", cap * 4)      # f32: 4 bytes per element, same layout
    assert red.get_members() == members
    for order in itertools.permutations(range(len(numel))):
        assert _run_dry(red, order) == _oracle_trace(members, order), order


def test_state_machine_bert_straggler_order(lib):
    numel = shapes.numels(shapes.bert_large())
    with open(os.path.join(GOLDEN, "bert_large_ready_order.txt")) as f:
        order = [int(l) for l in f if l.strip() and not l.startswith("#")]
    red = _make(numel, "f32", 25 << 20)
    members, _ = assign_buckets(numel, 4, 25 << 20)
    got = _run_dry(red, order)
    want = _oracle_trace(members, order)
    assert got == want
    assert any(parked for _, parked in got)           # the fixture really parks


def test_error_codes(lib):
    from reduction_reducer_gb300 import (AlreadyReady, InvalidArg, NotBound, OutOfOrder,
                                         PriorReductionUnfinished, Reducer)
    with pytest.raises(InvalidArg):
        Reducer([3, -1], "f32", 16)
    with pytest.raises(InvalidArg):
        Reducer([3], "f32", -1)
    red = _make([1, 1, 1], "f32", 4)                  # one bucket per tensor: v -> bucket 2 - v
    with pytest.raises(NotBound):
        red.mark_ready(0)                             # no bind and not dry
    red.set_dry_run(True)
    with pytest.raises(InvalidArg):
        red.mark_ready(3)
    red.begin_iteration()
    assert red.mark_ready(0) == []                    # bucket 2 parks
    with pytest.raises(AlreadyReady):
        red.mark_ready(0)
    with pytest.raises(OutOfOrder):
        red.reduce_bucket(2)
    red.mark_ready(2)                                 # bucket 0 goes
    # variable 1 never reports: the next iteration must refuse to start
    with pytest.raises(PriorReductionUnfinished) as ei:
        red.begin_iteration()
    assert "prior iteration" in str(ei.value)
    red.abort_iteration()
    red.begin_iteration()
    red.reduce_bucket(0)
    assert red.get_progress() == (1, [])
    red.reduce_all()
    assert red.get_progress() == (3, [])
    red.begin_iteration()                             # previous one finished
    with pytest.raises(InvalidArg):
        red.set_option(3, 300)


def test_empty_model(lib):
    red = _make([], "f32", 25 << 20)
    assert red.B == 0 and red.get_locators() == [] and red.get_bucket_info() == (0, [0])
    red.set_dry_run(True)
    red.begin_iteration()
    red.reduce_all()
    red.begin_iteration()


def test_explicit_launch_matches_oracle(lib):
    numel = [1, 1, 1, 1]
    members, _ = assign_buckets(numel, 4, 4)
    red = _make(numel, "f32", 4)
    red.set_dry_run(True)
    sm = ReadinessOracle(members)
    red.begin_iteration(); sm.begin_iteration()
    assert red.mark_ready(1) == sm.mark_ready(1)      # bucket 2 parks
    red.reduce_bucket(0); sm.launch_next(0)
    red.reduce_bucket(1); sm.launch_next(1)           # releases parked 2 too
    assert red.get_progress() == (sm.next, sm.parked())
    red.reduce_all(); sm.launch_rest()
    assert red.get_progress() == (sm.next, sm.parked())


def test_mark_ready_many_matches_oracle(lib):
    """The batch call is the same state machine: same launches and parked
    sets as one mark_ready per event, on every permutation of a tiny list."""
    numel = [3, 0, 2, 5, 1, 4]
    members, _ = assign_buckets(numel, 1, 3)
    red = _make(numel, "f32", 12)
    red.set_dry_run(True)
    for order in itertools.permutations(range(len(numel))):
        red.begin_iteration()
        k = 3
        assert red.mark_ready_many(list(order[:k])) == k
        sm = ReadinessOracle(members)
        sm.begin_iteration()
        for v in order[:k]:
            sm.mark_ready(v)
        assert red.get_progress() == (sm.next, sm.parked()), order
        assert red.mark_ready_many(list(order[k:])) == len(order) - k
        assert red.get_progress() == (len(members), [])


def test_mark_ready_many_error_stops_at_event(lib):
    from reduction_reducer_gb300 import AlreadyReady
    red = _make([1, 1, 1, 1], "f32", 4)
    red.set_dry_run(True)
    red.begin_iteration()
    with pytest.raises(AlreadyReady):
        red.mark_ready_many([3, 2, 3, 1])
    # events before the failing one stay applied: buckets 0 and 1 are out
    assert red.get_progress() == (2, [])


# ---------------------------------------------------------------- rebuild

def test_trace_and_rebuild_match_oracle(lib):
    from oracle.rebuild import rebuild_buckets
    numel = [3, 0, 2, 5, 1, 4, 7]
    for order in itertools.permutations(range(len(numel))):
        if hash(order) % 7:                      # a seeded subset of the 5040 orders
            continue
        red = _make(numel, "f32", 12)
        red.set_dry_run(True)
        red.begin_iteration()
        red.mark_ready_many(list(order))
        assert red.get_ready_trace() == list(order)
        for fc, cap in ((4, 12), (0, 8), (40, 4)):
            red.rebuild_buckets(None, fc, cap)
            members, locs = rebuild_buckets(numel, 4, list(order), fc, cap)
            assert red.get_locators() == [(l.bucket, l.intra, l.offset, l.length) for l in locs]
            assert red.B == len(members)
            # the state machine now runs on the new layout
            red.begin_iteration()
            sm = ReadinessOracle(members)
            sm.begin_iteration()
            for v in order:
                assert red.mark_ready(v) == sm.mark_ready(v)
            assert red.get_ready_trace() == list(order)
        red.destroy()


def test_rebuild_bert_trace_and_page_layouts(lib):
    from oracle.rebuild import rebuild_buckets
    numel = shapes.numels(shapes.bert_large())
    with open(os.path.join(GOLDEN, "bert_large_ready_order.txt")) as f:
        order = [int(l) for l in f if l.strip() and not l.startswith("#")]
    red = _make(numel, "f32", 25 << 20)
    red.set_dry_run(True)
    red.begin_iteration()
    red.mark_ready_many(order)
    red.rebuild_buckets(None, 1 << 20, 25 << 20)
    _, locs = rebuild_buckets(numel, 4, order, 1 << 20, 25 << 20)
    assert red.get_locators() == [(l.bucket, l.intra, l.offset, l.length) for l in locs]
    # course page: 12 x 4 MiB, one 48 MiB bucket first, then 1 / 3 / 12 after the rebuild
    n12 = [1 << 20] * 12
    red = _make(n12, "f32", (1 << 63) - 1)
    assert red.get_bucket_info() == (1, [0, 12 << 20])
    red.set_dry_run(True)
    red.begin_iteration()
    red.mark_ready_many(list(range(11, -1, -1)))
    for cap_mib, nb in ((64, 1), (16, 3), (4, 12)):
        red.rebuild_buckets(None, cap_mib << 20, cap_mib << 20)
        assert red.B == nb


def test_rebuild_errors(lib):
    from reduction_reducer_gb300 import InvalidArg
    red = _make([1, 1, 1, 1], "f32", 4)
    red.set_dry_run(True)
    with pytest.raises(InvalidArg):
        red.rebuild_buckets(None, 4, 4)           # no finished iteration yet
    red.begin_iteration()
    red.mark_ready(3)
    with pytest.raises(InvalidArg):
        red.rebuild_buckets([0, 1, 2, 3], 4, 4)   # inside an iteration
    red.abort_iteration()
    with pytest.raises(InvalidArg):
        red.rebuild_buckets([0, 1, 1, 3], 4, 4)   # not a permutation
    red.reduce_all()                              # explicit launch: no complete trace
    assert red.get_ready_trace() == []
    with pytest.raises(InvalidArg):
        red.rebuild_buckets(None, 4, 4)
    red.rebuild_buckets([0, 1, 2, 3], 8, 8)
    assert red.get_members() == [[0, 1], [2, 3]]


# ---------------------------------------------------------------- unused parameters

def _dry_bound(numel, W, cap, find_unused=True):
    from reduction_reducer_gb300 import _lib as L
    red = _make(numel, "f32", cap)
    red.set_dry_run(True)
    if find_unused:
        red.set_option(L.OPT_FIND_UNUSED, 1)
    fake = [[0x100000 + 0x1000 * (r * len(numel) + v) for v in range(len(numel))] for r in range(W)]
    red.bind(fake, 0x10000000, None)
    return red


def test_unused_state_machine_matches_oracle(lib):
    from oracle.unused import UnusedReadiness
    numel = [1, 2, 1, 3, 1, 2]
    members, _ = assign_buckets(numel, 4, 8)
    rng = np.random.default_rng(3)
    W = 3
    for trial in range(60):
        used = rng.random((W, len(numel))) < 0.6
        g = used.any(axis=0)
        reported = [v for v in range(len(numel)) if g[v]]
        if not reported:
            continue
        order = [int(v) for v in rng.permutation(reported)]
        red = _dry_bound(numel, W, 8)
        assert red.get_members() == members
        red.set_local_used(used.tolist())
        red.begin_iteration()
        sm = UnusedReadiness(members, used.tolist())
        sm.begin_iteration()
        for v in order:
            assert red.mark_ready(v) == sm.mark_ready(v), (used, order)
        assert red.get_progress() == (len(members), [])
        # a new iteration without new bits: every variable reports again
        red.begin_iteration()
        for v in range(len(numel)):
            red.mark_ready(v)
        red.destroy()


def test_unused_errors_and_bitmap_or(lib):
    from reduction_reducer_gb300 import AlreadyReady, InvalidArg
    numel = [1, 1, 1]
    red = _dry_bound(numel, 2, 4)
    red.set_local_used([[True, False, False], [False, False, False]])
    red.set_local_used([[False, False, False], [False, True, False]])     # OR: 0 and 1 used
    red.begin_iteration()
    with pytest.raises(AlreadyReady):
        red.mark_ready(2)                     # unused on every replica: already ready
    assert red.mark_ready(1) == [0, 1]        # buckets: v2 -> 0 (unused, marked), v1 -> 1
    assert red.mark_ready(0) == [2]
    # no_sync bits accumulate into the next reduction's bitmap
    W, P = 2, 3
    fake = red.pointers([[0x2000 + 16 * i for i in range(P)] for _ in range(W)])
    red.accumulate_nosync(fake, fake, True, used=[[True, False, False], [False, False, False]])
    red.accumulate_nosync(fake, fake, False, used=[[False, False, True], [False, False, False]])
    red.begin_iteration()
    # v1 is unused in both micro-steps on both replicas: marked ready at the
    # first event, so bucket 1 goes out right after bucket 0 (v2)
    assert red.mark_ready(2) == [0, 1]
    with pytest.raises(AlreadyReady):
        red.mark_ready(1)
    assert red.mark_ready(0) == [2]
    plain = _make(numel, "f32", 4)
    plain.set_dry_run(True)
    plain.bind([[0x3000] * 3], 0x10000000, None)
    with pytest.raises(InvalidArg):
        plain.set_local_used([[True] * 3])    # needs DDP_OPT_FIND_UNUSED


def test_hook_registration_rules(lib):
    from reduction_reducer_gb300 import InvalidArg, NotBound, _lib as L
    red = _make([4, 4], "f32", 16)
    with pytest.raises(NotBound):
        red.register_comm_hook("mean", [0x1000, 0x2000])
    red.set_dry_run(True)
    red.bind([[0x1000, 0x1100], [0x2000, 0x2100]], 0x10000000, None)
    with pytest.raises(InvalidArg):
        red.register_comm_hook("mean", [0x1000, 0x2008])      # misaligned replica buffer
    red.register_comm_hook("mean", [0x1000, 0x2000])
    with pytest.raises(InvalidArg):
        red.register_comm_hook("mean", [0x1000, 0x2000])      # once only
    with pytest.raises(InvalidArg):
        red.set_option(L.OPT_FIND_UNUSED, 1)
    assert lib.ddp_status_string(-8) == b"DDP_ERR_HOOK"
    # the route of a built-in hook: fused by default, switchable between iterations only
    assert red.get_option(L.OPT_HOOK_FUSED) == 1
    red.set_option(L.OPT_HOOK_FUSED, 0)
    assert red.get_option(L.OPT_HOOK_FUSED) == 0
    red.begin_iteration()
    red.mark_ready(1)                                         # bucket 0 = [1]; bucket 1 = [0] still pending
    with pytest.raises(InvalidArg):
        red.set_option(L.OPT_HOOK_FUSED, 1)
    red.mark_ready(0)
    red.set_option(L.OPT_HOOK_FUSED, 1)


def test_last_step_binding_rules(lib):
    """ddp_bind_last_step on the host side (dry run, no device table): needs
    a binding, fp32, no unused-parameter tracking, no hook, a complete
    iteration; NULL entries only for zero-length variables; ddp_bind drops it."""
    from reduction_reducer_gb300 import InvalidArg, NotBound
    from reduction_reducer_gb300 import _lib as L
    numel = [3, 5, 0, 7]
    W = 2
    fake = [[0x100000 + 0x1000 * (r * 4 + v) for v in range(4)] for r in range(W)]
    last = [[0x800000 + 0x1000 * (r * 4 + v) for v in range(4)] for r in range(W)]
    red = _make(numel, "f32", 16)
    red.set_dry_run(True)
    with pytest.raises(NotBound):
        red.bind_last_step(last)
    red.bind(fake, 0x10000000, None)
    red.bind_last_step(last)
    with pytest.raises(InvalidArg):
        red.set_option(L.OPT_FIND_UNUSED, 1)
    red.begin_iteration()
    red.mark_ready(3)
    with pytest.raises(InvalidArg):
        red.bind_last_step(None)
    red.abort_iteration()
    red.bind_last_step(None)
    red.set_option(L.OPT_FIND_UNUSED, 1)
    with pytest.raises(InvalidArg):
        red.bind_last_step(last)
    red.set_option(L.OPT_FIND_UNUSED, 0)
    holes = [row[:] for row in last]
    holes[1][2] = 0                       # zero-length variable: no pointer needed
    red.bind_last_step(holes)
    holes[0][1] = 0
    with pytest.raises(InvalidArg):
        red.bind_last_step(holes)
    red.bind(fake, 0x10000000, None)      # a new binding drops the last step
    red.set_option(L.OPT_FIND_UNUSED, 1)
    b = _make(numel, "bf16", 16)
    b.set_dry_run(True)
    b.bind(fake, 0x10000000, None)
    with pytest.raises(InvalidArg):
        b.bind_last_step(last)


def test_hook_on_bucket_views_rules(lib):
    """replica_buffers = NULL needs the bound gradients to be views of the
    bucket layout (dry run: addresses only)."""
    from reduction_reducer_gb300 import InvalidArg
    red = _make([4, 4, 4], "f32", 48)           # one bucket, push order v2, v1, v0
    red.set_dry_run(True)
    assert red.get_members() == [[2, 1, 0]]
    red.bind([[0x1000, 0x1010, 0x1020], [0x2000, 0x2010, 0x2020]], 0x10000000, None)   # registration order
    with pytest.raises(InvalidArg):
        red.register_comm_hook("mean", None)
    red.bind([[0x1020, 0x1010, 0x1000], [0x2020, 0x2010, 0x2000]], 0x10000000, None)   # bucket order
    red.register_comm_hook("mean", None)
    z = _make([0, 4, 0], "f32", 48)               # zero-length members need no address
    z.set_dry_run(True)
    z.bind([[0, 0x1000, 0]], 0x10000000, None)
    z.register_comm_hook("mean", None)


def test_debug_build_exports_every_declared_symbol(lib):
    """The bounds-checking build carries the same ABI."""
    from reduction_reducer_gb300 import _lib
    if not os.path.exists(_lib.DEBUG_LIB_PATH):
        from reduction_reducer_gb300 import build
        build.build_debug()
    dbg = _lib.load(_lib.DEBUG_LIB_PATH)
    for name in header_functions():
        assert hasattr(dbg, name), name
    assert dbg is not lib


def test_selftest_rejects_bad_limits(lib):
    import ctypes as C
    code = C.c_int32(7)
    assert lib.ddp_selftest_bounded_wait(0, C.byref(code)) == -1 and code.value == 0
    assert lib.ddp_selftest_bounded_wait(4_000_000_001, C.byref(code)) == -1
    assert lib.ddp_selftest_bounded_wait(1000, None) == -1


def test_debug_record_rules(lib):
    from reduction_reducer_gb300 import NotBound
    red = _make([4, 4], "f32", 16)
    with pytest.raises(NotBound):
        red.debug_record()
    red.set_dry_run(True)
    red.bind([[0x1000, 0x1100]], 0x10000000, None)
    assert red.debug_record() == (0, 0)      # dry run: nothing on a device


@pytest.mark.parametrize("seed", range(200))
def test_host_core_fuzz_matches_oracle(lib, seed):
    """Seeded random models (up to 300 tensors, empty ones included), caps,
    dtypes and ready orders (random, or reverse with stragglers so buckets
    park): locators, arena offsets and the launch/park sequence of every
    event match the oracle exactly."""
    rng = np.random.default_rng(60_000 + seed)
    P = int(rng.integers(1, 301))
    numel = [int(x) for x in rng.choice([0, 1, 3, 64, 1000, 4096, 70001, 1 << 20], size=P,
                                        p=[0.05, 0.1, 0.1, 0.2, 0.2, 0.2, 0.1, 0.05])]
    dtype = "f32" if rng.random() < 0.5 else "bf16"
    elem = 4 if dtype == "f32" else 2
    cap = int(rng.choice([0, 4096, 65536, 1 << 20, 4 << 20, 25 << 20]))
    red = _make(numel, dtype, cap)
    members, locs = assign_buckets(numel, elem, cap)
    assert red.get_members() == members
    assert red.get_locators() == [(l.bucket, l.intra, l.offset, l.length) for l in locs]
    B, offs = red.get_bucket_info()
    lens = [sum(numel[v] for v in m) for m in members]
    assert offs == [sum(lens[:b]) for b in range(B + 1)]
    if rng.random() < 0.5:
        order = [int(v) for v in rng.permutation(P)]
    else:
        order = gen.straggler_order(members, p=0.5, seed=seed)
    assert _run_dry(red, order) == _oracle_trace(members, order)
    red.destroy()


def test_launch_shape_options(lib):
    """Option ranges and defaults of the launch shapes: bulk-copy CTAs per SM
    0 (resident waves, the default) .. 8, register-streaming CTAs per SM
    0 (resident waves, the default) .. 64, and the kernel-choice threshold of
    6 x 2^20 median elements."""
    from reduction_reducer_gb300 import InvalidArg, _lib as L
    red = _make([4096] * 8, "f32", 64 << 10)
    assert red.get_option(L.OPT_TMA_CTAS_PER_SM) == 0
    assert red.get_option(L.OPT_CTAS_PER_SM) == 0
    assert red.get_option(L.OPT_AUTO_MIN_ELEMS) == 6 << 20
    for v in (0, 1, 2, 8):
        red.set_option(L.OPT_TMA_CTAS_PER_SM, v)
        assert red.get_option(L.OPT_TMA_CTAS_PER_SM) == v
    for bad in (-1, 9):
        with pytest.raises(InvalidArg):
            red.set_option(L.OPT_TMA_CTAS_PER_SM, bad)
    for bad in (-1, 65):
        with pytest.raises(InvalidArg):
            red.set_option(L.OPT_CTAS_PER_SM, bad)
    red.destroy()
