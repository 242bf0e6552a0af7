"""Checks of the shared workload definitions (no GPU)."""

import os

import numpy as np

from oracle.buckets import assign_buckets
from oracle.readiness import launch_events
from workloads import gen, shapes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_parameter_counts():
    # element counts of the models' published hyperparameters
    assert (len(shapes.resnet50()), sum(shapes.numels(shapes.resnet50()))) == (161, 25_557_032)
    assert (len(shapes.bert_large()), sum(shapes.numels(shapes.bert_large()))) == (391, 335_141_888)
    assert (len(shapes.gpt2_medium()), sum(shapes.numels(shapes.gpt2_medium()))) == (292, 354_823_168)
    assert shapes.numels(shapes.linear_10x10()) == [100, 10]


def read_order(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [int(l) for l in f if l.strip() and not l.startswith("#")]


def test_bert_ready_order_fixture():
    numel = shapes.numels(shapes.bert_large())
    members, _ = assign_buckets(numel, 4, 25 << 20)
    order = read_order("bert_large_ready_order.txt")
    assert sorted(order) == list(range(len(numel)))
    assert order == gen.straggler_order(members, p=0.25, seed=0)
    _, trace = launch_events(members, order)
    parks = sum(1 for (v, b, pend, launched, parked) in trace if pend == 0 and b not in launched)
    assert parks >= 1


def test_bf16_rne():
    x = np.array([1.0, 1.00390625, 1.01171875, -3.0, 1e-40], np.float32)
    bits = gen.f32_to_bf16_bits(x)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even (1.0); 1 + 3*2^-8 -> 1 + 2^-6
    assert list(bits[:4]) == [0x3F80, 0x3F80, 0x3F82, 0xC040]


def test_draws_are_seeded():
    a = gen.draw_flat_np(100, 3, 2)
    b = gen.draw_flat_np(100, 3, 2)
    c = gen.draw_flat_np(100, 4, 2)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    assert abs(float(np.std(gen.draw_flat_np(100000, 0))) - 1e-3) < 2e-5
