"""Write the stored ready orders of the synthetic workloads.

Calls only the oracle (for the bucket membership the straggler moves
need) and the shared workload generators.  Run from the repository root:

    python tests/golden/make_ready_orders.py

Output: ``tests/golden/bert_large_ready_order.txt`` -- one variable index
per line, the order in which BERT-large's gradients report ready: reverse
registration order with seeded straggler moves across bucket boundaries
(probability 0.25, ``random.Random(0)``) so that some buckets complete out
of order and have to park.
"""

import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle.buckets import assign_buckets  # noqa: E402
from workloads import gen, shapes  # noqa: E402

CAP = 25 << 20


def bert_order():
    numel = shapes.numels(shapes.bert_large())
    members, _ = assign_buckets(numel, 4, CAP)
    return gen.straggler_order(members, p=0.25, seed=0)


def main():
    order = bert_order()
    path = os.path.join(HERE, "bert_large_ready_order.txt")
    with open(path, "w") as f:
        f.write("# BERT-large ready order, 25 MiB buckets, straggler moves p=0.25 seed 0\n")
        f.write("# written by tests/golden/make_ready_orders.py\n")
        for v in order:
            f.write(f"{v}\n")
    print(path, len(order))


if __name__ == "__main__":
    main()
