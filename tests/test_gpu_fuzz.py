"""Seeded random combinations of the fused bucket pass against the oracle.

The fixed parity cases vary one thing at a time; these draw whole
configurations: parameter count and a size mix (empty tensors, odd small
sizes, sizes around the vector and tile widths, an occasional large one),
W (including widths without a compiled-in body), f32 or bf16, the cap
(per-gradient to one bucket), the output mode (as-view, one copy, W
copies), misaligned views, a random ready order, every launch mode and
every kernel choice.  Each case is compared bit for bit with the oracle,
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
    return dict(numel=numel, W=W, dtype=dtype, cap=cap, n_out=n_out, odd=bool(rng.random() < 0.3),
                mode=str(rng.choice(MODES)), kernel=str(rng.choice(KERNELS)))


@pytest.mark.parametrize("seed", range(200))
def test_fuzz_bucket_pass(seed):
    c = draw_case(seed)
    full_compare(c["numel"], c["W"], c["dtype"], c["cap"], order="random", n_out=c["n_out"], mode=c["mode"],
                 odd=c["odd"], kernel=c["kernel"])
