"""Synthetic workload definitions shared by tests, the oracle's pins and the bench.

Shapes of the evaluated models and seeded input generators only; nothing
here implements the reducer.
"""

from . import gen, shapes  # noqa: F401
