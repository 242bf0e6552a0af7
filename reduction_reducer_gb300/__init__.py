"""GB300-native DDP Reducer gradient path.

C++ host core + hand-written sm_103a CUDA kernels behind the C ABI of
``include/ddp_reducer.h`` (``libddpreducer.so``, built in-tree by
``reduction_reducer_gb300.build``); this package is the thin Python binding.
"""

from .reducer import (AlreadyReady, CudaError, DDPError, HookError, InvalidArg, NoMemory,  # noqa: F401
                      NotBound, OutOfOrder, PriorReductionUnfinished, Reducer, selftest_bounded_wait)
from ._lib import LIB_PATH, load  # noqa: F401
