"""ctypes declarations of the C ABI in include/ddp_reducer.h.

Argument marshalling only.  Loading fails loudly when the library has not
been built: there is no fallback implementation.
"""

from __future__ import annotations

import ctypes as C
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libddpreducer.so")

DDP_F32, DDP_BF16 = 0, 1

STATUS = {
    0: "DDP_OK",
    -1: "DDP_ERR_INVALID_ARG",
    -2: "DDP_ERR_ALREADY_READY",
    -3: "DDP_ERR_OUT_OF_ORDER",
    -4: "DDP_ERR_PRIOR_REDUCTION_UNFINISHED",
    -5: "DDP_ERR_NOT_BOUND",
    -6: "DDP_ERR_CUDA",
    -7: "DDP_ERR_NO_MEMORY",
    -8: "DDP_ERR_HOOK",
}

OPT_DRY_RUN, OPT_CTAS_PER_SM, OPT_PDL, OPT_BLOCK_THREADS = 0, 1, 2, 3
OPT_KERNEL, OPT_STAGES, OPT_STAGE_BYTES, OPT_TMA_CTAS_PER_SM = 4, 5, 6, 7
OPT_AUTO_MIN_ELEMS, OPT_CHAINED, OPT_QUERY_KERNEL, OPT_FIND_UNUSED = 8, 9, 10, 11
OPT_HOOK_FUSED, OPT_COALESCE_ELEMS = 12, 13
KERNEL_LDG, KERNEL_TMA, KERNEL_AUTO = 0, 1, 2


class Locator(C.Structure):
    _fields_ = [("bucket", C.c_int32), ("intra", C.c_int32), ("offset", C.c_int64), ("length", C.c_int64)]


class GradBucket(C.Structure):
    """struct ddp_grad_bucket."""
    _fields_ = [("index", C.c_int32), ("num_buckets", C.c_int32), ("is_last", C.c_int32), ("W", C.c_int32),
                ("dtype", C.c_int32), ("n_vars", C.c_int32), ("numel", C.c_int64),
                ("replicas", C.POINTER(C.c_void_p)), ("result", C.c_void_p),
                ("variables", C.POINTER(C.c_int32)), ("offsets", C.POINTER(C.c_int64)),
                ("lengths", C.POINTER(C.c_int64))]


# int (*ddp_comm_hook_fn)(void* state, const ddp_grad_bucket* bucket, void* stream)
HOOKFN = C.CFUNCTYPE(C.c_int, C.c_void_p, C.POINTER(GradBucket), C.c_void_p)

# name -> (restype, argtypes); every symbol of include/ddp_reducer.h
SIGNATURES = {
    "ddp_build_buckets": (C.c_int, [C.POINTER(C.c_int64), C.c_int32, C.c_int, C.c_int64, C.POINTER(C.c_void_p)]),
    "ddp_get_locators": (C.c_int, [C.c_void_p, C.POINTER(Locator)]),
    "ddp_get_bucket_info": (C.c_int, [C.c_void_p, C.POINTER(C.c_int32), C.POINTER(C.c_int64)]),
    "ddp_bind": (C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_void_p), C.c_void_p, C.POINTER(C.c_void_p), C.c_int32]),
    "ddp_begin_iteration": (C.c_int, [C.c_void_p]),
    "ddp_abort_iteration": (C.c_int, [C.c_void_p]),
    "ddp_mark_ready": (C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_int32), C.POINTER(C.c_int32), C.c_void_p]),
    "ddp_mark_ready_many": (C.c_int, [C.c_void_p, C.POINTER(C.c_int32), C.c_int32, C.POINTER(C.c_int32), C.c_void_p]),
    "ddp_reduce_bucket": (C.c_int, [C.c_void_p, C.c_int32, C.c_void_p]),
    "ddp_reduce_all": (C.c_int, [C.c_void_p, C.c_void_p]),
    "ddp_get_progress": (C.c_int, [C.c_void_p, C.POINTER(C.c_int32), C.POINTER(C.c_int32), C.POINTER(C.c_int32)]),
    "ddp_set_local_used": (C.c_int, [C.c_void_p, C.POINTER(C.c_uint8)]),
    "ddp_accumulate_nosync_used": (C.c_int, [C.c_void_p, C.POINTER(C.c_void_p), C.POINTER(C.c_void_p),
                                             C.POINTER(C.c_uint8), C.c_int32, C.c_void_p]),
    "ddp_register_comm_hook": (C.c_int, [C.c_void_p, HOOKFN, C.c_void_p, C.POINTER(C.c_void_p)]),
    "ddp_hook_mean": (C.c_int, [C.c_void_p, C.POINTER(GradBucket), C.c_void_p]),
    "ddp_hook_bf16_compress": (C.c_int, [C.c_void_p, C.POINTER(GradBucket), C.c_void_p]),
    "ddp_get_ready_trace": (C.c_int, [C.c_void_p, C.POINTER(C.c_int32), C.POINTER(C.c_int32)]),
    "ddp_rebuild_buckets": (C.c_int, [C.c_void_p, C.POINTER(C.c_int32), C.c_int64, C.c_int64]),
    "ddp_accumulate_nosync": (C.c_int, [C.c_void_p, C.POINTER(C.c_void_p), C.POINTER(C.c_void_p), C.c_int32, C.c_void_p]),
    "ddp_bind_last_step": (C.c_int, [C.c_void_p, C.POINTER(C.c_void_p)]),
    "ddp_set_option": (C.c_int, [C.c_void_p, C.c_int32, C.c_int64]),
    "ddp_get_option": (C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_int64)]),
    "ddp_get_launch_count": (C.c_int, [C.c_void_p, C.POINTER(C.c_int64)]),
    "ddp_get_device_status": (C.c_int, [C.c_void_p, C.POINTER(C.c_int32)]),
    "ddp_get_debug_record": (C.c_int, [C.c_void_p, C.POINTER(C.c_int32), C.POINTER(C.c_int64)]),
    "ddp_selftest_bounded_wait": (C.c_int, [C.c_int64, C.POINTER(C.c_int32)]),
    "ddp_reduce_all_noalloc": (C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_void_p), C.c_void_p,
                                         C.POINTER(C.c_void_p), C.c_int32, C.c_void_p]),
    "ddp_shard_range": (C.c_int, [C.c_int64, C.c_int32, C.c_int32, C.POINTER(C.c_int64), C.POINTER(C.c_int64),
                                  C.POINTER(C.c_int64)]),
    "ddp_shard_mean": (C.c_int, [C.c_int32, C.c_int, C.POINTER(C.c_void_p), C.c_void_p, C.c_int64, C.c_void_p]),
    "ddp_read_launch_trace": (C.c_int, [C.POINTER(C.c_uint64), C.POINTER(C.c_int32), C.POINTER(C.c_int64)]),
    "ddp_status_string": (C.c_char_p, [C.c_int]),
    "ddp_last_error": (C.c_char_p, [C.c_void_p]),
    "ddp_destroy": (None, [C.c_void_p]),
}

_lib = None


DEBUG_LIB_PATH = os.path.join(PKG, "libddpreducer_debug.so")
TRACE_LIB_PATH = os.path.join(PKG, "libddpreducer_trace.so")
TRACE_LAUNCHES, TRACE_CTAS = 64, 4096
_variants = {}


def load(path: str = LIB_PATH):
    """Load (once per path) and declare the library; raises if it is missing.
    ``DEBUG_LIB_PATH`` is the bounds-checking build of the same sources."""
    global _lib
    if path != LIB_PATH:
        if path not in _variants:
            _variants[path] = _open(path)
        return _variants[path]
    if _lib is None:
        _lib = _open(path)
    return _lib


def _open(path: str):
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it first with "
            "`python -c 'import __graft_entry__ as g; g.build()'` "
            "(or `python -m reduction_reducer_gb300.build`). There is no fallback implementation.")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib
