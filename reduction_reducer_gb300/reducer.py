"""Thin Python binding of the C ABI (same names as include/ddp_reducer.h).

Only argument marshalling happens here: tensors become device addresses,
streams become ``cudaStream_t`` handles, status codes become exceptions.
Every step of the gradient path runs in the library's C++ host core and
CUDA kernels.
"""

from __future__ import annotations

import ctypes as C

from . import _lib
from ._lib import DDP_BF16, DDP_F32, Locator

DTYPES = {"f32": DDP_F32, "bf16": DDP_BF16}


class DDPError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        self.name = _lib.STATUS.get(status, str(status))
        super().__init__(f"{self.name}: {detail}")


class InvalidArg(DDPError): pass
class AlreadyReady(DDPError): pass
class OutOfOrder(DDPError): pass
class PriorReductionUnfinished(DDPError): pass
class NotBound(DDPError): pass
class CudaError(DDPError): pass
class NoMemory(DDPError): pass
class HookError(DDPError): pass


_ERRORS = {-1: InvalidArg, -2: AlreadyReady, -3: OutOfOrder, -4: PriorReductionUnfinished,
           -5: NotBound, -6: CudaError, -7: NoMemory, -8: HookError}


def _check_status(st: int, detail) -> None:
    """Raise the exception of a nonzero status (``detail``: message or None)."""
    if st != 0:
        raise _ERRORS.get(st, DDPError)(st, detail or _lib.STATUS.get(st, ""))


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


_torch = None   # resolved on first use: torch.cuda when a GPU is present, else False


def _stream(stream) -> int:
    """cudaStream_t of a torch stream, an int handle, or (None) torch's
    current stream; 0 without a GPU (dry runs)."""
    global _torch
    if stream is None:
        if _torch is None:
            import torch
            _torch = torch.cuda if torch.cuda.is_available() else False
        return int(_torch.current_stream().cuda_stream) if _torch else 0
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _ptr_array(ptrs):
    arr = (C.c_void_p * max(len(ptrs), 1))()
    for i, p in enumerate(ptrs):
        arr[i] = p or None
    return arr


def read_launch_trace(lib_path: str = _lib.TRACE_LIB_PATH):
    """The launch trace of the trace build (``ddp_read_launch_trace``):
    (stamps [TRACE_LAUNCHES, TRACE_CTAS, 4] uint64 ns, grid per slot, launches
    traced so far; -1 for a build without the trace)."""
    import numpy as np
    lib = _lib.load(lib_path)
    buf = np.zeros((_lib.TRACE_LAUNCHES, _lib.TRACE_CTAS, 4), np.uint64)
    grid = (C.c_int32 * _lib.TRACE_LAUNCHES)()
    seq = C.c_int64()
    _check_status(lib.ddp_read_launch_trace(buf.ctypes.data_as(C.POINTER(C.c_uint64)), grid, C.byref(seq)), None)
    return buf, list(grid), seq.value


class Reducer:
    """One bucketed reducer context (``ddp_ctx``)."""

    def __init__(self, numel, dtype: str = "f32", cap_bytes: int = 25 << 20, lib_path: str = _lib.LIB_PATH):
        """lib_path: the library build to use (``_lib.DEBUG_LIB_PATH``: the
        bounds-checking build)."""
        self.lib = _lib.load(lib_path)
        self.numel = [int(n) for n in numel]
        self.dtype = dtype
        arr = (C.c_int64 * max(len(self.numel), 1))(*self.numel)
        h = C.c_void_p()
        st = self.lib.ddp_build_buckets(arr, len(self.numel), DTYPES[dtype], int(cap_bytes), C.byref(h))
        if st != 0:
            raise _ERRORS.get(st, DDPError)(st, self.lib.ddp_last_error(None).decode())
        self._h = h
        B = C.c_int32()
        self.lib.ddp_get_bucket_info(self._h, C.byref(B), None)
        self.B = B.value
        self.P = len(self.numel)
        self._launched = (C.c_int32 * max(self.B, 1))()
        self._n_launched = C.c_int32()                  # reused by every mark_ready call
        self._n_ref = C.byref(self._n_launched)
        self._keep = ()

    build_buckets = classmethod(lambda cls, numel, dtype="f32", cap_bytes=25 << 20: cls(numel, dtype, cap_bytes))

    # ---------------------------------------------------------------- helpers
    def _check(self, st: int):
        if st != 0:
            detail = self.lib.ddp_last_error(self._h) or b""
            raise _ERRORS.get(st, DDPError)(st, detail.decode())

    # ---------------------------------------------------------------- info
    def get_locators(self):
        out = (Locator * max(self.P, 1))()
        self._check(self.lib.ddp_get_locators(self._h, out))
        return [(out[v].bucket, out[v].intra, out[v].offset, out[v].length) for v in range(self.P)]

    def get_bucket_info(self):
        B = C.c_int32()
        offs = (C.c_int64 * (self.B + 1))()
        self._check(self.lib.ddp_get_bucket_info(self._h, C.byref(B), offs))
        return B.value, list(offs)

    def get_members(self):
        members = [[] for _ in range(self.B)]
        for v, (b, intra, _, _) in enumerate(self.get_locators()):
            members[b].append((intra, v))
        return [[v for _, v in sorted(m)] for m in members]

    def arena_numel(self) -> int:
        return self.get_bucket_info()[1][-1]

    # ---------------------------------------------------------------- bind
    def bind(self, grads, bucket_arena, grad_out=None):
        """grads: W lists of P tensors (or device addresses); bucket_arena: fp32
        tensor of ``arena_numel()`` elements; grad_out: None (gradient as bucket
        view), a list of P fp32 tensors (one shared copy) or W such lists."""
        W = len(grads)
        flat = []
        want = "torch.float32" if self.dtype == "f32" else "torch.bfloat16"
        for r in range(W):
            if len(grads[r]) != self.P:
                raise ValueError("each replica needs one gradient per parameter")
            for v, t in enumerate(grads[r]):
                if not isinstance(t, int) and t is not None:
                    if t.numel() != self.numel[v] or not t.is_contiguous() or str(t.dtype) != want:
                        raise ValueError(f"replica {r} gradient {v}: expected {self.numel[v]} contiguous {want}")
                flat.append(_ptr(t))
        if grad_out is None:
            outs = []
        elif len(grad_out) == self.P and (self.P == 0 or not isinstance(grad_out[0], (list, tuple))):
            outs = [grad_out]
        else:
            outs = list(grad_out)
        out_flat = []
        for o in outs:
            for v, t in enumerate(o):
                if not isinstance(t, int) and t is not None:
                    if t.numel() != self.numel[v] or not t.is_contiguous() or str(t.dtype) != "torch.float32":
                        raise ValueError(f"output {v}: expected {self.numel[v]} contiguous fp32")
                out_flat.append(_ptr(t))
        if not isinstance(bucket_arena, int) and bucket_arena is not None:
            if bucket_arena.numel() < self.arena_numel() or str(bucket_arena.dtype) != "torch.float32":
                raise ValueError("bucket_arena too small or not fp32")
        self._gp = _ptr_array(flat)
        self._op = _ptr_array(out_flat) if outs else None
        self._check(self.lib.ddp_bind(self._h, W, self._gp, _ptr(bucket_arena),
                                      self._op, len(outs)))
        self.W = W
        self._keep = (grads, bucket_arena, grad_out)

    # ---------------------------------------------------------------- iteration
    def begin_iteration(self):
        self._check(self.lib.ddp_begin_iteration(self._h))

    def abort_iteration(self):
        self._check(self.lib.ddp_abort_iteration(self._h))

    def mark_ready(self, var: int, stream=None):
        n = self._n_launched
        self._check(self.lib.ddp_mark_ready(self._h, int(var), self._launched, self._n_ref, _stream(stream)))
        return [self._launched[i] for i in range(n.value)] if n.value else []

    def mark_ready_many(self, vars_, stream=None):
        """Ready events in order, in one call; returns how many were processed."""
        n = len(vars_)
        arr = vars_ if isinstance(vars_, C.Array) else (C.c_int32 * max(n, 1))(*vars_)
        done = C.c_int32()
        self._check(self.lib.ddp_mark_ready_many(self._h, arr, n, C.byref(done), _stream(stream)))
        return done.value

    def reduce_bucket(self, bucket: int, stream=None):
        self._check(self.lib.ddp_reduce_bucket(self._h, int(bucket), _stream(stream)))

    def reduce_all(self, stream=None):
        self._check(self.lib.ddp_reduce_all(self._h, _stream(stream)))

    def get_progress(self):
        nxt, n = C.c_int32(), C.c_int32()
        parked = (C.c_int32 * max(self.B, 1))()
        self._check(self.lib.ddp_get_progress(self._h, C.byref(nxt), parked, C.byref(n)))
        return nxt.value, [parked[i] for i in range(n.value)]

    # ---------------------------------------------------------------- communication hooks
    def register_comm_hook(self, hook, replica_buffers=None, state=None):
        """hook: "mean" | "bf16_compress" (built-in) or a callable
        ``hook(bucket: _lib.GradBucket, stream: int) -> int|None`` that enqueues
        its reduction into ``bucket.result`` on ``stream``; replica_buffers: W
        device buffers (tensors or addresses) of ``arena_numel()`` elements of
        the gradient dtype, or None when the bound gradients are views of the
        bucket layout (the hook then reads them in place)."""
        if hook == "mean":
            fn = C.cast(self.lib.ddp_hook_mean, _lib.HOOKFN)
        elif hook == "bf16_compress":
            fn = C.cast(self.lib.ddp_hook_bf16_compress, _lib.HOOKFN)
        else:
            user = hook

            def trampoline(_state, bucket, stream):
                try:
                    rc = user(bucket.contents, stream)
                    return int(rc or 0)
                except Exception:       # noqa: BLE001 -- a Python error must not cross the C ABI
                    return 1
            fn = _lib.HOOKFN(trampoline)
        rb = None if replica_buffers is None else _ptr_array([_ptr(t) for t in replica_buffers])
        self._check(self.lib.ddp_register_comm_hook(self._h, fn, state, rb))
        self._hook_keep = (fn, rb, replica_buffers, hook)

    # ---------------------------------------------------------------- rebuild
    def get_ready_trace(self):
        n = C.c_int32()
        buf = (C.c_int32 * max(self.P, 1))()
        self._check(self.lib.ddp_get_ready_trace(self._h, buf, C.byref(n)))
        return [buf[i] for i in range(n.value)]

    def rebuild_buckets(self, order=None, first_cap_bytes=None, cap_bytes=25 << 20):
        """Re-pack in ``order`` (default: the last finished iteration's trace)."""
        arr = None if order is None else (C.c_int32 * max(self.P, 1))(*order)
        fc = cap_bytes if first_cap_bytes is None else first_cap_bytes
        self._check(self.lib.ddp_rebuild_buckets(self._h, arr, int(fc), int(cap_bytes)))
        B = C.c_int32()
        self.lib.ddp_get_bucket_info(self._h, C.byref(B), None)
        self.B = B.value
        self._launched = (C.c_int32 * max(self.B, 1))()
        self._n_launched = C.c_int32()                  # reused by every mark_ready call
        self._n_ref = C.byref(self._n_launched)

    # ---------------------------------------------------------------- no allocation
    def reduce_all_noalloc(self, grads, bucket_arena, grad_out=None, stream=None):
        """Every bucket in one pass without any device allocation: for callers
        that may not call cudaMalloc (a framework whose caching allocator owns
        the device memory budget, real-time loops where an allocation and the
        device synchronisation it implies are not allowed).  Arguments as in
        ``bind``; the table goes to the library's static device scratch
        (256 KiB), shared by all calls, so calls that can overlap on the GPU
        race.  The first call on a device looks up the scratch's address and
        should come before any stream capture.  The context's launch options
        are not used, and the bounded waits' status is not reported."""
        W = len(grads)
        flat = [_ptr(t) for rep in grads for t in rep]
        if grad_out is None:
            outs = []
        elif len(grad_out) == self.P and (self.P == 0 or not isinstance(grad_out[0], (list, tuple))):
            outs = [grad_out]
        else:
            outs = list(grad_out)
        out_flat = [_ptr(t) for o in outs for t in o]
        gp = _ptr_array(flat)
        op = _ptr_array(out_flat) if outs else None
        self._check(self.lib.ddp_reduce_all_noalloc(self._h, W, gp, _ptr(bucket_arena), op, len(outs),
                                                    _stream(stream)))

    # ---------------------------------------------------------------- no_sync
    @staticmethod
    def pointers(replicas):
        """W lists of P tensors -> a reusable array of W*P device addresses
        (marshalling done once instead of on every call)."""
        return _ptr_array([_ptr(t) for rep in replicas for t in rep])

    @staticmethod
    def bits(used):
        """W lists of P flags -> a reusable array of W*P local-use bytes."""
        if isinstance(used, C.Array):
            return used
        flat = [1 if u else 0 for rep in used for u in rep]
        return (C.c_uint8 * max(len(flat), 1))(*flat)

    def accumulate_nosync(self, acc, g, first_step: bool, stream=None, used=None):
        """acc, g: W lists of P fp32 tensors, or arrays from ``pointers``;
        used: W lists of P local-use flags of this micro-step (None = all)."""
        a = acc if isinstance(acc, C.Array) else self.pointers(acc)
        b = g if isinstance(g, C.Array) else self.pointers(g)
        if used is None:
            self._check(self.lib.ddp_accumulate_nosync(self._h, a, b, 1 if first_step else 0, _stream(stream)))
        else:
            self._check(self.lib.ddp_accumulate_nosync_used(self._h, a, b, self.bits(used),
                                                            1 if first_step else 0, _stream(stream)))

    def bind_last_step(self, g_last=None):
        """Fuse the synchronizing micro-step that ends a no_sync block into the
        reductions: g_last is W lists of P fp32 tensors (or an array from
        ``pointers``) added per replica to the bound accumulated gradients;
        None unbinds it."""
        if g_last is None:
            self._check(self.lib.ddp_bind_last_step(self._h, None))
            self._last = None
            return
        if not isinstance(g_last, C.Array) and getattr(self, "W", None) is not None:
            if len(g_last) != self.W or any(len(rep) != self.P for rep in g_last):
                raise ValueError("g_last needs W lists of P tensors")
            for rep in g_last:
                for v, t in enumerate(rep):
                    if not isinstance(t, int) and t is not None:
                        if t.numel() != self.numel[v] or not t.is_contiguous() or str(t.dtype) != "torch.float32":
                            raise ValueError(f"last-step gradient {v}: expected {self.numel[v]} contiguous fp32")
        arr = g_last if isinstance(g_last, C.Array) else self.pointers(g_last)
        self._check(self.lib.ddp_bind_last_step(self._h, arr))
        self._last = (g_last, arr)

    # ---------------------------------------------------------------- unused parameters
    def set_local_used(self, used):
        """used: W lists of P flags, or an array from ``bits`` (None = all used)."""
        self._check(self.lib.ddp_set_local_used(self._h, None if used is None else self.bits(used)))

    # ---------------------------------------------------------------- options
    def set_option(self, option: int, value: int):
        self._check(self.lib.ddp_set_option(self._h, int(option), int(value)))

    def get_option(self, option: int) -> int:
        v = C.c_int64()
        self._check(self.lib.ddp_get_option(self._h, int(option), C.byref(v)))
        return v.value

    def set_dry_run(self, on: bool = True):
        self.set_option(_lib.OPT_DRY_RUN, 1 if on else 0)

    def debug_record(self):
        """Read and clear the bounds-check record: (code, element index);
        (0, 0) when no check failed (always, in a release build)."""
        code, index = C.c_int32(), C.c_int64()
        self._check(self.lib.ddp_get_debug_record(self._h, C.byref(code), C.byref(index)))
        return code.value, index.value

    def device_status(self) -> int:
        """Read and clear the kernels' device status word (synchronous)."""
        st = C.c_int32()
        self._check(self.lib.ddp_get_device_status(self._h, C.byref(st)))
        return st.value

    def launch_count(self) -> int:
        n = C.c_int64()
        self._check(self.lib.ddp_get_launch_count(self._h, C.byref(n)))
        return n.value

    def destroy(self):
        if getattr(self, "_h", None):
            self.lib.ddp_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass


def selftest_bounded_wait(limit_cycles: int, lib_path: str = _lib.LIB_PATH) -> int:
    """Run the bounded-wait self-test on the current device; returns the
    status code the abandoned wait wrote (3 when it ended as designed)."""
    lib = _lib.load(lib_path)
    code = C.c_int32()
    st = lib.ddp_selftest_bounded_wait(int(limit_cycles), C.byref(code))
    if st != 0:
        raise _ERRORS.get(st, DDPError)(st, "ddp_selftest_bounded_wait")
    return code.value
