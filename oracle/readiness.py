"""Oracle: the per-iteration bucket readiness state machine.

Test infrastructure only; see the package docstring.

What the pages fix ("NCCL 专家课程 30", sections "Variable 到 Bucket" and
"Bucket 必须按序发起"; paper summary "The per-hook logic" and "Launching
AllReduce in order"):

* every bucket starts an iteration with ``pending`` = its member count;
* when a variable becomes ready its gradient goes into its bucket view and
  ``pending`` of its bucket drops by one; at zero the bucket is ready;
* a ready bucket whose index is above the next-to-launch cursor waits
  (it is "parked"); otherwise, starting at the cursor, every consecutive
  bucket whose ``pending`` is zero is launched and the cursor advances;
* so buckets are launched strictly in index order whatever the ready
  order (the sequence diagram in which bucket 2 is ready before bucket 1:
  2 parks, then 1 and 2 go out together).

Failure cases the pages name:

* a variable reported twice in one iteration has no meaning in the
  reducer's counting (its bucket would be released early): rejected;
* an iteration that did not launch every bucket (a parameter that never
  got a gradient) makes the *next* iteration's start fail with "Expected
  to have finished reduction in the prior iteration" ("Distributed Data
  Parallel" notes, "When a parameter never receives a gradient";
  "NCCL 专家课程 30", "未检测的失败").

Explicit launches (readings, no counterpart on the pages beyond the
in-order rule): ``launch_next(b)`` forces bucket ``b`` -- which must be the
cursor -- complete and then runs the same in-order release;
``launch_rest()`` completes and launches every bucket not yet launched.
"""

from __future__ import annotations


class ReducerStateError(Exception):
    pass


class AlreadyReady(ReducerStateError):
    pass


class OutOfOrder(ReducerStateError):
    pass


class PriorReductionUnfinished(ReducerStateError):
    pass


class ReadinessOracle:
    def __init__(self, members):
        self.members = [list(m) for m in members]
        self.B = len(self.members)
        self.bucket_of = {}
        for b, vs in enumerate(self.members):
            for v in vs:
                self.bucket_of[v] = b
        self.P = len(self.bucket_of)
        self.active = False          # an iteration has started and not finished
        self.trace = []
        self._reset()

    def _reset(self):
        self.pending = [len(m) for m in self.members]
        self.ready = [False] * self.P
        self.next = 0
        self.trace = []

    # ------------------------------------------------------------ iteration
    def begin_iteration(self):
        if self.active:
            raise PriorReductionUnfinished(
                "Expected to have finished reduction in the prior iteration")
        self._reset()
        self.active = self.B > 0

    def abort_iteration(self):
        self._reset()
        self.active = False

    def _ensure_started(self):
        if not self.active:
            self.begin_iteration()

    def _release(self):
        launched = []
        while self.next < self.B and self.pending[self.next] == 0:
            launched.append(self.next)
            self.next += 1
        if self.next == self.B:
            self.active = False
        return launched

    def parked(self):
        return [b for b in range(self.next, self.B) if self.pending[b] == 0]

    # ------------------------------------------------------------ events
    def mark_ready(self, v: int):
        """A variable's gradient is ready.  Returns the buckets launched
        by this event, in launch order."""
        if not (0 <= v < self.P):
            raise ValueError("variable index out of range")
        self._ensure_started()
        if self.ready[v]:
            raise AlreadyReady(v)
        self.ready[v] = True
        b = self.bucket_of[v]
        self.pending[b] -= 1
        launched = []
        if self.pending[b] == 0 and b <= self.next:
            launched = self._release()
        self.trace.append((v, b, self.pending[b], launched, self.parked()))
        return launched

    def launch_next(self, b: int):
        """Explicit launch of bucket ``b``; it must be the next one."""
        self._ensure_started()
        if b != self.next:
            raise OutOfOrder(b)
        for v in self.members[b]:
            self.ready[v] = True
        self.pending[b] = 0
        return self._release()

    def launch_rest(self):
        """Launch every bucket not launched yet, in index order."""
        self._ensure_started()
        out = []
        for b in range(self.next, self.B):
            for v in self.members[b]:
                self.ready[v] = True
            self.pending[b] = 0
            out.append(b)
        self.next = self.B
        self.active = False
        return out


def launch_events(members, order):
    """Run one iteration over a full ready order.

    Returns ``(launch_at, trace)`` where ``launch_at[b]`` is the index of the
    ready event that launched bucket b (None if never launched).
    """
    sm = ReadinessOracle(members)
    sm.begin_iteration()
    launch_at = [None] * len(members)
    for t, v in enumerate(order):
        for b in sm.mark_ready(v):
            launch_at[b] = t
    return launch_at, sm.trace
