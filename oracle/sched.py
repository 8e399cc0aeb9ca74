"""Iteration-level and request-level schedulers (oracle).

Iteration-level scheduling ([houmin] 3.1.1; [0h-n0] "Request-Level vs
Iteration-Level Scheduling"; [arcsin2] §3.1): the engine runs exactly one
iteration per call; after every iteration the scheduler appends each returned
token to its request, removes the requests that are done (freeing their K/V),
admits waiting ones, and calls the engine again.

Selection ([0h-n0] "スケジューラのアルゴリズム"; [arcsin2] §4.2; [houmin]
3.1.3 "by arrival time"): first-come-first-served under a maximum batch size,
the free K/V capacity (a reservation per admitted request) and, as in
[ultralytics] "制限と併用する手法", a cap on the tokens processed in one step.
Admission stops at the first request that does not fit (the pseudocode's
``break``): later requests never overtake an earlier one.

Readings taken where the pages are silent:

* Candidates are ordered by (arrival, request id).  Under FCFS admission with
  ``break`` every running request arrived no later than any waiting one, so
  running requests come first.  The batch is the longest prefix of that order
  that satisfies: batch size <= max_batch, sum of input rows <= max_tokens,
  and (for a waiting request) a successful K/V reservation.
* A request with output length T finishes after its T-th generated token; the
  initiation iteration (all prompt tokens at once) produces token 1.
* The reservation is ``kv_reserve`` tokens if set, else prompt length + output
  length (Orca's "prompt + maximum generation length" form).  Exactly what was
  reserved is freed.
* The clock counts iterations.  A request with arrival time a can be selected
  at iteration k when a <= k.  An iteration with nothing to run is an idle
  tick: the clock advances and the engine is not called.

Request-level scheduling ([0h-n0] "Request-Level vs Iteration-Level
Scheduling", T_batch = max T_gen; [ultralytics] "リクエスト単位のバッチ処理"):
a batch is formed (same FCFS prefix rule) only when the previous batch has
completely finished, and runs until its longest member is done.  Members that
finish early stop being executed (their slots idle); K/V of the whole batch is
released when it completes.

Cancellation ([houmin] 3.1.1: a request that is done leaves the pool and its
memory is freed at once; the same applies to a request the client drops).
Between iterations a request may be cancelled: it leaves the pool, never runs
again, and its K/V reservation is freed immediately, in either mode.  Its
tokens so far stay readable.  A request-level batch whose remaining members
are all done or cancelled completes at that moment.

Chunked prefill (optional, iteration-level only; a later system's idea that
the pages mention as a contrast: a prompt larger than what is left of an
iteration's token budget is split).  Reading taken: in the FCFS scan, a
request still in its prompt whose remaining prompt exceeds the budget left
takes exactly that budget as a chunk (at least one token) and the scan stops
there; its chunks run in consecutive selections, each with the tokens
processed so far as context; only the iteration that processes the last
prompt token yields a generated token (the engine's output for an earlier
chunk is ignored).  Prompts longer than max_tokens become admissible.

Pipelining ([houmin] 3.1.3, ``n_workers``: while one batch runs, the next is
scheduled; a request whose batch is still running is not selected again, so
the batches in flight are disjoint).  Up to ``n_workers`` selected batches may
be open; completions come oldest first.  The clock advances when a batch is
selected and at an idle tick; an iteration with nothing selectable while
batches are open just waits for the oldest to complete.  With n_workers = 1
this is the plain loop above.
"""

from __future__ import annotations

import bisect
import dataclasses
from typing import Callable, List, Optional, Sequence

from .kv import KVPool


@dataclasses.dataclass
class Req:
    rid: int
    arrival: float
    prompt: List[int]
    out_len: int
    ctx0: int = 0
    ctx: int = 0
    generated: List[int] = dataclasses.field(default_factory=list)
    pending: Optional[int] = None  # input token of the next increment iteration
    kv_off: Optional[int] = None
    state: str = "waiting"  # waiting | running | finished
    admitted_at: Optional[int] = None
    finished_at: Optional[int] = None
    chunk: int = 0  # input rows of the request in the batch being formed
    in_flight: bool = False  # member of an open batch

    @property
    def done(self) -> bool:
        return len(self.generated) >= self.out_len

    @property
    def in_prompt(self) -> bool:
        """Prompt tokens not yet processed remain (never for ctx0 > 0 requests)."""
        return self.ctx0 == 0 and self.ctx < len(self.prompt)

    def n_input(self) -> int:
        """Rows the request needs to finish its current phase in one iteration."""
        return len(self.prompt) - self.ctx if self.in_prompt else 1

    def input_tokens(self) -> List[int]:
        return list(self.prompt[self.ctx:self.ctx + self.chunk]) if self.in_prompt else [self.pending]


@dataclasses.dataclass
class OpenBatch:
    k: int  # the clock at its selection
    batch: List[Req]
    chunks: List[int]
    record: "Iteration" = None


@dataclasses.dataclass
class Iteration:
    """One engine call: the batch descriptor the scheduler hands over."""

    k: int
    rids: List[int]
    phase: List[int]  # 0 = initiation (no cached K/V), 1 = increment
    n_input: List[int]
    ctx: List[int]
    kv_off: List[int]
    tokens: List[int]  # flattened input tokens, request by request

    @property
    def offsets(self) -> List[int]:
        """Exclusive prefix sum of n_input (length B+1): request i owns rows
        offsets[i] .. offsets[i+1]-1 of the flattened [sum L, H] tensor."""
        off = [0]
        for n in self.n_input:
            off.append(off[-1] + n)
        return off


class Scheduler:
    def __init__(self, max_batch: int, max_tokens: int, kv_slots: int, kv_reserve: int = 0,
                 mode: str = "iteration", chunked_prefill: bool = False, n_workers: int = 1):
        if mode not in ("iteration", "request"):
            raise ValueError(mode)
        if chunked_prefill and mode != "iteration":
            raise ValueError("chunked prefill is an iteration-level option")
        if n_workers < 1 or (n_workers > 1 and mode != "iteration"):
            raise ValueError("pipelining is an iteration-level option")
        self.n_workers = n_workers
        self.open: List[OpenBatch] = []  # selected, not yet completed; oldest first
        self.max_batch, self.max_tokens, self.kv_reserve, self.mode = max_batch, max_tokens, kv_reserve, mode
        self.chunked_prefill = chunked_prefill
        self.cancelled_total = 0
        self.pool = KVPool(kv_slots)
        self.reqs: List[Req] = []
        self.k = 0
        self.current_batch: List[Req] = []  # request-level: members of the batch in flight
        self.generated_total = 0
        self.iterations = 0

    # -- request pool ------------------------------------------------------- #
    def reserve_size(self, r: Req) -> int:
        if self.kv_reserve > 0:
            return self.kv_reserve
        return (r.ctx0 if r.ctx0 else len(r.prompt)) + r.out_len

    def submit(self, rid: int, arrival: float, prompt: Sequence[int], out_len: int, ctx0: int = 0) -> Req:
        r = Req(rid, float(arrival), list(prompt), int(out_len), int(ctx0))
        if out_len < 1 or len(r.prompt) < 1:
            raise ValueError("empty request")
        need = (ctx0 + out_len) if ctx0 else (len(r.prompt) + out_len - 1)
        too_long = len(r.prompt) > self.max_tokens and not self.chunked_prefill
        if too_long or need > self.reserve_size(r):
            raise ValueError("request does not fit its reservation or the token budget")
        if ctx0:
            # already in the increment phase: its context is cached, so its
            # reservation is taken now and it runs from the start.
            if len(r.prompt) != 1:
                raise ValueError("a request with cached context has exactly one pending token")
            off = self.pool.alloc(rid, self.reserve_size(r))
            if off is None:
                raise MemoryError("K/V pool full")
            r.kv_off, r.ctx, r.pending, r.state, r.admitted_at = off, ctx0, r.prompt[0], "running", -1
        self.reqs.append(r)
        return r

    def _ordered(self, k: int) -> List[Req]:
        c = [r for r in self.reqs if r.state in ("waiting", "running") and r.arrival <= k and not r.in_flight]
        c.sort(key=lambda r: (r.arrival, r.rid))
        return c

    def _admit_prefix(self, cands: List[Req], k: int) -> List[Req]:
        batch, rows = [], 0
        for r in cands:
            n = r.n_input()
            if len(batch) >= self.max_batch:
                break
            if rows + n > self.max_tokens:
                left = self.max_tokens - rows
                if not (self.chunked_prefill and r.in_prompt and left >= 1):
                    break
                n = left  # a chunk of the prompt; the budget is now used up
            if r.state == "waiting":
                off = self.pool.alloc(r.rid, self.reserve_size(r))
                if off is None:
                    break
                r.kv_off, r.state, r.admitted_at = off, "running", k
            r.chunk = n
            batch.append(r)
            rows += n
        return batch

    def select(self) -> List[Req]:
        """Select the batch of iteration ``self.k``; a non-empty batch is open
        until ``complete`` and advances the clock (empty: nothing selectable)."""
        if len(self.open) >= self.n_workers:
            raise RuntimeError("n_workers batches are open")
        k = self.k
        if self.mode == "iteration":
            batch = self._admit_prefix(self._ordered(k), k)
        else:
            if not self.current_batch:
                self.current_batch = self._admit_prefix([r for r in self._ordered(k) if r.state == "waiting"], k)
            batch = [r for r in self.current_batch if r.state == "running" and not r.done]
            for r in batch:
                r.chunk = r.n_input()
        if batch:
            for r in batch:
                r.in_flight = True
            self.open.append(OpenBatch(k, batch, [r.chunk for r in batch]))
            self.k += 1
        return batch

    def _entry(self, batch: List[Req]) -> OpenBatch:
        for e in self.open:
            if e.batch is batch:
                return e
        raise ValueError("not an open batch")

    def describe(self, batch: List[Req]) -> Iteration:
        e = self._entry(batch)
        toks = []
        for r in batch:
            toks += r.input_tokens()
        e.record = Iteration(e.k, [r.rid for r in batch], [0 if r.ctx == 0 else 1 for r in batch], list(e.chunks),
                             [r.ctx for r in batch], [r.kv_off for r in batch], toks)
        return e.record

    def complete(self, batch: List[Req], next_tokens: Sequence[int]) -> None:
        """Engine returned for the oldest open batch: append tokens, advance
        contexts, retire finished requests."""
        e = self._entry(batch)
        if e is not self.open[0]:
            raise ValueError("batches complete oldest first")
        self.open.pop(0)
        for r, t, n in zip(batch, next_tokens, e.chunks):
            r.in_flight = False
            r.ctx += n
            if r.in_prompt:
                continue  # a prompt chunk before the last: its output is not a token
            r.generated.append(int(t))
            r.pending = int(t)
            self.generated_total += 1
            if r.done:
                r.state, r.finished_at = "finished", e.k
                if self.mode == "iteration":
                    self.pool.free(r.rid)
        self._close_request_batch()
        self.iterations += 1

    def _close_request_batch(self) -> None:
        """Request-level: the batch completes when every member is done or
        cancelled; the reservations still held are released then."""
        if self.mode == "request" and self.current_batch and all(
                r.done or r.state == "cancelled" for r in self.current_batch):
            for r in self.current_batch:
                if r.state != "cancelled":
                    self.pool.free(r.rid)
            self.current_batch = []

    def cancel(self, rid: int) -> None:
        """Drop a waiting or running request between iterations; its K/V is
        freed at once."""
        r = next((q for q in self.reqs if q.rid == rid), None)
        if r is None:
            raise KeyError(rid)
        if r.state not in ("waiting", "running") or (self.mode == "request" and r.done) or r.in_flight:
            raise ValueError("request is not live, or its batch is still open")
        if r.kv_off is not None:
            self.pool.free(r.rid)
        r.state = "cancelled"
        self.cancelled_total += 1
        self._close_request_batch()

    def idle(self) -> None:
        self.k += 1

    def unfinished(self) -> bool:
        return any(r.state in ("waiting", "running") for r in self.reqs)


def run(specs, max_batch: int, max_tokens: int, kv_slots: int, kv_reserve: int = 0, mode: str = "iteration",
        token_fn: Optional[Callable[[Iteration], Sequence[int]]] = None, max_iters: int = 10 ** 7,
        chunked_prefill: bool = False, cancel_at: Optional[dict] = None, n_workers: int = 1):
    """Drive a scheduler over request specs until every request finished.

    ``token_fn(iteration)`` plays the engine and returns one next token per
    request (default: a deterministic dummy).  ``cancel_at`` maps a clock value
    to the request ids cancelled just before a selection at that clock (ids
    that are no longer live, or whose batch is open, are skipped).  With
    ``n_workers`` > 1 up to that many batches are selected before the oldest
    completes.  Returns (scheduler, list of Iteration records, one per engine
    call, in selection order).
    """
    s = Scheduler(max_batch, max_tokens, kv_slots, kv_reserve, mode, chunked_prefill, n_workers)
    for sp in specs:
        s.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len, sp.ctx0)
    if token_fn is None:
        token_fn = lambda it: [(rid * 31 + it.k) % 50000 for rid in it.rids]
    records = []
    while True:
        if len(s.open) < s.n_workers and s.unfinished() and s.k < max_iters:
            for rid in (cancel_at or {}).get(s.k, ()):
                r = next((q for q in s.reqs if q.rid == rid), None)
                if (r is not None and r.state in ("waiting", "running") and not r.in_flight
                        and not (s.mode == "request" and r.done)):
                    s.cancel(rid)
            if s.unfinished():
                batch = s.select()
                if batch:
                    records.append(s.describe(batch))
                    continue
                if not s.open:
                    s.idle()
                    continue
        if not s.open:
            break
        e = s.open[0]
        s.complete(e.batch, token_fn(e.record))
    return s, records


def slots_busy(total_generated: int, iterations: int, slots: int) -> float:
    """[ultralytics] simulation: share of slot-steps that produced a token."""
    return total_generated / (iterations * slots)


# --------------------------------------------------------------------------- #
# closed forms of the pages' slot model (every request present at time 0,
# one token per step per occupied slot)
# --------------------------------------------------------------------------- #
def static_steps(output_lengths: Sequence[int], slots: int) -> int:
    """Request-level: consecutive groups of ``slots`` requests, each group runs
    for its longest member ([0h-n0]: T_batch = max over the batch of T_gen)."""
    total = 0
    for g in range(0, len(output_lengths), slots):
        total += max(output_lengths[g:g + slots])
    return total


def continuous_steps(output_lengths: Sequence[int], slots: int) -> int:
    """Iteration-level: in FCFS order each request starts on the slot that
    becomes free first ([ultralytics] simulation)."""
    free_at = [0] * slots  # kept sorted
    for length in output_lengths:
        start = free_at.pop(0)
        bisect.insort(free_at, start + length)
    return free_at[-1]
