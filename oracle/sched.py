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

    @property
    def done(self) -> bool:
        return len(self.generated) >= self.out_len

    def n_input(self) -> int:
        return len(self.prompt) if self.ctx == 0 else 1

    def input_tokens(self) -> List[int]:
        return list(self.prompt) if self.ctx == 0 else [self.pending]


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
                 mode: str = "iteration"):
        if mode not in ("iteration", "request"):
            raise ValueError(mode)
        self.max_batch, self.max_tokens, self.kv_reserve, self.mode = max_batch, max_tokens, kv_reserve, mode
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
        if len(r.prompt) > self.max_tokens or need > self.reserve_size(r):
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
        c = [r for r in self.reqs if r.state != "finished" and r.arrival <= k]
        c.sort(key=lambda r: (r.arrival, r.rid))
        return c

    def _admit_prefix(self, cands: List[Req], k: int) -> List[Req]:
        batch, rows = [], 0
        for r in cands:
            n = r.n_input()
            if len(batch) >= self.max_batch or rows + n > self.max_tokens:
                break
            if r.state == "waiting":
                off = self.pool.alloc(r.rid, self.reserve_size(r))
                if off is None:
                    break
                r.kv_off, r.state, r.admitted_at = off, "running", k
            batch.append(r)
            rows += n
        return batch

    def select(self) -> List[Req]:
        """Batch for the current iteration ``self.k`` (empty = idle tick)."""
        k = self.k
        if self.mode == "iteration":
            return self._admit_prefix(self._ordered(k), k)
        if not self.current_batch:
            self.current_batch = self._admit_prefix([r for r in self._ordered(k) if r.state == "waiting"], k)
        return [r for r in self.current_batch if not r.done]

    def describe(self, batch: List[Req]) -> Iteration:
        toks = []
        for r in batch:
            toks += r.input_tokens()
        return Iteration(self.k, [r.rid for r in batch], [0 if r.ctx == 0 else 1 for r in batch],
                         [r.n_input() for r in batch], [r.ctx for r in batch], [r.kv_off for r in batch], toks)

    def complete(self, batch: List[Req], next_tokens: Sequence[int]) -> None:
        """Engine returned: append tokens, advance contexts, retire finished requests."""
        for r, t in zip(batch, next_tokens):
            r.ctx += r.n_input()
            r.generated.append(int(t))
            r.pending = int(t)
            self.generated_total += 1
            if r.done:
                r.state, r.finished_at = "finished", self.k
                if self.mode == "iteration":
                    self.pool.free(r.rid)
        if self.mode == "request" and all(r.done for r in self.current_batch):
            for r in self.current_batch:
                self.pool.free(r.rid)
            self.current_batch = []
        self.iterations += 1
        self.k += 1

    def idle(self) -> None:
        self.k += 1

    def unfinished(self) -> bool:
        return any(r.state != "finished" for r in self.reqs)


def run(specs, max_batch: int, max_tokens: int, kv_slots: int, kv_reserve: int = 0, mode: str = "iteration",
        token_fn: Optional[Callable[[Iteration], Sequence[int]]] = None, max_iters: int = 10 ** 7):
    """Drive a scheduler over request specs until every request finished.

    ``token_fn(iteration)`` plays the engine and returns one next token per
    request (default: a deterministic dummy).  Returns (scheduler, list of
    Iteration records, one per engine call).
    """
    s = Scheduler(max_batch, max_tokens, kv_slots, kv_reserve, mode)
    for sp in specs:
        s.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len, sp.ctx0)
    if token_fn is None:
        token_fn = lambda it: [(rid * 31 + it.k) % 50000 for rid in it.rids]
    records = []
    while s.unfinished() and s.k < max_iters:
        batch = s.select()
        if not batch:
            s.idle()
            continue
        it = s.describe(batch)
        records.append(it)
        s.complete(batch, token_fn(it))
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
