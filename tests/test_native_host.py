"""Host-side parts of liborca.so that need no GPU: the library loads, exports
every function include/orca.h declares, and its C++ scheduler and K/V pool
make exactly the oracle's decisions (bit-exact batches, offsets and slots)."""

import os
import random
import re

import numpy as np
import pytest

from iteration_level_scheduling_gb300 import build, synth
from oracle import sched as osched

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def native():
    build.build()
    from iteration_level_scheduling_gb300 import native as n
    return n


def test_header_symbols_exported(native):
    hdr = open(os.path.join(ROOT, "include", "orca.h")).read()
    declared = sorted(set(re.findall(r"^\s*(?:const\s+)?[\w ]+?\**\s*\b(orca_\w+)\s*\(", hdr, re.M)))
    assert len(declared) >= 20
    for name in declared:
        assert hasattr(native.lib, name), name
    assert set(declared) == set(native.EXPORTS)


def test_strerror(native):
    assert native.lib.orca_strerror(0) == b"ok"
    assert b"K/V" in native.lib.orca_strerror(native.ERR_KV_FULL)


def drive_native(native, specs, max_batch, max_tokens, kv_slots, kv_reserve=0, mode=0, feedback=False):
    s = native.Scheduler(max_batch, max_tokens, kv_slots, kv_reserve, mode, feedback)
    for sp in specs:
        s.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len, sp.ctx0)
    recs = []
    while True:
        clock = s.stats().clock  # the selection's clock (a selection advances it)
        st, b = s.next()
        if st == 2:
            break
        if st == 0:
            continue
        toks = [(int(r) * 31 + clock) % 50000 for r in b.request_id]
        recs.append((clock, b))
        s.complete(toks)
    return s, recs


def drive_oracle(specs, max_batch, max_tokens, kv_slots, kv_reserve=0, mode="iteration"):
    return osched.run(specs, max_batch, max_tokens, kv_slots, kv_reserve, mode,
                      token_fn=lambda it: [(rid * 31 + it.k) % 50000 for rid in it.rids])


def assert_same(native_recs, oracle_recs):
    assert len(native_recs) == len(oracle_recs)
    for (k, b), it in zip(native_recs, oracle_recs):
        assert k == it.k
        assert b.request_id.tolist() == it.rids
        assert b.phase.tolist() == it.phase
        assert b.n_input.tolist() == it.n_input
        assert b.ctx_len.tolist() == it.ctx
        assert b.kv_offset.tolist() == it.kv_off
        assert b.tokens.tolist() == it.tokens


@pytest.mark.parametrize("mode", [0, 1])
def test_worked_example_native(native, mode):
    outs = [5, 50, 8, 12, 40, 3, 30, 7]
    specs = [synth.RequestSpec(i, 0.0, [1, 2], L) for i, L in enumerate(outs)]
    s, recs = drive_native(native, specs, 4, 4096, 10 ** 6, mode=mode)
    assert len(recs) == (50 if mode == 0 else 90)
    st = s.stats()
    assert st.generated == sum(outs) and st.finished == 8 and st.kv_reserved == 0
    _, orecs = drive_oracle(specs, 4, 4096, 10 ** 6, mode="iteration" if mode == 0 else "request")
    assert_same(recs, orecs)


@pytest.mark.parametrize("seed", range(5))
def test_native_matches_oracle_random_traces(native, seed):
    rnd = random.Random(100 + seed)
    trace = synth.poisson_trace(seed, n=80, rate=rnd.choice([0.1, 0.5, 3.0]), prompt_range=(1, 60),
                                out_range=(1, 40), vocab=1000)
    mb, mt = rnd.randint(1, 16), rnd.randint(60, 300)
    slots = rnd.randint(100, 1500)
    reserve = rnd.choice([0, 0, 100])
    for mode in (0, 1):
        s, recs = drive_native(native, trace, mb, mt, slots, reserve, mode)
        _, orecs = drive_oracle(trace, mb, mt, slots, reserve, "iteration" if mode == 0 else "request")
        assert_same(recs, orecs)
        for sp in trace:
            r = s.request(sp.rid)
            assert r.state == 2 and r.n_generated == sp.out_len


def test_native_cfg3_trace_prefix(native):
    """The 13B continuous-batching trace: 1000 requests, 64 x 1024-token reservations."""
    trace = synth.poisson_trace(0, n=1000, rate=0.5, with_tokens=False)
    s, recs = drive_native(native, trace, 64, 4096, 64 * 1024, kv_reserve=1024)
    _, orecs = drive_oracle(trace, 64, 4096, 64 * 1024, kv_reserve=1024)
    assert_same(recs, orecs)
    assert max(len(b.request_id) for _, b in recs) == 64


def test_cached_context_requests_and_kv_full(native):
    s = native.Scheduler(8, 4096, kv_slots=1000, kv_reserve=300)
    assert s.submit(0, 0.0, [5], 10, ctx0=200) == 0
    assert s.submit(1, 0.0, [6], 10, ctx0=250) == 300
    assert s.submit(2, 0.0, [7], 10, ctx0=100) == 600
    with pytest.raises(native.OrcaError) as e:
        s.submit(3, 0.0, [8], 10, ctx0=100)
    assert e.value.code == native.ERR_KV_FULL
    with pytest.raises(native.OrcaError):
        s.submit(4, 0.0, [1] * 295, 10)  # 295 + 10 - 1 > 300
    st, b = s.next()
    assert st == 1 and b.phase.tolist() == [1, 1, 1] and b.ctx_len.tolist() == [200, 250, 100]
    assert b.tokens.tolist() == [5, 6, 7]


def test_token_feedback_references(native):
    s = native.Scheduler(4, 4096, kv_slots=100, token_feedback=True)
    s.submit(0, 0.0, [1, 2, 3], 3)
    s.submit(1, 1.0, [4], 3)
    st, b = s.next()
    assert b.tokens.tolist() == [1, 2, 3]
    s.complete([9])
    st, b = s.next()
    # request 0 was index 0 of the previous iteration -> -1; request 1 is new
    assert b.request_id.tolist() == [0, 1] and b.tokens.tolist() == [-1, 4]
    s.complete([10, 11])
    st, b = s.next()
    assert b.tokens.tolist() == [-1, -2]
    assert s.tokens(0).tolist() == [9, 10]


def test_token_feedback_enabled_midway(native):
    s = native.Scheduler(4, 4096, kv_slots=100)
    s.submit(0, 0.0, [1, 2], 5)
    st, b = s.next()
    s.complete([7])
    s.set_token_feedback(True)
    st, b = s.next()
    assert b.tokens.tolist() == [7]  # the previous iteration ran without feedback: literal token
    s.complete([8])
    st, b = s.next()
    assert b.tokens.tolist() == [-1]


def drive_native_ext(native, specs, max_batch, max_tokens, kv_slots, mode=0, chunked=False, cancel_at=None):
    """drive_native with chunked prefill and cancellations before selections."""
    s = native.Scheduler(max_batch, max_tokens, kv_slots, 0, mode, False, chunked_prefill=chunked)
    for sp in specs:
        s.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len, sp.ctx0)
    recs = []
    while True:
        for rid in (cancel_at or {}).get(s.stats().clock, ()):
            info = s.request(rid)
            live = info.state in (0, 1) and not (mode == 1 and info.n_generated >= specs[rid].out_len)
            if live:
                s.cancel(rid)
        clock = s.stats().clock
        st, b = s.next()
        if st == 2:
            break
        if st == 0:
            continue
        toks = [(int(r) * 31 + clock) % 50000 for r in b.request_id]
        recs.append((clock, b))
        s.complete(toks)
    return s, recs


@pytest.mark.parametrize("seed", range(4))
def test_native_matches_oracle_chunked_prefill(native, seed):
    rnd = random.Random(300 + seed)
    mt = rnd.randint(8, 80)
    trace = synth.poisson_trace(seed, n=60, rate=rnd.choice([0.3, 1.0, 3.0]), prompt_range=(1, 3 * mt),
                                out_range=(1, 30), vocab=1000)
    mb = rnd.randint(1, 8)
    s, recs = drive_native_ext(native, trace, mb, mt, 10 ** 5, chunked=True)
    _, orecs = osched.run(trace, mb, mt, 10 ** 5, chunked_prefill=True,
                          token_fn=lambda it: [(rid * 31 + it.k) % 50000 for rid in it.rids])
    assert_same(recs, orecs)
    assert any(n > 1 and c > 0 for _, b in recs for n, c in zip(b.n_input.tolist(), b.ctx_len.tolist()))
    for sp in trace:
        assert s.request(sp.rid).n_generated == sp.out_len


@pytest.mark.parametrize("seed", range(4))
def test_native_matches_oracle_cancellation(native, seed):
    rnd = random.Random(400 + seed)
    trace = synth.poisson_trace(seed, n=60, rate=rnd.choice([0.3, 1.0, 3.0]), prompt_range=(1, 40),
                                out_range=(1, 30), vocab=1000)
    cancel_at = {}
    for sp in rnd.sample(trace, 20):
        cancel_at.setdefault(rnd.randint(0, 80), []).append(sp.rid)
    mb, mt = rnd.randint(1, 8), rnd.randint(40, 200)
    for mode in (0, 1):
        s, recs = drive_native_ext(native, trace, mb, mt, 3000, mode=mode, cancel_at=cancel_at)
        o, orecs = osched.run(trace, mb, mt, 3000, 0, "iteration" if mode == 0 else "request",
                              token_fn=lambda it: [(rid * 31 + it.k) % 50000 for rid in it.rids],
                              cancel_at=cancel_at)
        assert_same(recs, orecs)
        st = s.stats()
        assert st.cancelled == o.cancelled_total >= 1 and st.kv_reserved == 0
        for r in o.reqs:
            info = s.request(r.rid)
            assert info.state == {"finished": 2, "cancelled": 3}[r.state]
            assert s.tokens(r.rid).tolist() == r.generated


def test_cancel_errors(native):
    s = native.Scheduler(2, 4096, kv_slots=100)
    s.submit(0, 0.0, [1, 2], 3)
    s.submit(1, 0.0, [3], 3)
    with pytest.raises(native.OrcaError) as e:
        s.cancel(7)
    assert e.value.code == native.ERR_NOT_FOUND
    st, b = s.next()
    with pytest.raises(native.OrcaError) as e:  # a batch is open
        s.cancel(0)
    assert e.value.code == native.ERR_INVALID
    s.complete([5, 6])
    assert s.stats().kv_reserved == (2 + 3) + (1 + 3)
    s.cancel(0)
    assert s.stats().kv_reserved == 1 + 3 and s.request(0).state == 3
    with pytest.raises(native.OrcaError):
        s.cancel(0)                              # already cancelled
    assert s.tokens(0).tolist() == [5]
    with pytest.raises(native.OrcaError):        # chunked prefill is an iteration-level option
        native.Scheduler(2, 4096, kv_slots=100, mode=1, chunked_prefill=True)


def drive_native_pipelined(native, specs, max_batch, max_tokens, kv_slots, n_workers):
    s = native.Scheduler(max_batch, max_tokens, kv_slots, 0, 0, False, n_workers=n_workers)
    for sp in specs:
        s.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len, sp.ctx0)
    recs, queue = [], []
    while True:
        while len(queue) < n_workers:
            clock = s.stats().clock
            st, b = s.next()
            if st == 1:
                queue.append((clock, b))
                recs.append((clock, b))
                continue
            if st == 0:
                continue
            break
        if not queue:
            break
        clock, b = queue.pop(0)
        s.complete([(int(r) * 31 + clock) % 50000 for r in b.request_id])
    return s, recs


@pytest.mark.parametrize("seed", range(4))
def test_native_matches_oracle_pipelined(native, seed):
    rnd = random.Random(500 + seed)
    trace = synth.poisson_trace(seed, n=60, rate=rnd.choice([0.3, 1.0, 3.0]), prompt_range=(1, 40),
                                out_range=(1, 30), vocab=1000)
    mb, mt = rnd.randint(1, 8), rnd.randint(40, 200)
    for nw in (2, 3):
        s, recs = drive_native_pipelined(native, trace, mb, mt, 5000, nw)
        _, orecs = osched.run(trace, mb, mt, 5000, n_workers=nw,
                              token_fn=lambda it: [(rid * 31 + it.k) % 50000 for rid in it.rids])
        assert_same(recs, orecs)
        assert s.stats().kv_reserved == 0


def test_pipelined_protocol(native):
    s = native.Scheduler(1, 4096, kv_slots=100, n_workers=2)
    s.submit(0, 0.0, [1], 2)
    s.submit(1, 0.0, [2], 2)
    st, b = s.next()
    assert st == 1 and b.request_id.tolist() == [0]
    st, b = s.next()
    assert st == 1 and b.request_id.tolist() == [1]
    with pytest.raises(native.OrcaError):  # two batches already open
        s.next()
    s.complete([5])                         # completes the oldest: request 0
    assert s.tokens(0).tolist() == [5] and s.tokens(1).tolist() == []
    st, b = s.next()
    assert st == 1 and b.request_id.tolist() == [0] and b.tokens.tolist() == [5]
    with pytest.raises(native.OrcaError):   # request 1's batch is still open
        s.cancel(1)
    for bad in (dict(mode=1), dict(token_feedback=True)):
        with pytest.raises(native.OrcaError):
            native.Scheduler(2, 4096, kv_slots=100, n_workers=2, **bad)


def faulty_oracle_pool(monkeypatch, n):
    """The oracle's pool with its n-th reservation failing as if full (the
    oracle side of ORCA_FAULT=kv_alloc:n)."""
    from oracle import kv as okv
    orig = okv.KVPool.alloc

    def alloc(self, rid, n_tokens):
        if n_tokens <= 0 or rid in self.owned:
            return orig(self, rid, n_tokens)
        self._calls = getattr(self, "_calls", 0) + 1
        return None if self._calls == n else orig(self, rid, n_tokens)

    monkeypatch.setattr(okv.KVPool, "alloc", alloc)


@pytest.mark.parametrize("nth", [1, 3, 9, 25])
def test_injected_kv_alloc_failure_keeps_scheduler_consistent(native, monkeypatch, nth):
    """ORCA_FAULT=kv_alloc:N makes the N-th K/V reservation fail as if the pool
    were full ([0h-n0] scheduler algorithm: admission stops when K/V runs out).
    The scheduler must stall that admission and retry it later exactly as the
    oracle does under the same failure: identical batches, offsets and slots,
    every request finished, every reservation returned."""
    trace = synth.poisson_trace(40 + nth, n=60, rate=1.5, prompt_range=(1, 40), out_range=(1, 20), vocab=1000)
    clean_native = drive_native(native, trace, 6, 200, 6 * 64, kv_reserve=64)[1]
    monkeypatch.setenv("ORCA_FAULT", f"kv_alloc:{nth}")
    s, recs = drive_native(native, trace, 6, 200, 6 * 64, kv_reserve=64)
    monkeypatch.delenv("ORCA_FAULT")
    faulty_oracle_pool(monkeypatch, nth)
    _, orecs = drive_oracle(trace, 6, 200, 6 * 64, kv_reserve=64)
    assert_same(recs, orecs)
    # the fault changed the schedule (the failed admission waited)
    assert [(k, b.request_id.tolist()) for k, b in recs] != [(k, b.request_id.tolist()) for k, b in clean_native]
    st = s.stats()
    assert st.finished == len(trace) and st.kv_reserved == 0
    for sp in trace:
        assert s.request(sp.rid).n_generated == sp.out_len


def test_fault_injection_reads_only_its_point(native, monkeypatch):
    """Other entries in ORCA_FAULT, or none, leave the pool alone."""
    monkeypatch.setenv("ORCA_FAULT", "plan_h2d:1,kv_allocx:1")
    s = native.Scheduler(2, 100, kv_slots=100)
    assert s.submit(0, 0.0, [1], 5, ctx0=3) == 0
    monkeypatch.setenv("ORCA_FAULT", "other:4,kv_alloc:1")
    s2 = native.Scheduler(2, 100, kv_slots=100)
    with pytest.raises(native.OrcaError) as e:
        s2.submit(0, 0.0, [1], 5, ctx0=3)
    assert e.value.code == native.ERR_KV_FULL
    assert s2.submit(1, 0.0, [1], 5, ctx0=3) == 0  # only the first call fails
