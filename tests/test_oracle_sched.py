"""Pins of the scheduler / K/V-pool oracle against what the pages print."""

import json
import os
import random

import pytest

from oracle import sched
from oracle.kv import KVPool
from iteration_level_scheduling_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def specs_from_lengths(lengths, prompt_len=1):
    return [synth.RequestSpec(i, 0.0, [1] * prompt_len, L) for i, L in enumerate(lengths)]


# --------------------------------------------------------------------------- #
# [ultralytics] worked simulation: 90 / 50 steps, 43% / 78% busy
# --------------------------------------------------------------------------- #
def test_worked_example_closed_forms():
    g = load("ultralytics_slot_simulation.json")
    outs, S = g["output_lengths"], g["slots"]
    assert sched.static_steps(outs, S) == g["static_steps"]
    assert sched.continuous_steps(outs, S) == g["continuous_steps"]
    assert f"{sched.slots_busy(sum(outs), g['static_steps'], S):.0%}" == g["static_slots_busy"]
    assert f"{sched.slots_busy(sum(outs), g['continuous_steps'], S):.0%}" == g["continuous_slots_busy"]


@pytest.mark.parametrize("mode,key", [("iteration", "continuous"), ("request", "static")])
def test_worked_example_schedulers(mode, key):
    g = load("ultralytics_slot_simulation.json")
    outs, S = g["output_lengths"], g["slots"]
    s, recs = sched.run(specs_from_lengths(outs), max_batch=S, max_tokens=4096, kv_slots=10 ** 6, mode=mode)
    assert len(recs) == g[f"{key}_steps"]
    assert s.generated_total == sum(outs)
    assert f"{sched.slots_busy(s.generated_total, len(recs), S):.0%}" == g[f"{key}_slots_busy"]
    assert all(len(r.rids) <= S for r in recs)


def test_worked_example_with_prompts():
    """Prompt lengths do not change the step counts (one token per iteration)."""
    g = load("ultralytics_slot_simulation.json")
    reqs = synth.tiny_requests(0)
    assert [r.out_len for r in reqs] == g["output_lengths"]
    s, recs = sched.run(reqs, max_batch=4, max_tokens=4096, kv_slots=4 * 128)
    assert len(recs) == 50
    s, recs = sched.run(reqs, max_batch=4, max_tokens=4096, kv_slots=4 * 128, mode="request")
    assert len(recs) == 90


def test_closed_form_equals_scheduler_random():
    """With every request present at time 0 the iteration-level scheduler is the
    slot model of the closed form; the request-level one is the group model."""
    rnd = random.Random(5)
    for _ in range(200):
        n = rnd.randint(1, 14)
        S = rnd.randint(1, 5)
        outs = [rnd.randint(1, 30) for _ in range(n)]
        _, recs = sched.run(specs_from_lengths(outs), S, 4096, 10 ** 6)
        assert len(recs) == sched.continuous_steps(outs, S)
        _, recs = sched.run(specs_from_lengths(outs), S, 4096, 10 ** 6, mode="request")
        assert len(recs) == sched.static_steps(outs, S)


# --------------------------------------------------------------------------- #
# [estelledc] case 1: D joins at step 11, E at 51, F at 101
# --------------------------------------------------------------------------- #
def test_case1_join_steps():
    g = load("estelledc_case1.json")
    first = g["first_requests"]
    names = list(first) + list(g["continuous_join_step_1_indexed"])
    outs = [first["A"], first["B"], first["C"], 500, 500, 500]
    s, recs = sched.run(specs_from_lengths(outs), g["slots"], 4096, 10 ** 6, token_fn=lambda it: [0] * len(it.rids))
    by_id = {r.rid: r for r in s.reqs}
    for j, name in enumerate(names[3:]):
        assert by_id[3 + j].admitted_at + 1 == g["continuous_join_step_1_indexed"][name]
    for rec in recs[:100]:
        assert len(rec.rids) == 3  # the batch never has an idle slot


def test_case1_static_phases():
    g = load("estelledc_case1.json")
    first = g["first_requests"]
    _, recs = sched.run(specs_from_lengths([first["A"], first["B"], first["C"]]), 3, 4096, 10 ** 6, mode="request")
    names = {0: "A", 1: "B", 2: "C"}
    for lo, hi, members in g["static_phases_1_indexed"]:
        for step in range(lo, hi + 1):
            assert sorted(names[r] for r in recs[step - 1].rids) == sorted(members)
    assert len(recs) == 100


# --------------------------------------------------------------------------- #
# [houmin] the (x1, x2, x3, x4) batch: 7 flattened rows
# --------------------------------------------------------------------------- #
def test_houmin_batch_descriptor():
    g = load("houmin_selective_batch.json")
    specs = [synth.RequestSpec(1, 0.0, [11, 12], 10), synth.RequestSpec(2, 1.0, [21], 10),
             synth.RequestSpec(3, 2.0, [31, 32], 10), synth.RequestSpec(4, 2.0, [41, 42, 43], 10)]
    s, recs = sched.run(specs, 4, 4096, 10 ** 6, token_fn=lambda it: [0] * len(it.rids), max_iters=3)
    it = recs[2]
    assert it.rids == [1, 2, 3, 4]
    assert it.phase == [1, 1, 0, 0]
    assert it.n_input == [1, 1, 2, 3]
    assert it.offsets[-1] == g["rows_batch"]
    assert it.offsets[4] - it.offsets[2] == g["rows_x3_x4"]
    by = {r.rid: r for r in s.reqs}
    # token index of the token each request returns at this iteration
    for name, idx in g["returned_token_index"].items():
        r = by[int(name[1])]
        assert len(r.prompt) + len(r.generated) == idx


# --------------------------------------------------------------------------- #
# [0h-n0] admission pseudocode: reservation, stall when full, no overtaking
# --------------------------------------------------------------------------- #
def test_kv_full_stall_and_fcfs():
    # pool of 100 tokens; each request reserves prompt + output
    specs = [synth.RequestSpec(0, 0.0, [1] * 10, 50),  # 60
             synth.RequestSpec(1, 0.0, [1] * 10, 40),  # 50 -> does not fit beside 60
             synth.RequestSpec(2, 0.0, [1] * 5, 5)]    # 10 -> would fit, but must not overtake
    s, recs = sched.run(specs, 8, 4096, 100)
    assert recs[0].rids == [0]
    by = {r.rid: r for r in s.reqs}
    assert by[1].admitted_at == by[0].finished_at + 1
    assert by[2].admitted_at == by[1].admitted_at
    assert by[1].kv_off == 0 and by[2].kv_off == 50


def test_token_budget():
    specs = [synth.RequestSpec(i, 0.0, [1] * 30, 3) for i in range(5)]
    s, recs = sched.run(specs, 8, 64, 10 ** 6)
    assert recs[0].rids == [0, 1] and sum(recs[0].n_input) == 60
    for r in recs:
        assert sum(r.n_input) <= 64


def test_invariants_random_traces():
    for seed in range(6):
        rnd = random.Random(seed)
        trace = synth.poisson_trace(seed, n=60, rate=rnd.choice([0.2, 0.5, 2.0]), prompt_range=(1, 40),
                                    out_range=(1, 30), vocab=100)
        max_batch, max_tokens, slots = rnd.randint(1, 8), rnd.randint(40, 200), rnd.randint(80, 400)
        s, recs = sched.run(trace, max_batch, max_tokens, slots)
        admitted = sorted((r for r in s.reqs), key=lambda r: (r.admitted_at, r.arrival, r.rid))
        order = sorted(s.reqs, key=lambda r: (r.arrival, r.rid))
        assert [r.rid for r in admitted] == [r.rid for r in order]  # FCFS, never overtaken
        live = {}
        for rec in recs:
            assert 1 <= len(rec.rids) <= max_batch
            assert sum(rec.n_input) <= max_tokens
            for rid, ph, n, c in zip(rec.rids, rec.phase, rec.n_input, rec.ctx):
                assert (ph == 0) == (c == 0)
        # reservations never overlap and stay inside the pool
        for r in s.reqs:
            assert r.state == "finished" and len(r.generated) == r.out_len
        assert s.pool.used() == 0 and s.pool.free_list == [(0, slots)]
        # replay the reservation intervals per iteration
        for rec in recs:
            iv = sorted(zip(rec.kv_off, [s.reserve_size(r) for r in (next(q for q in s.reqs if q.rid == x) for x in rec.rids)]))
            for (o1, l1), (o2, _) in zip(iv, iv[1:]):
                assert o1 + l1 <= o2
            assert all(o + l <= slots for o, l in iv)


# --------------------------------------------------------------------------- #
# K/V pool: first fit at the lowest address, coalescing frees
# --------------------------------------------------------------------------- #
def test_kv_pool_script():
    p = KVPool(100)
    assert p.alloc(1, 30) == 0
    assert p.alloc(2, 30) == 30
    assert p.alloc(3, 30) == 60
    assert p.alloc(4, 20) is None
    p.free(2)
    assert p.alloc(5, 10) == 30  # first fit in the hole
    assert p.alloc(6, 25) is None  # hole left is 20, tail is 10
    assert p.alloc(7, 20) == 40
    assert p.alloc(8, 10) == 90
    p.free(1)
    p.free(5)
    assert p.free_list == [(0, 40)]  # merged across the freed neighbours
    p.free(7)
    p.free(3)
    p.free(8)
    assert p.free_list == [(0, 100)] and p.used() == 0


def test_kv_pool_random_no_overlap():
    rnd = random.Random(1)
    p = KVPool(500)
    live = {}
    for step in range(3000):
        if live and rnd.random() < 0.45:
            rid = rnd.choice(sorted(live))
            p.free(rid)
            del live[rid]
        else:
            rid = step
            n = rnd.randint(1, 80)
            off = p.alloc(rid, n)
            # brute force: the lowest offset where n slots are free
            busy = [False] * 500
            for o, l in live.values():
                for t in range(o, o + l):
                    busy[t] = True
            expect = next((o for o in range(500 - n + 1) if not any(busy[o:o + n])), None)
            assert off == expect
            if off is not None:
                live[rid] = (off, n)
        assert p.used() == sum(l for _, l in live.values())
        assert sum(l for _, l in p.free_list) == 500 - p.used()


# --------------------------------------------------------------------------- #
# cancellation: the request leaves the pool and its K/V is freed at once
# --------------------------------------------------------------------------- #
def test_cancel_worked_example_iteration_level():
    # pool 100, reservations prompt + output: A 2+10 = 12 at 0, B 2+10 at 12, C 2+10 waits (max_batch 2)
    specs = [synth.RequestSpec(i, 0.0, [1, 2], 10) for i in range(3)]
    s = sched.Scheduler(2, 4096, 100)
    for sp in specs:
        s.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len)
    b = s.select()
    assert [r.rid for r in b] == [0, 1] and s.pool.used() == 24
    s.complete(b, [7, 8])
    s.cancel(1)                      # between iterations: B's 12 slots come back at once
    assert s.pool.used() == 12 and s.cancelled_total == 1
    b = s.select()                   # C takes the freed place (first fit: B's old offset)
    assert [r.rid for r in b] == [0, 2]
    by = {r.rid: r for r in s.reqs}
    assert by[2].kv_off == 12 and by[1].state == "cancelled" and by[1].generated == [8]
    with pytest.raises(ValueError):
        s.cancel(1)                  # not live any more
    with pytest.raises(KeyError):
        s.cancel(9)


def test_cancel_worked_example_request_level():
    specs = [synth.RequestSpec(i, 0.0, [1], L) for i, L in enumerate([2, 5, 3])]
    s = sched.Scheduler(2, 4096, 100, mode="request")
    for sp in specs:
        s.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len)
    b = s.select()
    s.complete(b, [1, 1])
    s.cancel(1)                      # immediate release even in request-level mode
    assert s.pool.used() == 1 + 2    # request 0 (1 + 2) keeps its reservation until the batch completes
    b = s.select()
    assert [r.rid for r in b] == [0]
    s.complete(b, [1])               # request 0 done: the batch (0, cancelled 1) completes
    assert s.pool.used() == 0 and s.current_batch == []
    b = s.select()
    assert [r.rid for r in b] == [2]


def test_cancel_invariants_random_traces():
    for seed in range(6):
        rnd = random.Random(50 + seed)
        trace = synth.poisson_trace(seed, n=50, rate=rnd.choice([0.3, 1.0, 3.0]), prompt_range=(1, 30),
                                    out_range=(1, 25), vocab=100)
        cancel_at = {}
        for sp in rnd.sample(trace, 15):
            cancel_at.setdefault(rnd.randint(0, 60), []).append(sp.rid)
        for mode in ("iteration", "request"):
            s, recs = sched.run(trace, rnd.randint(1, 6), rnd.randint(30, 120), 2000, 0, mode, cancel_at=cancel_at)
            gone = {}
            for r in s.reqs:
                if r.state == "cancelled":
                    gone[r.rid] = r
            assert s.cancelled_total == len(gone) >= 1
            for rec in recs:  # a cancelled request never runs after its cancellation
                for rid in rec.rids:
                    if rid in gone:
                        t = min(k for k, ids in cancel_at.items() if rid in ids)
                        assert rec.k < t
            for r in s.reqs:
                assert r.state in ("finished", "cancelled")
                if r.state == "finished":
                    assert len(r.generated) == r.out_len
                else:
                    assert len(r.generated) < r.out_len
            assert s.pool.used() == 0 and s.pool.free_list == [(0, 2000)]


# --------------------------------------------------------------------------- #
# chunked prefill: a prompt larger than the budget left runs in chunks
# --------------------------------------------------------------------------- #
def test_chunked_prefill_worked_example():
    a = synth.RequestSpec(0, 0.0, list(range(100, 110)), 2)   # prompt 10
    b = synth.RequestSpec(1, 0.0, [7, 8, 9], 2)                # prompt 3
    with pytest.raises(ValueError):
        sched.run([a, b], 4, 8, 100)                           # 10 > max_tokens without chunking
    s, recs = sched.run([a, b], 4, 8, 100, chunked_prefill=True)
    assert [(r.rids, r.n_input, r.ctx, r.phase) for r in recs] == [
        ([0], [8], [0], [0]),             # A's first 8 prompt tokens use the whole budget; B waits
        ([0, 1], [2, 3], [8, 0], [1, 0]),  # A's last 2 prompt tokens (8 cached), B's prompt
        ([0, 1], [1, 1], [10, 3], [1, 1]),
    ]
    assert recs[0].tokens == list(range(100, 108))
    assert recs[1].tokens == [108, 109, 7, 8, 9]
    by = {r.rid: r for r in s.reqs}
    # A's first token comes from the iteration that processed its last prompt token
    assert by[0].generated == [(0 * 31 + 1) % 50000, (0 * 31 + 2) % 50000]
    assert by[1].generated == [(1 * 31 + 1) % 50000, (1 * 31 + 2) % 50000]


def test_chunked_prefill_invariants_random_traces():
    for seed in range(6):
        rnd = random.Random(70 + seed)
        mt = rnd.randint(8, 60)
        trace = synth.poisson_trace(seed, n=40, rate=rnd.choice([0.3, 1.0, 3.0]), prompt_range=(1, 3 * mt),
                                    out_range=(1, 20), vocab=1000)
        s, recs = sched.run(trace, rnd.randint(1, 6), mt, 10 ** 5, chunked_prefill=True)
        fed = {sp.rid: [] for sp in trace}
        first_token_at = {}
        for rec in recs:
            assert sum(rec.n_input) <= mt
            p = 0
            for rid, ph, n, c in zip(rec.rids, rec.phase, rec.n_input, rec.ctx):
                assert (ph == 0) == (c == 0)
                spec = trace[rid]
                if c < len(spec.prompt):  # a prompt chunk: the next unprocessed tokens, in order
                    assert c == len(fed[rid])
                    fed[rid] += rec.tokens[p:p + n]
                    if c + n == len(spec.prompt):
                        first_token_at[rid] = rec.k
                else:
                    assert n == 1
                p += n
        for sp in trace:
            assert fed[sp.rid] == list(sp.prompt)
        for r in s.reqs:
            assert r.state == "finished" and len(r.generated) == r.out_len
            assert r.generated[0] == (r.rid * 31 + first_token_at[r.rid]) % 50000
        assert s.pool.used() == 0


# --------------------------------------------------------------------------- #
# pipelining ([houmin] 3.1.3 n_workers): open batches are disjoint
# --------------------------------------------------------------------------- #
def test_pipelined_worked_example():
    specs = [synth.RequestSpec(i, 0.0, [1], L) for i, L in enumerate([2, 2, 1, 3])]
    s, recs = sched.run(specs, 2, 4096, 100, n_workers=2)
    assert [(r.k, r.rids, r.ctx) for r in recs] == [
        (0, [0, 1], [0, 0]),   # A
        (1, [2, 3], [0, 0]),   # B, selected while A runs: 0 and 1 are in flight
        (2, [0, 1], [1, 1]),   # after A completed
        (3, [3], [1]),         # after B completed (2 finished); 0, 1 in flight
        (4, [3], [2]),         # nothing else selectable at clock 4 until the previous batch completed
    ]
    assert all(len(r.generated) == r.out_len for r in s.reqs) and s.pool.used() == 0


def test_pipelined_invariants_random_traces():
    for seed in range(6):
        rnd = random.Random(90 + seed)
        trace = synth.poisson_trace(seed, n=60, rate=rnd.choice([0.3, 1.0, 3.0]), prompt_range=(1, 40),
                                    out_range=(1, 30), vocab=100)
        mb, mt = rnd.randint(1, 8), rnd.randint(40, 200)
        s1, r1 = sched.run(trace, mb, mt, 5000)
        s1b, r1b = sched.run(trace, mb, mt, 5000, n_workers=1)
        assert [vars(a) for a in r1] == [vars(b) for b in r1b]  # one worker is the plain loop
        for nw in (2, 3):
            s = sched.Scheduler(mb, mt, 5000, n_workers=nw)
            for sp in trace:
                s.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len)
            recs, most_open = [], 0
            while True:
                if len(s.open) < nw and s.unfinished():
                    open_ids = [{r.rid for r in e.batch} for e in s.open]
                    batch = s.select()
                    if batch:  # a new batch shares no request with the batches still open
                        assert all(not ({r.rid for r in batch} & o) for o in open_ids)
                        recs.append(s.describe(batch))
                        most_open = max(most_open, len(s.open))
                        continue
                    if not s.open:
                        s.idle()
                        continue
                if not s.open:
                    break
                e = s.open[0]
                s.complete(e.batch, [7] * len(e.batch))
            assert most_open == nw
            for r in s.reqs:
                assert r.state == "finished" and len(r.generated) == r.out_len
            assert s.pool.used() == 0
            assert sum(len(r.rids) for r in recs) == sum(sp.out_len for sp in trace)
