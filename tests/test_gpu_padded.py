"""The conventional padded + masked batch on the GPU (the request-level
baseline Orca is compared with: [houmin] 3.1.2 "问题", [arcsin2] 3.2,
[0h-n0] "Request-Level vs Iteration-Level Scheduling").

A request-level batch runs through orca_run_iteration_padded: every request
padded to the batch's longest input with token 0, the increment phase
attending over the batch's longest key range with each request's keys past its
own context masked, and members that have finished kept in the batch as
single-row requests on token 0 until the longest member is done.  Teacher
forced, every iteration's real requests must match the oracle's padded +
masked computation (oracle/padded.py), which itself equals selective batching.
"""

import numpy as np
import pytest

from iteration_level_scheduling_gb300 import synth
from oracle import padded as opadded
from oracle import sched as osched
from oracle.model import BatchItem, KVStore
from gpu_util import assert_agreement, disagreements, make_engine, normwise

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def native():
    from iteration_level_scheduling_gb300 import build
    build.build()
    from iteration_level_scheduling_gb300 import native as n
    return n


def f64(w):
    f = lambda a: np.asarray(a, np.float64)
    out = {k: f(v) for k, v in w.items() if k != "layers"}
    out["layers"] = [{k: f(v) for k, v in L.items()} for L in w["layers"]]
    return out


@pytest.mark.parametrize("cfg,tol", [
    (synth.TINY, 1e-4),
    (synth.ModelConfig(n_layers=2, hidden=256, n_heads=2, ffn=512, vocab=1000, max_pos=256, dtype="bf16"), 2e-2),
])
def test_padded_request_level_batches_match_oracle(native, cfg, tol):
    w = synth.make_weights(cfg, 21, random_affine=True)
    w64 = f64(w)
    rnd = np.random.default_rng(21)
    outs = [5, 12, 3, 8, 6, 2]
    specs = [synth.RequestSpec(i, 0.0, rnd.integers(0, cfg.vocab, int(L)).tolist(), outs[i])
             for i, L in enumerate([3, 9, 5, 14, 7, 1])]
    reserve = 64  # every member's reservation holds its padded prompt and its ghost rows
    max_batch = 4
    eng = make_engine(cfg, w, 256, max_batch, max_batch * reserve)
    store = KVStore(cfg.n_layers, cfg.hidden)
    members, ctx, kv = [], {}, {}
    worst = 0.0
    agree = total = padded_rows = real_rows = 0
    mismatches = []

    def token_fn(it):
        nonlocal members, worst, agree, total, padded_rows, real_rows
        if all(p == 0 for p in it.phase):  # a new request-level batch forms: its members' reservations
            for r in members:
                eng.kv_free(r)
            members = list(it.rids)
            for r in members:
                kv[r] = eng.kv_alloc(r, reserve)
        real = dict(zip(it.rids, range(len(it.rids))))
        offs = it.offsets
        rid, ph, n, cx, ko, toks = [], [], [], [], [], []
        for r in members:
            if r in real:
                i = real[r]
                rid.append(r), ph.append(it.phase[i]), n.append(it.n_input[i]), cx.append(it.ctx[i])
                ko.append(kv[r]), toks.extend(it.tokens[offs[i]:offs[i + 1]])
            else:  # a finished member: a single row on token 0 after its own context
                rid.append(r), ph.append(1), n.append(1), cx.append(ctx[r]), ko.append(kv[r]), toks.append(0)
        b = native.BatchDesc(rid, ph, n, cx, ko, toks)
        assert eng.plan_words(b, padded=True) >= eng.plan_words(b)
        got = eng.run_iteration_padded(b)
        hid = eng.last_hidden(len(rid))
        lg = eng.last_logits(len(rid))
        idx = [rid.index(r) for r in it.rids]
        items = [BatchItem(r, it.tokens[offs[i]:offs[i + 1]], it.ctx[i]) for i, r in enumerate(it.rids)]
        ref = opadded.iteration(w64, cfg.n_heads, items, store)
        worst = max(worst, normwise(hid[idx], ref.hidden), normwise(lg[idx], ref.logits))
        agree += sum(int(got[j] == t) for j, t in zip(idx, ref.next_tokens))
        mismatches.extend(disagreements(got[idx], lg[idx], ref.logits, ref.next_tokens))
        total += len(idx)
        padded_rows += max(n) * len(rid)
        real_rows += sum(it.n_input)
        for r, nn, c in zip(rid, n, cx):
            ctx[r] = c + nn
        return ref.next_tokens

    s, recs = osched.run(specs, max_batch, 256, max_batch * reserve, kv_reserve=reserve, mode="request",
                         token_fn=token_fn)
    eng.close()
    assert s.generated_total == sum(outs)
    assert len(recs) == max(outs[:4]) + max(outs[4:])  # request level: each batch runs for its longest member
    assert padded_rows > real_rows  # the padding and the finished members' rows are really computed
    assert worst <= tol, worst
    assert_agreement(agree / total, total, mismatches, wide=cfg.dtype == "bf16")
