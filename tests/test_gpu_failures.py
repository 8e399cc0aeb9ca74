"""Failure detection on the GPU without a GPU fault.

The kernels never trap: an index they cannot use is clamped and recorded in the
engine's device error word, and every wait on a barrier is bounded and
recorded when it runs out.  The host reads the word after an iteration
(orca_run_iteration, orca_engine_sync), reports ORCA_ERR_DEVICE_FLAG, clears
it, and the engine stays usable.  These tests make each of those happen on
purpose -- an expired wait on a barrier nothing completes, an out-of-range
token id and a feedback reference past the previous batch in a device plan --
and then check that a normal iteration still matches the oracle.
"""

import numpy as np
import pytest
import torch

from iteration_level_scheduling_gb300 import synth
from oracle import model as omodel
from oracle.model import BatchItem, KVStore
from gpu_util import make_engine, normwise

pytestmark = pytest.mark.gpu

TOL_FP32 = 1e-4
# word of a plan's header that holds the offset of its token ids (the plan
# layout of orca_plan_build: magic, n_req, rows, decode / prefill counts,
# chunk, then the table offsets request offsets, contexts, K/V offsets, tokens)
PLAN_TOKENS_FIELD = 11


@pytest.fixture(scope="module")
def native():
    from iteration_level_scheduling_gb300 import build
    build.build()
    from iteration_level_scheduling_gb300 import native as n
    return n


def fresh_iteration_matches_oracle(native, eng, w, cfg, rid0):
    """Two new initiation requests through orca_run_iteration, against the oracle."""
    prompts = [[3, 1, 4, 1, 5], [9, 2, 6]]
    offs = [eng.kv_alloc(rid0 + i, 32) for i in range(2)]
    b = native.BatchDesc([rid0, rid0 + 1], [0, 0], [5, 3], [0, 0], offs, sum(prompts, []))
    got = eng.run_iteration(b)
    ref = omodel.iteration(w, cfg.n_heads, [BatchItem(rid0 + i, p, 0) for i, p in enumerate(prompts)],
                           KVStore(cfg.n_layers, cfg.hidden))
    assert normwise(eng.last_logits(2), ref.logits) <= TOL_FP32
    assert got.tolist() == ref.next_tokens


def engine(native):
    cfg = synth.TINY
    w = synth.make_weights(cfg, 11, random_affine=True)
    return cfg, w, make_engine(cfg, w, 64, 4, 512)


def test_expired_bounded_wait_is_reported_and_engine_stays_usable(native):
    cfg, w, eng = engine(native)
    try:
        eng.debug_expire_wait(50_000_000)  # a 50 ms limit on a barrier nothing completes
        with pytest.raises(native.OrcaError) as e:
            eng.sync()
        assert e.value.code == native.ERR_DEVICE_FLAG
        eng.sync()  # reported once, then cleared
        fresh_iteration_matches_oracle(native, eng, w, cfg, 100)
        with pytest.raises(native.OrcaError) as e:
            eng.debug_expire_wait(0)
        assert e.value.code == native.ERR_INVALID
    finally:
        eng.close()


@pytest.mark.parametrize("bad", ["token_id", "feedback_reference"])
def test_bad_index_in_a_device_plan_is_clamped_and_reported(native, bad):
    """A plan validated on the host, then changed on its way to the device: the
    embedding kernel meets an index it cannot use, clamps it, records it, and
    the next iteration is unaffected."""
    cfg, w, eng = engine(native)
    try:
        offs = [eng.kv_alloc(i, 32) for i in range(2)]
        b = native.BatchDesc([0, 1], [0, 0], [3, 2], [0, 0], offs, [7, 8, 9, 10, 11])
        plan = np.zeros(eng.plan_words(b), np.int32)
        eng.plan_build(b, plan)
        tokens_at = int(plan[PLAN_TOKENS_FIELD])
        assert plan[tokens_at:tokens_at + 5].tolist() == [7, 8, 9, 10, 11]
        plan[tokens_at + 3] = cfg.vocab + 7 if bad == "token_id" else -1000
        dev = torch.from_numpy(plan).cuda()
        eng.run_planned(plan, dev.data_ptr())
        with pytest.raises(native.OrcaError) as e:
            eng.sync()
        assert e.value.code == native.ERR_DEVICE_FLAG
        eng.sync()
        fresh_iteration_matches_oracle(native, eng, w, cfg, 200)
    finally:
        eng.close()
