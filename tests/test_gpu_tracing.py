"""NVTX ranges (ORCA_NVTX=1, read once per process): the same iteration, with
every launch and the iteration wrapped in a named range, still matches the
oracle."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

CHILD = r"""
import sys
sys.path.insert(0, sys.argv[1])
import numpy as np
from iteration_level_scheduling_gb300 import build, synth
build.build()
from iteration_level_scheduling_gb300 import native
from oracle import model as omodel
from oracle.model import BatchItem, KVStore
sys.path.insert(0, sys.argv[1] + "/tests")
from gpu_util import make_engine, normwise
cfg = synth.TINY
w = synth.make_weights(cfg, 5, random_affine=True)
eng = make_engine(cfg, w, 64, 4, 512)
prompts = [[3, 1, 4, 1, 5], [9, 2, 6]]
offs = [eng.kv_alloc(i, 32) for i in range(2)]
got = eng.run_iteration(native.BatchDesc([0, 1], [0, 0], [5, 3], [0, 0], offs, sum(prompts, [])))
ref = omodel.iteration(w, cfg.n_heads, [BatchItem(i, p, 0) for i, p in enumerate(prompts)],
                       KVStore(cfg.n_layers, cfg.hidden))
err = normwise(eng.last_logits(2), ref.logits)
eng.close()
assert err <= 1e-4, err
assert got.tolist() == ref.next_tokens
print("ok", err)
"""


def test_iteration_with_nvtx_ranges_matches_oracle():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, ORCA_NVTX="1")
    out = subprocess.run([sys.executable, "-c", CHILD, root], env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip().splitlines()[-1].startswith("ok")
