"""Run by test_gpu_attention in a process of its own (kernel-choice overrides
are read once per process): through orca_op_attention, the ragged causal
prefill case at head_dim 128 and 64 and a decode batch with many work items
per CTA at head_dim 128, one JSON line each with the error against the
oracle."""

import json
import sys

sys.path.insert(0, __file__.rsplit("/", 2)[0])
sys.path.insert(0, __file__.rsplit("/", 1)[0])
import numpy as np  # noqa: E402
import torch  # noqa: E402

from iteration_level_scheduling_gb300 import native  # noqa: E402
from test_gpu_attention import make_case, oracle_out, rel, run_op  # noqa: E402


def main():
    eng = native.Engine(1, 64 * 16, 64, 64, 64, 4096, native.DTYPE_BF16, 1024, 64, 16, None,
                        torch.cuda.current_stream().cuda_stream)
    reqs = [(2, 0), (17, 0), (64, 0), (65, 0), (130, 0), (7, 50), (70, 200), (1, 9), (300, 0)]
    for d in (128, 64):
        offs, kv_slots, pool, qkv = make_case(2, 3, d, reqs, "bf16")
        got = run_op(eng, "bf16", reqs, offs, kv_slots, pool, qkv, 3, d)
        ref = oracle_out(reqs, offs, pool, qkv, 3, d)
        print(json.dumps(dict(case="prefill", d=d, rel=rel(got, ref))), flush=True)
    g = np.random.default_rng(7)
    reqs = [(1, int(c)) for c in g.integers(1, 3000, size=48)]
    offs, kv_slots, pool, qkv = make_case(7, 40, 128, reqs, "bf16")
    got = run_op(eng, "bf16", reqs, offs, kv_slots, pool, qkv, 40, 128)
    ref = oracle_out(reqs, offs, pool, qkv, 40, 128)
    print(json.dumps(dict(case="decode", d=128, rel=rel(got, ref))), flush=True)
    eng.close()


if __name__ == "__main__":
    main()
