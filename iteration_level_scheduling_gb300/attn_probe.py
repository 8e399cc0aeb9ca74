"""Time the attention of one layer for a batch of prompts through the C ABI
(orca_op_attention), for kernel-level profiling:
``python -m iteration_level_scheduling_gb300.attn_probe --prompts 8 --len 2048 --heads 40``.

Each of ``--prompts`` requests brings ``--len`` new rows after ``--ctx`` cached
keys (initiation phase when the context is 0), so every request is one causal
prefill of its own keys.  Inputs are seeded random bf16 values: q rows of a
[rows, 3H] matrix, K and V in a pool with each request's keys contiguous.
Each timed call is bracketed by CUDA events; the call uploads its small plan
before the kernel, so the time is an upper bound of the kernel's (the kernel
alone: ncu).  Prints one JSON line with the average time and the achieved
TFLOP/s over the causal pairs (4 * head_dim flops per pair and head).
ORCA_ATTN_PREFILL_TC=-1 in the environment selects the mma.sync kernel.
"""

from __future__ import annotations

import argparse
import json


def main() -> None:
    import torch

    from . import build
    build.build()
    from . import native

    p = argparse.ArgumentParser()
    p.add_argument("--prompts", type=int, default=8)
    p.add_argument("--len", type=int, default=2048, help="new rows per request")
    p.add_argument("--ctx", type=int, default=0, help="cached keys before them")
    p.add_argument("--heads", type=int, default=40)
    p.add_argument("--d", type=int, default=128, help="head_dim (64 or 128)")
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--reps", type=int, default=10)
    a = p.parse_args()

    torch.manual_seed(0)
    stream = torch.cuda.current_stream().cuda_stream
    H = a.heads * a.d
    rows = a.prompts * a.len
    per_req = a.ctx + a.len
    kv_slots = a.prompts * per_req
    eng = native.Engine(1, H, a.heads, 64, 64, per_req, native.DTYPE_BF16, rows, max(a.prompts, 1), 16, None, stream)
    qkv = torch.randn(rows, 3 * H, device="cuda").to(torch.bfloat16)
    pool = torch.randn(2, a.heads, kv_slots, a.d, device="cuda").to(torch.bfloat16)
    out = torch.empty(rows, H, device="cuda", dtype=torch.bfloat16)
    n_input = [a.len] * a.prompts
    ctx = [a.ctx] * a.prompts
    offs = [i * per_req for i in range(a.prompts)]

    def call():
        eng.op_attention(native.DTYPE_BF16, qkv.data_ptr(), pool.data_ptr(), kv_slots, a.heads, a.d, n_input, ctx,
                         offs, out.data_ptr(), sync=False)

    for _ in range(a.warmup):
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.reps)]
    for s, e in ev:
        s.record()
        call()
        e.record()
    torch.cuda.synchronize()
    t = sum(s.elapsed_time(e) for s, e in ev) / len(ev) * 1e-3
    pairs = a.prompts * sum(a.ctx + r + 1 for r in range(a.len))
    flops = 4.0 * a.d * a.heads * pairs
    print(json.dumps({"prompts": a.prompts, "len": a.len, "ctx": a.ctx, "heads": a.heads, "d": a.d,
                      "us": t * 1e6, "TFLOP/s": flops / t / 1e12}), flush=True)
    eng.close()


if __name__ == "__main__":
    main()
