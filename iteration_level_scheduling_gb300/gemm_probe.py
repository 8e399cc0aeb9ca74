"""Time one flattened linear layer through the C ABI (orca_op_linear), for
kernel-level profiling: ``python -m iteration_level_scheduling_gb300.gemm_probe
--m 24765 --n 20480 --k 5120 --epilogue bias_gelu_bf16``.

The weight is packed tile-contiguous as an engine streams it; inputs are
seeded random bf16 values.  Each timed launch is bracketed by CUDA events
with an L2 flush (a 512 MiB write) before it.  Prints one JSON line with the
average time and the achieved TFLOP/s and GB/s of the algorithmic work.  The
kernel chosen is the engine's own choice for a stand-alone call (stream-K
from 129 rows when every SM gets a tile); ORCA_GEMM_SK=-1 in the
environment keeps the one-tile kernel, as an iteration does for every layer
but FFN1.

``--library`` times the vendor library instead (``torch.matmul``, bf16, no
epilogue), the same way, for calibration only: nothing in the engine calls it.
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
    p.add_argument("--m", type=int, required=True, help="token rows")
    p.add_argument("--n", type=int, required=True, help="output features")
    p.add_argument("--k", type=int, required=True, help="input features (multiple of 64)")
    p.add_argument("--epilogue", default="bias_gelu_bf16", choices=["bf16", "bias_gelu_bf16", "bias_resid_f32"])
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--reps", type=int, default=10)
    p.add_argument("--library", action="store_true", help="time torch.matmul on the same shape instead")
    a = p.parse_args()
    if a.library:
        library(a)
        return

    torch.manual_seed(0)
    stream = torch.cuda.current_stream().cuda_stream
    eng = native.Engine(1, 64, 4, 64, 64, 16, native.DTYPE_BF16, 16, 4, 16, None, stream)
    w = (torch.randn(a.n, a.k, device="cuda") * 0.02).to(torch.bfloat16)
    wp = torch.empty(eng.packed_weight_elems(a.n, a.k), dtype=torch.bfloat16, device="cuda")
    eng.pack_weight(w.data_ptr(), a.n, a.k, wp.data_ptr())
    del w
    x = torch.randn(a.m, a.k, device="cuda").to(torch.bfloat16)
    bias = torch.randn(a.n, device="cuda") * 0.02
    if a.epilogue == "bias_resid_f32":
        out = torch.zeros(a.m, a.n, device="cuda", dtype=torch.float32)
        kw = dict(resid=out.data_ptr(), out_f32=out.data_ptr(), bias=bias.data_ptr())
    else:
        out = torch.empty(a.m, a.n, device="cuda", dtype=torch.bfloat16)
        kw = dict(out_bf16=out.data_ptr(), bias=bias.data_ptr() if a.epilogue != "bf16" else 0,
                  gelu=a.epilogue == "bias_gelu_bf16")
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")

    def launch():
        eng.op_linear(native.DTYPE_BF16, x.data_ptr(), wp.data_ptr(), a.m, a.n, a.k, sync=False, w_packed=True, **kw)

    for _ in range(a.warmup):
        launch()
    eng.sync()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    total = 0.0
    for _ in range(a.reps):
        flush.zero_()
        s.record()
        launch()
        e.record()
        e.synchronize()
        total += s.elapsed_time(e)
    eng.sync()
    t = total / a.reps / 1000.0
    flops = 2.0 * a.m * a.n * a.k
    byts = 2.0 * (a.n * a.k + a.m * a.k) + out.element_size() * a.m * a.n * (2 if a.epilogue == "bias_resid_f32" else 1)
    print(json.dumps({"m": a.m, "n": a.n, "k": a.k, "epilogue": a.epilogue, "us": t * 1e6,
                      "TFLOP/s": flops / t / 1e12, "GB/s": byts / t / 1e9}), flush=True)
    eng.close()


def library(a) -> None:
    """torch.matmul (cuBLAS) on x [m, k] @ w[n, k]^T in bf16, timed as above."""
    import torch

    torch.manual_seed(0)
    x = torch.randn(a.m, a.k, device="cuda").to(torch.bfloat16)
    w = (torch.randn(a.n, a.k, device="cuda") * 0.02).to(torch.bfloat16)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(a.warmup):
        y = x @ w.t()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    total = 0.0
    for _ in range(a.reps):
        flush.zero_()
        s.record()
        y = x @ w.t()
        e.record()
        e.synchronize()
        total += s.elapsed_time(e)
    t = total / a.reps / 1000.0
    flops = 2.0 * a.m * a.n * a.k
    byts = 2.0 * (a.n * a.k + a.m * a.k + a.m * a.n)
    print(json.dumps({"m": a.m, "n": a.n, "k": a.k, "library": "torch.matmul", "us": t * 1e6,
                      "TFLOP/s": flops / t / 1e12, "GB/s": byts / t / 1e9}), flush=True)
    del y


if __name__ == "__main__":
    main()
