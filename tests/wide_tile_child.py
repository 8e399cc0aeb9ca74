"""Run by test_gpu_ops in a process of its own (the kernel-choice overrides are
read once per process).  With ORCA_GEMM_SK=-1 (test_linear_wide_token_tile)
stand-alone linear calls take the one-tile-per-CTA kernel: shapes with
257..448 rows whose launch model picks one wide token tile (two MMAs per K
step).  With ORCA_GEMM_WHOLE=2 (test_linear_whole_walk_one_to_two_waves) the
same shapes, 160..240 tiles, take the whole-tile walk with one or two tiles
per CTA.  Prints one JSON line per case."""

import json
import sys

import numpy as np
import torch

sys.path.insert(0, __file__.rsplit("/", 2)[0])
from iteration_level_scheduling_gb300 import native, synth  # noqa: E402
from oracle.model import gelu  # noqa: E402

SHAPES = [(300, 15360, 512), (448, 12800, 320), (264, 10240, 256), (401, 12288, 128)]


def main():
    eng = native.Engine(1, 64, 4, 64, 64, 16, native.DTYPE_BF16, 16, 4, 16, None,
                        torch.cuda.current_stream().cuda_stream)
    for m, n, k in SHAPES:
        g = np.random.default_rng(m * 131 + n + k)
        x = synth.bf16_round(g.standard_normal((m, k), dtype=np.float32))
        w = synth.bf16_round(g.standard_normal((n, k), dtype=np.float32) * np.float32(1 / np.sqrt(k)))
        bias = g.standard_normal(n, dtype=np.float32)
        resid = g.standard_normal((m, n), dtype=np.float32)
        xd = torch.from_numpy(x).cuda().to(torch.bfloat16)
        wd = torch.from_numpy(w).cuda().to(torch.bfloat16)
        wp = torch.zeros(eng.packed_weight_elems(n, k), dtype=torch.bfloat16, device="cuda")
        eng.pack_weight(wd.data_ptr(), n, k, wp.data_ptr())
        bd = torch.from_numpy(bias).cuda()
        y = x.astype(np.float64) @ w.astype(np.float64).T
        for mode in ("plain_bf16", "bias_gelu_bf16", "bias_resid_f32"):
            for packed in (False, True):
                wptr = wp.data_ptr() if packed else wd.data_ptr()
                if mode == "bias_resid_f32":
                    out = torch.from_numpy(resid).cuda()
                    eng.op_linear(native.DTYPE_BF16, xd.data_ptr(), wptr, m, n, k, bias=bd.data_ptr(),
                                  resid=out.data_ptr(), out_f32=out.data_ptr(), w_packed=packed)
                    ref = y + bias + resid
                    got = out.cpu().numpy().astype(np.float64)
                else:
                    act = mode == "bias_gelu_bf16"
                    out = torch.zeros((m, n), dtype=torch.bfloat16, device="cuda")
                    eng.op_linear(native.DTYPE_BF16, xd.data_ptr(), wptr, m, n, k,
                                  bias=bd.data_ptr() if act else 0, gelu=act, out_bf16=out.data_ptr(),
                                  w_packed=packed)
                    ref = gelu(y + bias) if act else y
                    got = out.float().cpu().numpy().astype(np.float64)
                rel = float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))
                print(json.dumps(dict(m=m, n=n, k=k, mode=mode, packed=packed, rel=rel)), flush=True)
    eng.close()


if __name__ == "__main__":
    main()
