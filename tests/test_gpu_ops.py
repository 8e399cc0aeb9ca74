"""Kernel-level parity of the flattened linear layer (tcgen05 bf16 and SIMT fp32)
against the oracle's definition y = x W^T + b, GeLU, + residual, on the same
bf16-rounded inputs.  Sizes span several tiles, ragged edges in both the token
and the feature dimension, the split-K path and the multi-token-tile path."""

import numpy as np
import pytest
import torch

from iteration_level_scheduling_gb300 import synth
from oracle.model import gelu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eng():
    from iteration_level_scheduling_gb300 import build, native
    build.build()
    e = native.Engine(1, 64, 4, 64, 64, 16, native.DTYPE_BF16, 16, 4, 16, None,
                      torch.cuda.current_stream().cuda_stream)
    yield e
    e.close()


def ref_linear(x, w, bias=None, act=False, resid=None):
    y = x.astype(np.float64) @ w.astype(np.float64).T
    if bias is not None:
        y = y + bias.astype(np.float64)
    if act:
        y = gelu(y)
    if resid is not None:
        y = y + resid.astype(np.float64)
    return y


def rel(a, ref):
    return float(np.max(np.abs(a.astype(np.float64) - ref)) / max(np.max(np.abs(ref)), 1e-30))


SHAPES = [
    (1, 128, 64), (16, 256, 128), (5, 130, 64), (64, 384, 1024), (100, 200, 512), (64, 5120, 1024),
    (300, 640, 256), (477, 1024, 1024), (600, 1280, 320), (1000, 384, 128), (2048, 512, 64), (64, 128, 20480),
    (16, 128, 64), (33, 15360, 128), (256, 2560, 5120),
    # stream-K (>= 129 rows): tiles cut into several pieces at odd offsets, CTAs
    # holding a first and a last piece, three whole tiles per CTA (accumulator
    # buffer reuse), ragged rows and features
    (136, 12800, 320), (200, 6400, 192), (144, 51200, 64), (129, 1000, 2048),
    # stream-K over several token tiles: feature-tile major with cut tiles (2
    # token tiles), token-tile major with cut tiles (5 token tiles)
    (300, 12800, 320), (1100, 5120, 512),
    # more output tiles than SMs at decode sizes (two CTAs on some SMs),
    # 1..128 rows, the vocabulary-sized tail
    (64, 20480, 256), (7, 50257, 192), (128, 19584, 128), (100, 25600, 320), (1, 50257, 64),
    # the persistent whole-tile walk (1025+ rows, two waves of tiles or more):
    # several tiles per CTA through both accumulator buffers, a partial raster
    # group (63 feature tiles, the last one ragged), ragged token tiles
    (1100, 12800, 128), (2100, 8000, 192), (4097, 5120, 64),
]


def packed(eng, wd, n, k):
    """The tile-contiguous copy of a bf16 weight the engine streams."""
    buf = torch.zeros(eng.packed_weight_elems(n, k), dtype=torch.bfloat16, device="cuda")
    eng.pack_weight(wd.data_ptr(), n, k, buf.data_ptr())
    return buf


@pytest.mark.parametrize("m,n,k", SHAPES)
@pytest.mark.parametrize("mode", ["plain_bf16", "bias_gelu_bf16", "bias_resid_f32"])
@pytest.mark.parametrize("w_packed", [False, True])
def test_linear_tc_bf16(eng, m, n, k, mode, w_packed):
    from iteration_level_scheduling_gb300 import native
    g = np.random.default_rng(m * 7919 + n * 31 + k)
    x = synth.bf16_round(g.standard_normal((m, k), dtype=np.float32))
    w = synth.bf16_round(g.standard_normal((n, k), dtype=np.float32) * np.float32(1 / np.sqrt(k)))
    bias = g.standard_normal(n, dtype=np.float32)
    resid = g.standard_normal((m, n), dtype=np.float32)
    xd = torch.from_numpy(x).cuda().to(torch.bfloat16)
    wd = torch.from_numpy(w).cuda().to(torch.bfloat16)
    if w_packed:
        wd = packed(eng, wd, n, k)
    bd = torch.from_numpy(bias).cuda()
    if mode == "bias_resid_f32":
        out = torch.from_numpy(resid).cuda()
        eng.op_linear(native.DTYPE_BF16, xd.data_ptr(), wd.data_ptr(), m, n, k, bias=bd.data_ptr(),
                      resid=out.data_ptr(), out_f32=out.data_ptr(), w_packed=w_packed)
        ref = ref_linear(x, w, bias, False, resid)
        # fp32 accumulation of k products: rounding error grows like sqrt(k)
        assert rel(out.cpu().numpy(), ref) < 1e-5 * max(1.0, np.sqrt(k / 1024))
    else:
        out = torch.zeros((m, n), dtype=torch.bfloat16, device="cuda")
        act = mode == "bias_gelu_bf16"
        eng.op_linear(native.DTYPE_BF16, xd.data_ptr(), wd.data_ptr(), m, n, k,
                      bias=bd.data_ptr() if act else 0, gelu=act, out_bf16=out.data_ptr(), w_packed=w_packed)
        ref = ref_linear(x, w, bias if act else None, act)
        assert rel(out.float().cpu().numpy(), ref) < 8e-3


def test_pack_weight_layout(eng):
    """The packed layout is the documented one: tile (ft, kb) at (ft * k/64 + kb) * 8192, row r of the
    tile at r * 64 elements, 8-element chunk c at chunk position c ^ (r % 8), rows past n_out zero."""
    n, k = 200, 192
    w = torch.arange(n * k, dtype=torch.float32).reshape(n, k).remainder(251).to(torch.bfloat16).cuda()
    p = packed(eng, w, n, k).view(torch.int16).cpu().numpy()
    wn = w.view(torch.int16).cpu().numpy()
    kbn = k // 64
    for ft in range(2):
        for kb in range(kbn):
            tile = p[(ft * kbn + kb) * 8192:(ft * kbn + kb + 1) * 8192].reshape(128, 8, 8)
            for r in range(128):
                for c in range(8):
                    row = ft * 128 + r
                    expect = wn[row, kb * 64 + c * 8: kb * 64 + c * 8 + 8] if row < n else np.zeros(8, np.int16)
                    assert (tile[r, c ^ (r % 8)] == expect).all()


def test_linear_tc_lm_head_shape(eng):
    """Tied LM head: V = 50257 (not a multiple of the 128-row tile), fp32 logits."""
    from iteration_level_scheduling_gb300 import native
    m, n, k = 7, 50257, 1024
    g = np.random.default_rng(3)
    x = synth.bf16_round(g.standard_normal((m, k), dtype=np.float32))
    w = synth.bf16_round(g.standard_normal((n, k), dtype=np.float32) * np.float32(0.02))
    out = torch.zeros((m, n), dtype=torch.float32, device="cuda")
    xd = torch.from_numpy(x).cuda().to(torch.bfloat16)
    wd = packed(eng, torch.from_numpy(w).cuda().to(torch.bfloat16), n, k)
    eng.op_linear(native.DTYPE_BF16, xd.data_ptr(), wd.data_ptr(), m, n, k, out_f32=out.data_ptr(), w_packed=True)
    ref = ref_linear(x, w)
    got = out.cpu().numpy()
    assert rel(got, ref) < 1e-5
    assert (got.argmax(1) == ref.argmax(1)).all()


def test_linear_tc_repeatable(eng):
    """Split-K reduces the partials in a fixed order: two launches agree bit for bit."""
    from iteration_level_scheduling_gb300 import native
    m, n, k = 64, 384, 5120
    g = np.random.default_rng(4)
    xd = torch.from_numpy(synth.bf16_round(g.standard_normal((m, k), dtype=np.float32))).cuda().to(torch.bfloat16)
    wd = torch.from_numpy(synth.bf16_round(g.standard_normal((n, k), dtype=np.float32))).cuda().to(torch.bfloat16)
    a = torch.zeros((m, n), device="cuda")
    b = torch.zeros((m, n), device="cuda")
    eng.op_linear(native.DTYPE_BF16, xd.data_ptr(), wd.data_ptr(), m, n, k, out_f32=a.data_ptr())
    eng.op_linear(native.DTYPE_BF16, xd.data_ptr(), wd.data_ptr(), m, n, k, out_f32=b.data_ptr())
    assert torch.equal(a, b)


def test_linear_sk_repeatable(eng):
    """Stream-K sums the pieces of a cut tile in CTA order whoever finishes last:
    launches agree bit for bit (and the arrival counters are back at zero after each)."""
    from iteration_level_scheduling_gb300 import native
    m, n, k = 300, 1280, 1024
    g = np.random.default_rng(5)
    xd = torch.from_numpy(synth.bf16_round(g.standard_normal((m, k), dtype=np.float32))).cuda().to(torch.bfloat16)
    wd = torch.from_numpy(synth.bf16_round(g.standard_normal((n, k), dtype=np.float32))).cuda().to(torch.bfloat16)
    outs = [torch.zeros((m, n), device="cuda") for _ in range(4)]
    for o in outs:
        eng.op_linear(native.DTYPE_BF16, xd.data_ptr(), wd.data_ptr(), m, n, k, out_f32=o.data_ptr())
    for o in outs[1:]:
        assert torch.equal(outs[0], o)


def run_child(env_extra):
    import json
    import os
    import subprocess
    import sys
    env = dict(os.environ, **env_extra)
    child = os.path.join(os.path.dirname(__file__), "wide_tile_child.py")
    out = subprocess.run([sys.executable, child], env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    return [json.loads(line) for line in out.stdout.splitlines() if line.startswith("{")]


def test_linear_whole_walk_one_to_two_waves(eng):
    """The whole-tile walk between one and two waves of tiles (as QKV takes it
    inside an iteration at 257..512 rows): CTAs holding one tile beside CTAs
    holding two, every epilogue, packed and unpacked weights, ragged rows."""
    rows = run_child({"ORCA_GEMM_WHOLE": "2"})
    assert len(rows) == 4 * 3 * 2
    for r in rows:
        tol = 1e-5 * max(1.0, np.sqrt(r["k"] / 1024)) if r["mode"] == "bias_resid_f32" else 8e-3
        assert r["rel"] < tol, r


def test_linear_wide_token_tile(eng):
    """257..448 rows in one token tile (two MMAs per K step, the epilogue in two
    256-column halves), in a process where stand-alone calls may not take the
    stream-K kernel: every epilogue, packed and unpacked weights, ragged rows."""
    import json
    import os
    import subprocess
    import sys
    env = dict(os.environ, ORCA_GEMM_SK="-1")
    child = os.path.join(os.path.dirname(__file__), "wide_tile_child.py")
    out = subprocess.run([sys.executable, child], env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    rows = [json.loads(line) for line in out.stdout.splitlines() if line.startswith("{")]
    assert len(rows) == 4 * 3 * 2
    for r in rows:
        tol = 1e-5 * max(1.0, np.sqrt(r["k"] / 1024)) if r["mode"] == "bias_resid_f32" else 8e-3
        assert r["rel"] < tol, r


@pytest.mark.parametrize("m,n,k", [(1, 64, 64), (37, 256, 64), (130, 200, 256), (64, 512, 20)])
def test_linear_simt_f32(eng, m, n, k):
    from iteration_level_scheduling_gb300 import native
    g = np.random.default_rng(m + n + k)
    x = g.standard_normal((m, k), dtype=np.float32)
    w = g.standard_normal((n, k), dtype=np.float32)
    bias = g.standard_normal(n, dtype=np.float32)
    resid = g.standard_normal((m, n), dtype=np.float32)
    out = torch.from_numpy(resid).cuda()
    xd, wd, bd = (torch.from_numpy(a).cuda() for a in (x, w, bias))  # keep the device copies alive
    eng.op_linear(native.DTYPE_FP32, xd.data_ptr(), wd.data_ptr(), m, n, k, bias=bd.data_ptr(), gelu=True,
                  resid=out.data_ptr(), out_f32=out.data_ptr())
    assert rel(out.cpu().numpy(), ref_linear(x, w, bias, True, resid)) < 1e-5
