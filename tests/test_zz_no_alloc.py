"""The allocation-free decode attention entry point.

Callers that cannot allocate device memory at call time (their process has
given all device memory to its own allocator, or their serving thread may not
call cudaMalloc) cannot create an engine; orca_attention_decode_noalloc runs
the engine's split-K decode kernel with its scratch in a fixed device array
inside the library.  Its output must match the engine entry point
orca_op_attention on the same inputs and the oracle's single-query attention,
call after call (the array is shared and keeps the previous call's contents).
This file is collected last on purpose.
"""

import numpy as np
import pytest
import torch

from iteration_level_scheduling_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def native():
    from iteration_level_scheduling_gb300 import build
    build.build()
    from iteration_level_scheduling_gb300 import native as n
    return n


def decode_case(seed, n_req, n_heads, d, dtype, ctx_range):
    g = np.random.default_rng(seed)
    rnd = synth.bf16_round if dtype == "bf16" else (lambda a: a)
    ctx = g.integers(ctx_range[0], ctx_range[1], size=n_req, endpoint=True)
    offs, o = [], 0
    for c in ctx:
        o += int(g.integers(0, 7))
        offs.append(o)
        o += int(c) + 1
    kv_slots = o + 5
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    pool = torch.from_numpy(rnd(g.standard_normal((2, n_heads, kv_slots, d), dtype=np.float32))).cuda().to(tdt)
    qkv = torch.from_numpy(rnd(g.standard_normal((n_req, 3 * n_heads * d), dtype=np.float32))).cuda().to(tdt)
    return ctx.tolist(), offs, kv_slots, pool, qkv


def rel(a, ref):
    a, ref = a.float().cpu().numpy().astype(np.float64), ref.float().cpu().numpy().astype(np.float64)
    return float(np.max(np.abs(a - ref)) / np.max(np.abs(ref)))


def oracle_decode(qkv, pool, ctx, offs, n_heads, d):
    """The oracle's attention for one query row per request: request i's row sits
    at position ctx[i] and sees its keys 0 .. ctx[i] (slots offs[i] ..)."""
    from oracle.model import attention_one
    H = n_heads * d
    q = qkv.float().cpu().numpy().astype(np.float64)[:, :H]
    out = np.zeros((len(ctx), H))
    for i, (c, o) in enumerate(zip(ctx, offs)):
        kv = pool[:, :, o:o + c + 1, :].float().cpu().numpy().astype(np.float64)  # [K|V][head][key][d]
        k = kv[0].transpose(1, 0, 2).reshape(c + 1, H)
        v = kv[1].transpose(1, 0, 2).reshape(c + 1, H)
        out[i] = attention_one(q[i:i + 1], k, v, np.array([c]), n_heads)[0]
    return out


@pytest.mark.parametrize("dtype,d,n_heads,tol", [("bf16", 128, 40, 1e-2), ("fp32", 64, 8, 1e-5)])
def test_noalloc_matches_engine_entry_point(native, dtype, d, n_heads, tol):
    dt = native.DTYPE_BF16 if dtype == "bf16" else native.DTYPE_FP32
    eng = native.Engine(1, n_heads * d, n_heads, 64, 64, 4096, native.DTYPE_BF16, 64, 64, 16, None,
                        torch.cuda.current_stream().cuda_stream)
    try:
        # two calls in a row, on different batches
        for seed, n_req, ctx_range in ((11, 64, (32, 1100)), (12, 37, (0, 2100))):
            ctx, offs, kv_slots, pool, qkv = decode_case(seed, n_req, n_heads, d, dtype, ctx_range)
            tdt = pool.dtype
            ref = torch.zeros((n_req, n_heads * d), dtype=tdt, device="cuda")
            eng.op_attention(dt, qkv.data_ptr(), pool.data_ptr(), kv_slots, n_heads, d, [1] * n_req, ctx, offs,
                             ref.data_ptr())
            got = torch.full((n_req, n_heads * d), float("nan"), dtype=tdt, device="cuda")
            native.attention_decode_noalloc(dt, qkv.data_ptr(), pool.data_ptr(), kv_slots, n_heads, d, ctx, offs,
                                            got.data_ptr(), torch.cuda.current_stream().cuda_stream)
            torch.cuda.synchronize()
            assert torch.isfinite(got.float()).all()
            assert rel(got, ref) <= tol
            exact = oracle_decode(qkv, pool, ctx, offs, n_heads, d)
            g64 = got.float().cpu().numpy().astype(np.float64)
            assert float(np.max(np.abs(g64 - exact)) / np.max(np.abs(exact))) <= tol
    finally:
        eng.close()


def test_noalloc_rejects_sizes_beyond_its_scratch(native):
    n_heads, d = 4, 64
    with pytest.raises(native.OrcaError) as e:
        native.attention_decode_noalloc(native.DTYPE_BF16, 16, 16, 10 ** 6, n_heads, d, [5] * 257, [0] * 257, 16)
    assert e.value.code == native.ERR_LIMIT
    with pytest.raises(native.OrcaError) as e:  # too many work items for the plan tables: 256 x 63 chunks
        native.attention_decode_noalloc(native.DTYPE_BF16, 16, 16, 40000, 128, 128, [32000] * 256, [0] * 256, 16)
    assert e.value.code == native.ERR_LIMIT
    with pytest.raises(native.OrcaError) as e:  # tables fit (1024 work items) but the partials do not (17 Mi floats)
        native.attention_decode_noalloc(native.DTYPE_BF16, 16, 16, 40000, 128, 128, [2000] * 256, [0] * 256, 16)
    assert e.value.code == native.ERR_LIMIT
