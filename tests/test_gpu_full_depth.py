"""Parity at full depth and size, in the launch configuration bench.py times:
the engine runs one whole iteration of each large configuration (device-drawn
weights and synthetic K/V contexts as in bench.py) and a few sampled requests
are recomputed by the oracle, which streams the same weights and K/V back one
layer at a time.  Requests are independent, so the sampled rows of the full
batch must equal the oracle's result for those requests alone."""

import numpy as np
import pytest
import torch

import bench
from iteration_level_scheduling_gb300 import synth
from gpu_util import assert_agreement, full_depth_check

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


@pytest.fixture(scope="module", autouse=True)
def built():
    from iteration_level_scheduling_gb300 import build
    build.build()


def make(cfg, max_tokens, max_batch, kv_slots, seed):
    from iteration_level_scheduling_gb300 import native
    keep, ptrs = bench.gpu_weights(cfg, seed)
    eng = native.Engine(cfg.n_layers, cfg.hidden, cfg.n_heads, cfg.ffn, cfg.vocab, cfg.max_pos, native.DTYPE_BF16,
                        max_tokens, max_batch, kv_slots, ptrs, torch.cuda.current_stream().cuda_stream)
    bench.fill_kv_pool(eng, seed)
    return keep, eng


def release(keep, eng):
    eng.close()
    keep.clear()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def pick(ctx, n, want_prefill=True, n_dec=16):
    """Indices: n_dec single-row requests spread evenly over the sorted cached
    context lengths (the shortest and the longest included), and the shortest
    multi-row request if any."""
    dec = [i for i in range(len(n)) if n[i] == 1]
    dec.sort(key=lambda i: ctx[i])
    k = min(n_dec, len(dec))
    idx = {dec[round(j * (len(dec) - 1) / max(k - 1, 1))] for j in range(k)}
    pre = [i for i in range(len(n)) if n[i] > 1]
    if want_prefill and pre:
        idx.add(min(pre, key=lambda i: n[i]))
    return sorted(idx)


def check(r):
    print(r)
    assert r["argmax_ok"]
    assert r["n"] >= 16
    assert r["h"] <= TOL_BF16 and r["l"] <= TOL_BF16, r
    assert_agreement(r["agree"], r["n"], r["mismatches"], wide=True)


def test_gpt3_13b_bench_window_iteration():
    """The first iteration of the timed window of bench.py (40 layers, 64 requests)."""
    from iteration_level_scheduling_gb300 import native
    cfg = bench.MODEL
    keep, eng = make(cfg, bench.MAX_TOKENS, bench.MAX_BATCH, bench.MAX_BATCH * bench.KV_RESERVE, 0)
    s = native.Scheduler(bench.MAX_BATCH, bench.MAX_TOKENS, kv_reserve=bench.KV_RESERVE, engine=eng)
    for sp in bench.make_trace(0):
        s.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len)
    bench.advance(s, 256)
    st, b = s.next()
    assert st == 1 and b.n_req == bench.MAX_BATCH
    idx = pick(b.ctx_len.tolist(), b.n_input.tolist())
    r = full_depth_check(eng, keep, cfg, b, idx)
    s.close()
    release(keep, eng)
    check(r)


def test_gpt3_6_7b_decode_heavy_iteration():
    """6.7B shape (32 layers, H 4096): 128 increment requests, contexts U[256, 1024], 1280-token reservations."""
    from iteration_level_scheduling_gb300 import native
    cfg = synth.GPT3_6_7B
    B, reserve = 128, 1280
    keep, eng = make(cfg, 4096, B, B * reserve, 1)
    g = np.random.default_rng(4)
    ctx = g.integers(256, 1025, B).tolist()
    offs = [eng.kv_alloc(i, reserve) for i in range(B)]
    b = native.BatchDesc(list(range(B)), [1] * B, [1] * B, ctx, offs, g.integers(0, cfg.vocab, B).tolist())
    r = full_depth_check(eng, keep, cfg, b, pick(ctx, [1] * B))
    release(keep, eng)
    check(r)


def test_gpt3_13b_prefill_heavy_iteration():
    """13B shape, 40 layers: 16 initiation requests with prompts U[1024, 2048] and
    128 increment requests with contexts U[128, 2048] in one iteration (the
    compute-bound flattened-GEMM regime)."""
    from iteration_level_scheduling_gb300 import native
    cfg = bench.MODEL
    g = np.random.default_rng(5)
    prompts = g.integers(1024, 2049, 16).tolist()
    ctx_inc = g.integers(128, 2049, 128).tolist()
    n = prompts + [1] * 128
    ctx = [0] * 16 + ctx_inc
    B, rows = len(n), sum(n)
    need = [c + k for c, k in zip(ctx, n)]
    keep, eng = make(cfg, rows, B, sum(need), 2)
    offs = [eng.kv_alloc(i, need[i]) for i in range(B)]
    toks = g.integers(0, cfg.vocab, rows).tolist()
    b = native.BatchDesc(list(range(B)), [1 if c else 0 for c in ctx], n, ctx, offs, toks)
    r = full_depth_check(eng, keep, cfg, b, pick(ctx, n))
    release(keep, eng)
    check(r)


def test_gpt3_13b_mid_rows_iteration():
    """13B shape, 40 layers: one 300-token prompt with 63 increment requests (363
    rows, like the prompt-carrying iterations of the bench trace): the linear
    layers run one wide token tile (two MMAs per K step), the residual
    projections with split-K slabs."""
    from iteration_level_scheduling_gb300 import native
    cfg = bench.MODEL
    g = np.random.default_rng(6)
    ctx_inc = g.integers(64, 900, 63).tolist()
    n = [300] + [1] * 63
    ctx = [0] + ctx_inc
    B, rows = len(n), sum(n)
    need = [c + k for c, k in zip(ctx, n)]
    keep, eng = make(cfg, rows, B, sum(need), 3)
    offs = [eng.kv_alloc(i, need[i]) for i in range(B)]
    toks = g.integers(0, cfg.vocab, rows).tolist()
    b = native.BatchDesc(list(range(B)), [1 if c else 0 for c in ctx], n, ctx, offs, toks)
    r = full_depth_check(eng, keep, cfg, b, pick(ctx, n))
    release(keep, eng)
    check(r)
