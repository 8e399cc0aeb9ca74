"""Kernel-level parity of the per-request attention (split-K decode kernel and
prefill kernels) through orca_op_attention, against the oracle's attention of
one request (each row at position ctx + j sees keys 0 .. ctx + j of its own
cache).  Inputs are seeded; K/V are bf16-rounded for the bf16 kernels."""

import numpy as np
import pytest
import torch

from iteration_level_scheduling_gb300 import synth
from oracle.model import attention_one

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eng():
    from iteration_level_scheduling_gb300 import build, native
    build.build()
    # an engine only for its stream and scratch: 64 requests, 1024 rows, 64 heads, 4096 positions
    e = native.Engine(1, 64 * 16, 64, 64, 64, 4096, native.DTYPE_BF16, 1024, 64, 16, None,
                      torch.cuda.current_stream().cuda_stream)
    yield e
    e.close()


def make_case(seed, n_heads, d, reqs, dtype):
    """reqs: list of (n_input, ctx).  Returns host arrays and device tensors."""
    g = np.random.default_rng(seed)
    H = n_heads * d
    rnd = synth.bf16_round if dtype == "bf16" else (lambda a: a)
    offs, o = [], 0
    for n, c in reqs:
        o += int(g.integers(0, 5))  # gaps between reservations
        offs.append(o)
        o += c + n
    kv_slots = o + 3
    pool = rnd(g.standard_normal((2, n_heads, kv_slots, d), dtype=np.float32))
    rows = sum(n for n, _ in reqs)
    qkv = rnd(g.standard_normal((rows, 3 * H), dtype=np.float32))
    return offs, kv_slots, pool, qkv


def oracle_out(reqs, offs, pool, qkv, n_heads, d):
    H = n_heads * d
    out = np.zeros((qkv.shape[0], H))
    r = 0
    for (n, c), off in zip(reqs, offs):
        T = c + n
        k = pool[0, :, off:off + T, :].transpose(1, 0, 2).reshape(T, H).astype(np.float64)
        v = pool[1, :, off:off + T, :].transpose(1, 0, 2).reshape(T, H).astype(np.float64)
        q = qkv[r:r + n, :H].astype(np.float64)
        out[r:r + n] = attention_one(q, k, v, c + np.arange(n), n_heads)
        r += n
    return out


def run_op(eng, dtype, reqs, offs, kv_slots, pool, qkv, n_heads, d):
    from iteration_level_scheduling_gb300 import native
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    pd = torch.from_numpy(pool).cuda().to(tdt)
    qd = torch.from_numpy(qkv).cuda().to(tdt)
    out = torch.zeros((qkv.shape[0], n_heads * d), dtype=tdt, device="cuda")
    eng.op_attention(native.DTYPE_BF16 if dtype == "bf16" else native.DTYPE_FP32, qd.data_ptr(), pd.data_ptr(),
                     kv_slots, n_heads, d, [n for n, _ in reqs], [c for _, c in reqs], offs, out.data_ptr())
    return out.float().cpu().numpy()


def rel(a, ref):
    return float(np.max(np.abs(a - ref)) / np.max(np.abs(ref)))


DECODE_CTX = [0, 1, 31, 32, 33, 63, 64, 255, 256, 511, 512, 513, 1023, 2047, 3000]


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("bf16", 32), ("fp32", 16), ("fp32", 64)])
def test_decode_split_k(eng, dtype, d):
    n_heads = 4
    reqs = [(1, c) for c in DECODE_CTX]
    offs, kv_slots, pool, qkv = make_case(1, n_heads, d, reqs, dtype)
    got = run_op(eng, dtype, reqs, offs, kv_slots, pool, qkv, n_heads, d)
    ref = oracle_out(reqs, offs, pool, qkv, n_heads, d)
    assert rel(got, ref) < (1e-2 if dtype == "bf16" else 1e-5)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("bf16", 32), ("fp32", 16)])
def test_prefill_ragged_causal(eng, dtype, d):
    n_heads = 3
    # initiation prompts of ragged lengths, plus multi-row requests with cached context
    reqs = [(2, 0), (17, 0), (64, 0), (65, 0), (130, 0), (7, 50), (70, 200), (1, 9)]
    offs, kv_slots, pool, qkv = make_case(2, n_heads, d, reqs, dtype)
    got = run_op(eng, dtype, reqs, offs, kv_slots, pool, qkv, n_heads, d)
    ref = oracle_out(reqs, offs, pool, qkv, n_heads, d)
    assert rel(got, ref) < (2e-2 if dtype == "bf16" else 1e-5)


def test_attention_13b_head_shape(eng):
    """40 heads of 128, a decode-heavy batch like the continuous-batching trace."""
    n_heads, d = 40, 128
    g = np.random.default_rng(3)
    reqs = [(1, int(c)) for c in g.integers(32, 1100, size=30)] + [(int(n), 0) for n in (300, 45)]
    offs, kv_slots, pool, qkv = make_case(3, n_heads, d, reqs, "bf16")
    got = run_op(eng, "bf16", reqs, offs, kv_slots, pool, qkv, n_heads, d)
    ref = oracle_out(reqs, offs, pool, qkv, n_heads, d)
    assert rel(got, ref) < 2e-2


def used_slots(reqs, offs, kv_slots):
    used = np.zeros(kv_slots, bool)
    for (n, c), off in zip(reqs, offs):
        used[off:off + c + n] = True
    return used


@pytest.mark.parametrize("d", [128, 64])
def test_prefill_tc_multi_tile(eng, d):
    """The tcgen05 prefill at the prompt lengths of the traces: several 128-key
    tiles per query tile, ragged query tiles (127 rows; 513 and 129 rows leave one),
    cached context before the prompt (chunked prefill) and the causal diagonal
    inside a key tile (the test engine takes up to 1024 rows)."""
    n_heads = 2
    reqs = [(513, 0), (127, 300), (129, 0), (1, 5), (128, 128), (100, 77)]
    offs, kv_slots, pool, qkv = make_case(4, n_heads, d, reqs, "bf16")
    got = run_op(eng, "bf16", reqs, offs, kv_slots, pool, qkv, n_heads, d)
    ref = oracle_out(reqs, offs, pool, qkv, n_heads, d)
    assert rel(got, ref) < 2e-2


def test_prefill_tc_rescale(eng):
    """Keys whose scale grows along the sequence, so a row's max keeps growing by
    more than 2^8 from tile to tile and O is rescaled in tensor memory many
    times."""
    n_heads, d = 2, 128
    reqs = [(600, 0), (300, 400), (60, 0)]
    offs, kv_slots, pool, qkv = make_case(5, n_heads, d, reqs, "bf16")
    for (n, c), off in zip(reqs, offs):
        t = np.arange(c + n, dtype=np.float32)
        pool[0, :, off:off + c + n, :] *= (1.0 + t / 48.0)[None, :, None]
    pool = synth.bf16_round(pool)
    got = run_op(eng, "bf16", reqs, offs, kv_slots, pool, qkv, n_heads, d)
    ref = oracle_out(reqs, offs, pool, qkv, n_heads, d)
    assert np.isfinite(got).all()
    assert rel(got, ref) < 2e-2


@pytest.mark.parametrize("d", [128, 64])
def test_attention_ignores_foreign_slots(eng, d):
    """Every pool slot that holds none of the batch's keys is NaN (slots between
    reservations and after the last): the prefill tile that reaches past its
    keys and the decode items must neither read them into a score nor let P V
    carry them into a row."""
    n_heads = 2
    reqs = [(200, 0), (1, 77), (130, 10), (1, 300), (3, 0), (64, 64)]
    offs, kv_slots, pool, qkv = make_case(6, n_heads, d, reqs, "bf16")
    pool[:, :, ~used_slots(reqs, offs, kv_slots), :] = np.nan
    got = run_op(eng, "bf16", reqs, offs, kv_slots, pool, qkv, n_heads, d)
    clean = np.where(np.isnan(pool), 0.0, pool).astype(np.float32)
    ref = oracle_out(reqs, offs, clean, qkv, n_heads, d)
    assert np.isfinite(got).all()
    assert rel(got, ref) < 2e-2


def run_child(env_extra):
    import json
    import os
    import subprocess
    import sys
    child = os.path.join(os.path.dirname(__file__), "attention_kernel_child.py")
    env = dict(os.environ, **env_extra)
    out = subprocess.run([sys.executable, child], env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    return [json.loads(line) for line in out.stdout.splitlines() if line.startswith("{")]


def test_prefill_mma_sync_kernel_when_chosen(eng):
    """The mma.sync prefill kernel (kept for comparisons, ORCA_ATTN_PREFILL_TC=-1,
    read once per process): the 128-row plan tiles as two 64-row halves."""
    rows = run_child({"ORCA_ATTN_PREFILL_TC": "-1"})
    assert len(rows) == 3
    for r in rows:
        assert r["rel"] < 2e-2, r


def test_decode_fixed_share_when_chosen(eng):
    """The tensor-core decode kernel with a fixed share of work items per CTA
    (ORCA_ATTN_DECODE_CLAIM=-1, as the allocation-free entry point runs it)
    instead of items claimed at run time: 48 requests x 40 heads, contexts up
    to 3000 keys (several items per CTA, split requests merged)."""
    rows = run_child({"ORCA_ATTN_DECODE_CLAIM": "-1"})
    assert len(rows) == 3
    for r in rows:
        assert r["rel"] < 2e-2, r


def test_decode_claimed_many_items_per_cta(eng):
    """The same decode batch with items claimed at run time, three launches in a
    row: each finds the claim counters back at zero (a counter left behind
    would skip items and leave rows unwritten)."""
    g = np.random.default_rng(7)
    reqs = [(1, int(c)) for c in g.integers(1, 3000, size=48)]
    offs, kv_slots, pool, qkv = make_case(7, 40, 128, reqs, "bf16")
    ref = oracle_out(reqs, offs, pool, qkv, 40, 128)
    for _ in range(3):
        got = run_op(eng, "bf16", reqs, offs, kv_slots, pool, qkv, 40, 128)
        assert rel(got, ref) < 2e-2
