"""Multi-GPU is replicas only: each rank serves its own trace and the job's
number is every rank's tokens over the slowest rank's time.  The aggregation
is checked here with two gloo ranks on the CPU."""

import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    elapsed = [12.5, 20.0][rank]
    tokens = [640, 576][rank]
    e, t = bench.reduce_replicas(elapsed, tokens, world, "cpu")
    out[rank] = (e, t)
    dist.destroy_process_group()


def test_reduce_replicas_two_ranks():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(2):
        assert out[r] == (20.0, 1216.0)  # slowest rank's time, all ranks' tokens


def test_reduce_replicas_single():
    import bench
    assert bench.reduce_replicas(3.0, 7, 1, "cpu") == (3.0, 7)


def test_iteration_work_counts():
    """Per-iteration roofline inputs: FLOPs and weight + K/V bytes of one batch."""
    import bench
    from iteration_level_scheduling_gb300 import synth
    cfg = synth.GPT3_13B
    w = bench.iteration_work([3, 1], [0, 10], cfg)
    H, F, V, L = cfg.hidden, cfg.ffn, cfg.vocab, cfg.n_layers
    assert w["R"] == 4 and w["B"] == 2
    pairs = 3 * 0 + 3 * 4 // 2 + 11  # prefill rows see 1, 2, 3 keys; the decode row sees 11
    assert w["flops"] == 2.0 * 4 * L * (4 * H * H + 2 * H * F) + 2.0 * 2 * H * V + 4.0 * H * pairs * L
    assert w["kv_bytes"] == (3 + 11) * L * 2 * H * 2
    assert w["bytes"] == 2.0 * (L * (4 * H * H + 2 * H * F) + V * H) + 2.0 * 4 * H + w["kv_bytes"]


def test_split_by_prefill():
    """Decode-only vs prompt-carrying iterations: counts, mean times, rows and fractions."""
    import bench
    work = [dict(R=64, B=64), dict(R=300, B=64), dict(R=64, B=64), dict(R=500, B=64)]
    out = bench.split_by_prefill(work, [8.0, 14.0, 10.0, 18.0], [0.8, 0.5, 0.6, 0.4])
    assert out["decode_only"] == {"iterations": 2, "mean_ms": 9.0, "mean_rows": 64.0, "mean_frac": 0.7}
    assert out["with_prefill"]["iterations"] == 2 and out["with_prefill"]["mean_ms"] == 16.0
    assert out["with_prefill"]["mean_rows"] == 400.0 and abs(out["with_prefill"]["mean_frac"] - 0.45) < 1e-12
    assert "with_prefill" not in bench.split_by_prefill(work[:1], [8.0], [0.8])


def test_kernel_breakdown_by_kind_splits_at_embed():
    """Records of three iterations (decode-only, prompt-carrying, decode-only):
    split at each embedding launch and grouped by the iterations' kind."""
    import bench
    def it(prefill):
        r = [dict(kind="embed", layer=-1, ms=0.01, bytes=1.0, flops=0.0),
             dict(kind="gemm_qkv", layer=0, ms=0.04, bytes=1e6, flops=1e9),
             dict(kind="attn_decode", layer=0, ms=0.10, bytes=1e6, flops=0.0)]
        if prefill:
            r.append(dict(kind="attn_prefill", layer=0, ms=0.02, bytes=1e5, flops=1e8))
        return r + [dict(kind="lm_head", layer=-1, ms=0.09, bytes=5e8, flops=1e10)]
    recs = it(False) + it(True) + it(False)
    work = [dict(R=64, B=64), dict(R=400, B=64), dict(R=64, B=64)]
    out = bench.kernel_breakdown_by_kind(recs, work, 40)
    assert set(out) == {"decode_only", "with_prefill"}
    assert "attn_prefill" in out["with_prefill"] and "attn_prefill" not in out["decode_only"]
    assert out["decode_only"]["attn_decode"]["launches_timed"] == 2
    assert abs(out["decode_only"]["attn_decode"]["est_ms_per_iteration"] - 40 * 0.10) < 1e-9
    assert out["with_prefill"]["gemm (all linear layers)"]["launches_timed"] == 2  # QKV and the LM head


def test_gemm_roofline_weights_launches_per_iteration():
    """The linear-layer family's achieved bandwidth weights each sampled-layer
    launch by the model depth and the LM head by one: bytes per iteration over
    GEMM time per iteration, checked against a hand-weighted sum."""
    import bench
    peaks = dict(hbm=6788.3, tc_sus=1731.7)
    L = 40
    recs = []
    for _ in range(2):  # two iterations, one sampled layer each
        recs += [dict(kind="gemm_qkv", layer=3, ms=0.039, bytes=160e6, flops=1e10),
                 dict(kind="gemm_o", layer=3, ms=0.018, bytes=55e6, flops=3e9),
                 dict(kind="gemm_ffn1", layer=3, ms=0.050, bytes=213e6, flops=1.3e10),
                 dict(kind="gemm_ffn2", layer=3, ms=0.043, bytes=215e6, flops=1.3e10),
                 dict(kind="lm_head", layer=-1, ms=0.093, bytes=530e6, flops=3e10),
                 dict(kind="layernorm", layer=3, ms=0.009, bytes=2e6, flops=0.0)]
    tot, kinds = bench.gemm_roofline(recs, L, peaks)
    byts = 2 * (L * (160e6 + 55e6 + 213e6 + 215e6) + 530e6)
    ms = 2 * (L * (0.039 + 0.018 + 0.050 + 0.043) + 0.093)
    assert abs(tot["bytes"] - byts) < 1 and abs(tot["ms"] - ms) < 1e-9
    assert tot["launches"] == 2 * (4 * L + 1)
    frac = byts / (ms / 1000) / 1e9 / peaks["hbm"]
    # the unweighted pooling would give the LM head the weight of one projection
    pooled = 2 * (160e6 + 55e6 + 213e6 + 215e6 + 530e6) / (2 * (0.039 + 0.018 + 0.050 + 0.043 + 0.093) / 1000) / 1e9
    assert abs(tot["bytes"] / (tot["ms"] / 1000) / 1e9 / peaks["hbm"] - frac) < 1e-12
    assert pooled / peaks["hbm"] > frac
    assert kinds["lm_head"]["launches_per_iteration"] == 1 and kinds["gemm_qkv"]["launches_per_iteration"] == L
    assert "layernorm" not in kinds


def test_traffic_record_follows_the_kernel_source(tmp_path, monkeypatch):
    """roofline.traffic comes from a recorded ncu capture only while the GEMM
    source is the one that was captured."""
    import json
    import bench
    src = ["iteration_level_scheduling_gb300/csrc/k_gemm_tc.cu"]
    f = tmp_path / "t.json"
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.traffic_record("gemm_decode")[0] is None
    f.write_text(json.dumps({"gemm_decode": {"sources": src, "source_sha": bench.source_sha(src),
                                             "dram_over_algorithmic": 1.002, "workload": "w"}}))
    rec, why = bench.traffic_record("gemm_decode")
    assert rec["dram_over_algorithmic"] == 1.002 and why is None
    f.write_text(json.dumps({"gemm_decode": {"sources": src, "source_sha": "0" * 16,
                                             "dram_over_algorithmic": 1.002, "workload": "w"}}))
    rec, why = bench.traffic_record("gemm_decode")
    assert rec is None and "changed" in why


def test_trace_phases():
    """Ramp = before the batch first fills, drain = after it is last full."""
    import bench
    B = bench.MAX_BATCH
    work = [dict(B=b) for b in [1, 5, B, B, 30, B, 12, 3]]
    assert bench.phases(work) == {"ramp": [0, 1], "steady": [2, 3, 4, 5], "drain": [6, 7]}


def test_reference_arm_never_loads_the_engine_library():
    """bench.py's reference arm (the oracle on the host) takes its batches from
    the oracle's own scheduler and times the oracle's model: the process never
    maps liborca.so."""
    import subprocess
    import sys
    code = (
        "import bench, numpy as np\n"
        "from iteration_level_scheduling_gb300 import synth\n"
        "b = bench.oracle_window_batches(256, 2)\n"
        "assert len(b) == 2 and all(len(r[0]) == 64 for r in b)\n"
        "cfg = synth.ModelConfig(n_layers=2, hidden=64, n_heads=4, ffn=256, vocab=512, max_pos=2048, dtype='bf16')\n"
        "r = bench.OracleRunner(cfg, 0, np.float32)\n"
        "t, B, m = r.step([1, 2], [3, 1], [0, 5], [7, 8, 9, 10])\n"
        "assert B == 2 and t > 0\n"
        "maps = open('/proc/self/maps').read()\n"
        "print('liborca' in maps)\n")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300,
                         cwd=__file__.rsplit("/", 2)[0])
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip().splitlines()[-1] == "False"


def test_request_latency_on_the_device_timeline():
    """Three iterations of 2, 3 and 5 ms selected at logical clocks 0, 1, 3 (an
    idle tick at 2): request 0 arrives at 0 and runs in iterations 0-1; request
    1 arrives at 1 and runs in 1-2; request 2 arrives at 2 (runs first at clock
    3, iteration 2) and runs in 2 only."""
    import bench
    out = bench.request_latency({0: 0, 1: 1, 2: 2}, {0: 2, 1: 2, 2: 1}, [[0], [0, 1], [1, 2]], [0, 1, 3],
                                [2.0, 3.0, 5.0])
    assert out["requests"] == 3
    lat = sorted([5.0, 8.0, 5.0])  # 0: [0, 5); 1: [2, 10); 2: [5, 10)
    assert abs(out["latency_ms"]["mean"] - sum(lat) / 3) < 1e-12
    assert out["latency_ms"]["p50"] == 5.0
    assert abs(out["queue_ms"]["mean"] - 0.0) < 1e-12  # each runs in the first iteration it may
    assert abs(out["ms_per_output_token"]["mean"] - (2.5 + 4.0 + 5.0) / 3) < 1e-12
