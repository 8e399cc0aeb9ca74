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
    import ctypes as C
    import numpy as np
    import bench
    from iteration_level_scheduling_gb300 import build, synth
    build.build()
    from iteration_level_scheduling_gb300 import native
    cfg = synth.GPT3_13B
    b = native.BatchDesc([1, 2], [0, 1], [3, 1], [0, 10], [0, 100], [5, 6, 7, 8])
    w = bench.iteration_work(b.c, cfg)
    H, F, V, L = cfg.hidden, cfg.ffn, cfg.vocab, cfg.n_layers
    assert w["R"] == 4 and w["B"] == 2
    pairs = 3 * 0 + 3 * 4 // 2 + 11  # prefill rows see 1, 2, 3 keys; the decode row sees 11
    assert w["flops"] == 2.0 * 4 * L * (4 * H * H + 2 * H * F) + 2.0 * 2 * H * V + 4.0 * H * pairs * L
    assert w["kv_bytes"] == (3 + 11) * L * 2 * H * 2


def test_split_by_prefill():
    """Decode-only vs prompt-carrying iterations: counts, mean times, rows and fractions."""
    import bench
    work = [dict(R=64, B=64), dict(R=300, B=64), dict(R=64, B=64), dict(R=500, B=64)]
    out = bench.split_by_prefill(work, [8.0, 14.0, 10.0, 18.0], [0.8, 0.5, 0.6, 0.4])
    assert out["decode_only"] == {"iterations": 2, "mean_ms": 9.0, "mean_rows": 64.0, "mean_frac": 0.7}
    assert out["with_prefill"]["iterations"] == 2 and out["with_prefill"]["mean_ms"] == 16.0
    assert out["with_prefill"]["mean_rows"] == 400.0 and abs(out["with_prefill"]["mean_frac"] - 0.45) < 1e-12
    assert "with_prefill" not in bench.split_by_prefill(work[:1], [8.0], [0.8])


def test_profiled_traffic_ratio_present():
    """bench.py reads roofline.traffic's DRAM/algorithmic ratio from the committed
    decode-GEMM ncu summary; the line must be there and near 1 (no re-reads)."""
    import bench
    r = bench.profiled_traffic_ratio()
    assert r is not None and 0.9 < r < 1.1
