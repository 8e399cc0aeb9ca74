#!/usr/bin/env python
"""Benchmark: Orca iteration-level scheduling + selective batching on one GB300.

Workload (the headline configuration): GPT-3 13B shape in bf16 (40 layers,
H=5120, 40 heads, FFN 20480, vocab 50257), random N(0, 0.02) weights, serving
a seeded continuous-batching trace of 1000 requests (Poisson arrivals at 0.5
requests per iteration, prompts U[32,512], outputs U[1,512], max_batch 64,
max_tokens 4096, K/V reserved at 1024 tokens per request).  A "step" is one
scheduler iteration: one pass of the whole hot path over that iteration's
selectively batched mix of initiation and increment requests.

The timed window starts at iteration ``--window-start`` (default 256, when
the batch has saturated at 64 requests); the iterations before it are
scheduled on the host only, and the K/V pool they would have written is
filled with seeded N(0,1) values instead.

value : device-resident -- the plans of the window's iterations (batch
        descriptors + derived tables, built by the C++ scheduler ahead of time:
        output lengths are fixed, so the schedule does not depend on token
        values) sit in HBM before the timed region; increment inputs are the
        previous iteration's device-side outputs.  Timed with CUDA events.
e2e   : the synchronous serving loop through the public C ABI: every step the
        scheduler picks the batch on the host, orca_run_iteration copies the
        descriptor from pinned host memory, runs the iteration and copies the
        next tokens back, and the scheduler appends them.

--impl reference times the CPU oracle (float64 NumPy) on the same workload.
Multi-GPU: the path does not shard; N ranks are N independent replicas, each
with its own trace (seed = rank), no collective on the data path.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from iteration_level_scheduling_gb300 import synth  # noqa: E402

METRIC = "generated tokens/s and ms/iteration at GPT-3 13B shape, 1×GB300, % of roofline"
WORKLOAD = ("gpt3-13b continuous-batching trace: 1000 requests, Poisson 0.5 req/iteration, prompts U[32,512], "
            "outputs U[1,512], max_batch 64, max_tokens 4096, K/V reserve 1024")
MODEL = synth.GPT3_13B
MAX_BATCH, MAX_TOKENS, KV_RESERVE = 64, 4096, 1024


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="orca", choices=["orca", "reference"])
    p.add_argument("--window-start", type=int, default=256)
    p.add_argument("--layers", type=int, default=MODEL.n_layers, help="model depth (40 = the GPT-3 13B shape)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--request-level", action="store_true",
                   help="also time the request-level baseline scheduler on the same trace and engine")
    p.add_argument("--out", default="")
    return p.parse_args()


def profiled_traffic_ratio():
    """DRAM traffic / algorithmic bytes of the GEMM launches in the committed ncu
    capture (profiles/gemm_tc_decode_gpt3_13b.md), or None."""
    try:
        with open(os.path.join(ROOT, "profiles", "gemm_tc_decode_gpt3_13b.md")) as f:
            for line in f:
                if line.startswith("traffic_over_algorithmic:"):
                    return float(line.split(":", 1)[1])
    except (OSError, ValueError):
        pass
    return None


def reduce_replicas(elapsed, tokens, world, device):
    """Replicas run independently; the job's time is the slowest rank's and its
    work is every rank's tokens."""
    if world <= 1:
        return elapsed, tokens
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed, float(tokens)], dtype=torch.float64, device=device)
    mx = t.clone()
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return mx[0].item(), t[1].item()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return dict(hbm=m["hbm_gbs"], tc=m["bf16_tflops"], tc_sus=m["bf16_tflops_sustained"], src="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=6800.0, tc=1900.0, tc_sus=1700.0, src="fallback")


# --------------------------------------------------------------------------- #
# clocks during the timed region
# --------------------------------------------------------------------------- #
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index: str):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                       "-lms", "200", "-i", str(dev_index)], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.f.name)
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[j] for r in rows for j in range(4) if r[5 + j].strip() == "Active"})
        pw = [float(r[3]) for r in rows if r[3].strip().replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(pw) if pw else None}


# --------------------------------------------------------------------------- #
# model set-up on the GPU (weights drawn on the device: 25.7 GB)
# --------------------------------------------------------------------------- #
def gpu_weights(cfg: synth.ModelConfig, seed: int):
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    keep = []

    def mat(*shape):
        t = torch.empty(shape, dtype=torch.bfloat16, device="cuda").normal_(0.0, 0.02, generator=g)
        keep.append(t)
        return t.data_ptr()

    def const(n, v):
        t = torch.full((n,), v, dtype=torch.float32, device="cuda")
        keep.append(t)
        return t.data_ptr()

    H, F = cfg.hidden, cfg.ffn
    layers = []
    for _ in range(cfg.n_layers):
        layers.append(dict(w_qkv=mat(3 * H, H), w_o=mat(H, H), w_1=mat(F, H), w_2=mat(H, F), b_qkv=const(3 * H, 0.0),
                           b_o=const(H, 0.0), b_1=const(F, 0.0), b_2=const(H, 0.0), ln1_g=const(H, 1.0),
                           ln1_b=const(H, 0.0), ln2_g=const(H, 1.0), ln2_b=const(H, 0.0)))
    ptrs = dict(tok_emb=mat(cfg.vocab, H), pos_emb=mat(cfg.max_pos, H), lnf_g=const(H, 1.0), lnf_b=const(H, 0.0),
                layers=layers)
    return keep, ptrs


def fill_kv_pool(eng, seed: int):
    """Seeded N(0,1) contents for every cached K/V slot (stands in for the
    contexts built by the iterations before the window)."""
    import torch
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    lay = eng.kv_layout()
    g = torch.Generator(device="cuda")
    g.manual_seed(1000 + seed)
    per_layer = 2 * lay.n_heads * lay.kv_slots * lay.head_dim
    for l in range(lay.n_layers):
        ptr = lay.base + l * per_layer * lay.elem_bytes
        cai = {"shape": (per_layer,), "typestr": "<i2", "data": (ptr, False), "version": 3, "strides": None}
        holder = type("H", (), {"__cuda_array_interface__": cai})()
        t = torch.as_tensor(holder, device="cuda").view(torch.bfloat16)
        t.normal_(0.0, 1.0, generator=g)
    torch.cuda.synchronize()


def iteration_work(b, cfg: synth.ModelConfig):
    """Algorithmic FLOPs and bytes of one iteration (per-iteration roofline)."""
    n = np.ctypeslib.as_array(b.n_input, (b.n_req,)).astype(np.int64)
    ctx = np.ctypeslib.as_array(b.ctx_len, (b.n_req,)).astype(np.int64)
    R, B, H, F, V, L = int(n.sum()), b.n_req, cfg.hidden, cfg.ffn, cfg.vocab, cfg.n_layers
    pre = n > 1
    pairs = int((n[pre] * ctx[pre] + n[pre] * (n[pre] + 1) // 2).sum()) + int((ctx[~pre] + 1).sum())
    flops = 2.0 * R * L * (4 * H * H + 2 * H * F) + 2.0 * B * H * V + 4.0 * H * pairs * L
    w_bytes = 2.0 * (L * (4 * H * H + 2 * H * F) + V * H) + 2.0 * R * H  # + the position rows used
    kv_bytes = float((ctx + n).sum()) * L * 2 * H * 2
    return dict(B=B, R=R, flops=flops, bytes=w_bytes + kv_bytes, kv_bytes=kv_bytes)


def make_trace(rank: int):
    return synth.poisson_trace(seed=rank, n=1000, rate=0.5, prompt_range=(32, 512), out_range=(1, 512),
                               vocab=MODEL.vocab)


def advance(sched, n_iters: int):
    """Host-only scheduling of n engine iterations (dummy tokens)."""
    done = 0
    while done < n_iters:
        st, b = sched.next_raw()
        if st == 2:
            raise RuntimeError("trace ended before the window")
        if st == 0:
            continue
        sched.complete(np.zeros(b.n_req, np.int32))
        done += 1


# --------------------------------------------------------------------------- #
# the CPU oracle on a bounded sample (baseline / reference arm)
# --------------------------------------------------------------------------- #
class OracleRunner:
    """Times the oracle (float64 NumPy) on one iteration's batch at 13B width
    with ONE layer, and extrapolates: t = t_head + n_layers * (t_1layer - t_head),
    where t_head is the final LayerNorm + LM head on the batch's last rows."""

    def __init__(self, seed: int = 0):
        from oracle import model as omodel
        self.om = omodel
        cfg1 = MODEL.with_layers(1)
        w = synth.make_weights(cfg1, seed)
        f64 = lambda a: np.asarray(a, np.float64)
        self.w = {k: f64(v) for k, v in w.items() if k != "layers"}
        self.w["layers"] = [{k: f64(v) for k, v in L.items()} for L in w["layers"]]
        self.store = omodel.KVStore(1, MODEL.hidden)
        self.seed = seed

    def step(self, rids, ns, ctxs, toks):
        om = self.om
        items, p = [], 0
        for rid, n, c in zip(rids, ns, ctxs):
            tk = [t if t >= 0 else 0 for t in toks[p:p + n]]
            p += n
            have = self.store.length(rid)
            if have != c:  # first sight of a request that entered with a cached context
                self.store.drop(rid)
                if c:
                    k, v = synth.kv_context(self.seed, rid, 0, c, MODEL.hidden, "bf16")
                    self.store.load(rid, 0, k, v)
            items.append(om.BatchItem(rid, tk, c))
        t0 = time.perf_counter()
        r = om.iteration(self.w, MODEL.n_heads, items, self.store)
        t1 = time.perf_counter()
        # head alone: final LN + tied LM head over the B last rows
        x = np.random.default_rng(0).standard_normal((len(items), MODEL.hidden))
        t2 = time.perf_counter()
        y = om.layer_norm(x, self.w["lnf_g"], self.w["lnf_b"])
        lg = y @ self.w["tok_emb"].T
        _ = [om.argmax_lowest(row) for row in lg]
        t3 = time.perf_counter()
        t_head = t3 - t2
        return t_head + MODEL.n_layers * max(t1 - t0 - t_head, 0.0), len(items)


def collect_batches(rank: int, window_start: int, n: int):
    """Batches of the window, scheduled by the C++ scheduler on the host."""
    from iteration_level_scheduling_gb300 import native
    s = native.Scheduler(MAX_BATCH, MAX_TOKENS, kv_slots=MAX_BATCH * KV_RESERVE, kv_reserve=KV_RESERVE)
    for sp in make_trace(rank):
        s.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len)
    advance(s, window_start)
    out = []
    while len(out) < n:
        st, b = s.next()
        if st == 2:
            break
        if st == 0:
            continue
        out.append((b.request_id.tolist(), b.n_input.tolist(), b.ctx_len.tolist(), b.tokens.tolist()))
        s.complete(np.zeros(b.n_req, np.int32))
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return None
    cores = len(os.sched_getaffinity(0))
    batches = collect_batches(0, args.window_start, args.warmup + args.steps)
    runner = OracleRunner(0)
    for b in batches[:args.warmup]:
        runner.step(*b)
    times, toks = [], 0
    for b in batches[args.warmup:args.warmup + args.steps]:
        t, B = runner.step(*b)
        times.append(t)
        toks += B
    total = sum(times)
    value = toks / total
    sample = (f"each step: one iteration of the window at full batch width, 1 of {MODEL.n_layers} layers timed "
              f"(float64 NumPy oracle) plus the LM head, extrapolated to {MODEL.n_layers} layers")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": len(times), "warmup": args.warmup, "ms_per_step": 1000 * total / max(len(times), 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "window_start": args.window_start},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    return line


# --------------------------------------------------------------------------- #
# our arm
# --------------------------------------------------------------------------- #
def request_level_window(args, eng, trace):
    """The request-level baseline (a batch is formed only when the previous one
    has completely finished) on the same trace, engine and device-resident
    path: tokens/s over a window of args.steps iterations from
    args.window_start of its own schedule."""
    import torch

    from iteration_level_scheduling_gb300 import native
    s = native.Scheduler(MAX_BATCH, MAX_TOKENS, kv_reserve=KV_RESERVE, mode=1, engine=eng)
    for sp in trace:
        s.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len)
    advance(s, args.window_start)
    s.set_token_feedback(True)
    n_it = args.warmup + args.steps
    plans, batch = [], []
    while len(plans) < n_it:
        st, b = s.next_raw()
        if st == 2:
            break
        if st == 0:
            continue
        words = native.check(native.lib.orca_plan_words(eng.handle, native.C.byref(b)), "orca_plan_words")
        buf = np.zeros(words, np.int32)
        native.check(native.lib.orca_plan_build(eng.handle, native.C.byref(b), buf.ctypes.data, words),
                     "orca_plan_build")
        plans.append(buf)
        batch.append(int(b.n_req))
        s.complete(np.zeros(b.n_req, np.int32))
    s.close()
    if len(plans) < n_it:
        raise RuntimeError("trace too short for the request-level window")
    offs = np.cumsum([0] + [((p.size + 63) // 64) * 64 for p in plans])
    host_all = np.zeros(int(offs[-1]), np.int32)
    for p, o in zip(plans, offs):
        host_all[o:o + p.size] = p
    dev_all = torch.from_numpy(host_all).cuda()
    base = dev_all.data_ptr()
    for i in range(args.warmup):
        eng.run_planned(plans[i], base + 4 * int(offs[i]))
    eng.sync()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for i in range(args.warmup, n_it):
        eng.run_planned(plans[i], base + 4 * int(offs[i]))
    b.record()
    torch.cuda.synchronize()
    eng.sync()
    ms = a.elapsed_time(b)
    tokens = sum(batch[args.warmup:])
    return {"value": tokens / (ms / 1000.0), "unit": "tokens/s", "ms_per_step": ms / args.steps,
            "mean_batch": float(np.mean(batch[args.warmup:])),
            "scheduler": "request-level: a batch forms only when the previous one has finished"}


def split_by_prefill(work, it_ms, fr):
    """Iterations with only increment rows vs iterations that also carry prompt rows."""
    out = {}
    for name, sel in (("decode_only", lambda w: w["R"] == w["B"]), ("with_prefill", lambda w: w["R"] > w["B"])):
        idx = [i for i, w in enumerate(work) if sel(w)]
        if idx:
            out[name] = {"iterations": len(idx), "mean_ms": float(np.mean([it_ms[i] for i in idx])),
                         "mean_rows": float(np.mean([work[i]["R"] for i in idx])),
                         "mean_frac": float(np.mean([fr[i] for i in idx]))}
    return out


def run_orca(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from iteration_level_scheduling_gb300 import native

    torch.cuda.set_device(local_rank)
    cfg = MODEL.with_layers(args.layers)
    peaks = load_peaks()
    keep, ptrs = gpu_weights(cfg, seed=rank)
    stream = torch.cuda.current_stream().cuda_stream
    eng = native.Engine(cfg.n_layers, cfg.hidden, cfg.n_heads, cfg.ffn, cfg.vocab, cfg.max_pos, native.DTYPE_BF16,
                        MAX_TOKENS, MAX_BATCH, MAX_BATCH * KV_RESERVE, ptrs, stream)
    fill_kv_pool(eng, rank)
    trace = make_trace(rank)

    # ---------------- device-resident window -------------------------------
    s = native.Scheduler(MAX_BATCH, MAX_TOKENS, kv_reserve=KV_RESERVE, engine=eng)
    for sp in trace:
        s.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len)
    advance(s, args.window_start)
    s.set_token_feedback(True)  # from here on, increment inputs are the engine's own previous outputs
    n_it = args.warmup + args.steps
    plans, work = [], []
    while len(plans) < n_it:
        st, b = s.next_raw()
        if st == 2:
            break
        if st == 0:
            continue
        words = native.check(native.lib.orca_plan_words(eng.handle, native.C.byref(b)), "orca_plan_words")
        buf = np.zeros(words, np.int32)
        native.check(native.lib.orca_plan_build(eng.handle, native.C.byref(b), buf.ctypes.data, words),
                     "orca_plan_build")
        plans.append(buf)
        work.append(iteration_work(b, cfg))
        s.complete(np.zeros(b.n_req, np.int32))
    if len(plans) < n_it:
        raise RuntimeError("trace too short for the requested window")
    offs = np.cumsum([0] + [((p.size + 63) // 64) * 64 for p in plans])
    host_all = np.zeros(int(offs[-1]), np.int32)
    for p, o in zip(plans, offs):
        host_all[o:o + p.size] = p
    dev_all = torch.from_numpy(host_all).cuda()
    base = dev_all.data_ptr()
    torch.cuda.synchronize()

    for i in range(args.warmup):
        eng.run_planned(plans[i], base + 4 * int(offs[i]))
    eng.sync()
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    clocks = Clocks(vis.split(",")[local_rank].strip() if vis else str(torch.cuda.current_device()))
    time.sleep(0.3)
    launches0 = eng.stats().launches
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    evs[0].record()
    for j in range(args.steps):
        i = args.warmup + j
        eng.run_planned(plans[i], base + 4 * int(offs[i]))
        evs[j + 1].record()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    launches = eng.stats().launches - launches0
    clk = clocks.stop()
    eng.sync()
    # Per-kernel breakdown: a separate pass over the same plans with CUDA events
    # around every launch of one sampled layer per iteration (events between
    # launches forgo their programmatic-launch overlap, so this pass is not timed).
    eng.timing(True)
    for j in range(args.steps):
        i = args.warmup + j
        eng.run_planned(plans[i], base + 4 * int(offs[i]))
    eng.sync()
    recs = eng.timing_read()
    eng.timing(False)
    it_ms = [evs[j].elapsed_time(evs[j + 1]) for j in range(args.steps)]
    elapsed_ms = evs[0].elapsed_time(evs[-1])
    tokens = sum(w["B"] for w in work[args.warmup:])

    elapsed_ms, tokens = reduce_replicas(elapsed_ms, tokens, world, "cuda")
    value = tokens / (elapsed_ms / 1000.0)

    # per-iteration roofline (tensor peak: sustained, the kernels run inside a long step)
    fr, t_roof_sum = [], 0.0
    for w, t in zip(work[args.warmup:], it_ms):
        t_roof = max(w["flops"] / (peaks["tc_sus"] * 1e12), w["bytes"] / (peaks["hbm"] * 1e9)) * 1000.0
        fr.append(t_roof / t)
        t_roof_sum += t_roof

    # per-kernel breakdown from the engine's events
    # Each record is one launch of the sampled layer (layer >= 0) or a per-iteration
    # kernel (layer == -1); a layer launch stands for n_layers launches of the
    # iteration, so the per-iteration time of a kind is sum(ms * weight) / steps.
    kinds = {}
    for r in recs:
        k = "gemm (all linear layers)" if r["kind"].startswith("gemm") or r["kind"] == "lm_head" else r["kind"]
        wgt = cfg.n_layers if r["layer"] >= 0 else 1
        for key in (k, "lm_head (gemm)") if r["kind"] == "lm_head" else (k,):
            d = kinds.setdefault(key, dict(ms=0.0, bytes=0.0, flops=0.0, n=0, est=0.0))
            d["ms"] += r["ms"]
            d["bytes"] += r["bytes"]
            d["flops"] += r["flops"]
            d["n"] += 1
            d["est"] += r["ms"] * wgt
    est_tot = sum(d["est"] for k, d in kinds.items() if k != "lm_head (gemm)") or 1.0
    breakdown = {k: {"share_of_iteration": d["est"] / est_tot, "est_ms_per_iteration": d["est"] / args.steps,
                     "launches_timed": d["n"], "avg_us": 1000 * d["ms"] / max(d["n"], 1),
                     "GB/s": d["bytes"] / (d["ms"] / 1000) / 1e9 if d["ms"] else None,
                     "TFLOP/s": d["flops"] / (d["ms"] / 1000) / 1e12 if d["ms"] else None}
                 for k, d in sorted(kinds.items(), key=lambda kv: -kv[1]["est"])}
    # the linear layers one by one (sampled-layer launches; lm_head once per iteration)
    gk = {}
    for r in recs:
        if r["kind"].startswith("gemm") or r["kind"] == "lm_head":
            d = gk.setdefault(r["kind"], dict(ms=0.0, bytes=0.0, flops=0.0, n=0))
            d["ms"] += r["ms"]
            d["bytes"] += r["bytes"]
            d["flops"] += r["flops"]
            d["n"] += 1
    gemm_by_kind = {k: {"launches_timed": d["n"], "avg_us": 1000 * d["ms"] / d["n"],
                        "GB/s": d["bytes"] / (d["ms"] / 1000) / 1e9, "TFLOP/s": d["flops"] / (d["ms"] / 1000) / 1e12}
                    for k, d in gk.items() if d["n"] and d["ms"]}
    dom_name, dom = max(((k, d) for k, d in kinds.items() if k != "lm_head (gemm)"), key=lambda kv: kv[1]["est"])
    t_hbm = dom["bytes"] / (peaks["hbm"] * 1e9)
    t_tc = dom["flops"] / (peaks["tc_sus"] * 1e12)
    if t_tc > t_hbm:
        ach = dom["flops"] / (dom["ms"] / 1000) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peaks["tc_sus"], "unit": "TFLOP/s"}
    else:
        ach = dom["bytes"] / (dom["ms"] / 1000) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm"], "unit": "GB/s"}
    ratio = profiled_traffic_ratio() if dom_name.startswith("gemm") else None
    traffic = ratio * dom["bytes"] / dom["n"] if ratio else None
    roof.update({"frac": roof["achieved"] / roof["peak"], "traffic": traffic, "kernel": dom_name,
                 "traffic_source": ("DRAM bytes per launch: algorithmic bytes x the traffic/algorithmic ratio "
                                    "of profiles/gemm_tc_decode_gpt3_13b.md (2-layer capture, decode shapes); "
                                    "the stream-K FFN1 launches of prompt-carrying iterations (about 4 % of the "
                                    "launches) read their weights up to once per token tile "
                                    "(profiles/gemm_sk_prompt_gpt3_13b.md)")
                 if traffic else None,
                 "peak_source": peaks["src"], "launches_timed": dom["n"],
                 "algorithmic_bytes_per_launch": dom["bytes"] / dom["n"],
                 "algorithmic_flops_per_launch": dom["flops"] / dom["n"]})
    s.close()

    # ---------------- end to end through the public API ---------------------
    e2e = None
    if not args.no_e2e:
        s2 = native.Scheduler(MAX_BATCH, MAX_TOKENS, kv_reserve=KV_RESERVE, engine=eng)
        for sp in trace:
            s2.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len)
        advance(s2, args.window_start)
        h2d = d2h = 0
        e2e_tokens = 0

        def step(count):
            nonlocal h2d, d2h, e2e_tokens
            while True:
                st, b = s2.next()
                if st == 1:
                    break
                if st == 2:
                    raise RuntimeError("trace ended")
            nxt = eng.run_iteration(b)
            s2.complete(nxt)
            if count:
                h2d += 4 * eng.plan_words(b)
                d2h += 4 * b.n_req + 4
                e2e_tokens += b.n_req

        for _ in range(args.warmup):
            step(False)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step(True)
        torch.cuda.synchronize()
        e2e_s = time.perf_counter() - t0
        e2e_s, e2e_tokens = reduce_replicas(e2e_s, e2e_tokens, world, "cuda")
        e2e = {"value": e2e_tokens / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d / args.steps,
               "d2h_bytes_per_step": d2h / args.steps, "ms_per_step": 1000 * e2e_s / args.steps}
        s2.close()

    req = None
    if args.request_level and world == 1:
        req = request_level_window(args, eng, trace)
        req["iteration_level_over_request_level"] = value / req["value"]

    # ---------------- CPU oracle on a bounded sample (rank 0, N=1) ----------
    cpu = None
    if not args.no_cpu and rank == 0 and world == 1:
        batches = collect_batches(0, args.window_start + args.warmup, 3)
        runner = OracleRunner(0)
        runner.step(*batches[0])
        ts = [runner.step(*b) for b in batches[1:]]
        t = sum(x[0] for x in ts)
        cpu = {"value": sum(x[1] for x in ts) / t, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
               "kind": "oracle",
               "sample": (f"2 window iterations at full batch width; 1 of {MODEL.n_layers} layers timed "
                          f"(float64 NumPy oracle) plus the LM head, extrapolated to {MODEL.n_layers} layers")}

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "window_start_iteration": args.window_start, "layers": cfg.n_layers,
                   "replicas": world, "l2": "inputs larger than L2 (25.7 GB of weights streamed every iteration)"},
        "iteration_roofline": {"mean_frac": float(np.mean(fr)), "aggregate_frac": t_roof_sum / sum(it_ms),
                               "peaks": {"hbm_GBs": peaks["hbm"], "bf16_TFLOPs_sustained": peaks["tc_sus"],
                                         "source": peaks["src"]},
                               "mean_batch": float(np.mean([w["B"] for w in work[args.warmup:]])),
                               "mean_rows": float(np.mean([w["R"] for w in work[args.warmup:]])),
                               "by_kind": split_by_prefill(work[args.warmup:], it_ms, fr)},
        "roofline": roof, "kernels": breakdown, "gemm_by_kind": gemm_by_kind, "gpu_launches": launches,
        "clocks": clk, "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if req is not None:
        line["request_level"] = req
    del keep
    return line


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            import torch.distributed as dist
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
        line = run_orca(args, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if line is not None and rank == 0:
        s = json.dumps(line)
        print(s, flush=True)
        if args.out:
            with open(args.out, "w") as f:
                f.write(s + "\n")


if __name__ == "__main__":
    main()
