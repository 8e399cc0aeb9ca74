#!/usr/bin/env python
"""Benchmark: Orca iteration-level scheduling + selective batching on one GB300.

Headline workload: GPT-3 13B shape in bf16 (40 layers, H=5120, 40 heads, FFN
20480, vocab 50257), random N(0, 0.02) weights, serving a seeded
continuous-batching trace of 1000 requests (Poisson arrivals at 0.5 requests
per iteration, prompts U[32,512], outputs U[1,512], max_batch 64, max_tokens
4096, K/V reserved at 1024 tokens per request).  A "step" is one scheduler
iteration: one pass of the whole hot path over that iteration's selectively
batched mix of initiation and increment requests.

value     : `--steps` iterations from `--window-start` (the batch has
            saturated at 64 requests there), device-resident: the plans of the
            iterations (batch descriptors + derived tables, built by the C++
            scheduler ahead of time -- output lengths are fixed, so the
            schedule does not depend on token values) sit in HBM before the
            timed region; increment inputs are the previous iteration's
            device-side outputs.  Timed with CUDA events.  The iterations
            before the window are scheduled on the host only and the K/V pool
            they would have written is filled with seeded N(0,1) values.
e2e       : the same window through the public serve loop (orca_sched_run):
            every iteration the scheduler picks the batch on the host,
            orca_run_iteration copies the descriptor from pinned host memory,
            runs the iteration and copies the next tokens back.
full_trace: every iteration of the trace, from the first arrival to the last
            completion (ramp, steady state and drain), device-resident and
            through the serve loop; the per-iteration roofline averaged over
            all of them.
configs   : the other workloads (tiny fp32 trace, GPT-2-medium mixed batch,
            6.7B decode pool, 13B prefill-heavy mix), each with tokens/s,
            ms/iteration, its per-iteration roofline and an oracle CPU baseline.

--impl reference times the CPU oracle (float32 NumPy; the float64 figure is
reported beside it) on the headline workload, with the batches scheduled by
the oracle's own scheduler.
Multi-GPU: the path does not shard; N ranks are N independent replicas, each
with its own trace (seed = rank), no collective on the data path.
"""

from __future__ import annotations

import argparse
import hashlib
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

CFG_WORKLOADS = {
    "tiny-fp32": ("tiny GPT decoder in fp32 (2 layers, H 64, 4 heads, FFN 256, vocab 512): 8 requests with prompts "
                  "U[2,16], outputs [5,50,8,12,40,3,30,7], max_batch 4; iteration-level and request-level"),
    "gpt2-medium-mixed": ("GPT-2-medium shape in bf16 (24 layers, H 1024, 16 heads, FFN 4096, vocab 50257): one mixed "
                          "batch of 3 initiation requests (prompts 128, 64, 256) + 29 increment requests with contexts "
                          "U[1,1024] (sum L = 477)"),
    "gpt3-6.7b-decode": ("GPT-3 6.7B shape in bf16 (32 layers, H 4096, 32 heads, FFN 16384): 128 increment requests with "
                         "contexts U[256,1024], K/V reserve 1280, 256 iterations, finished slots refilled by requests "
                         "with 64-token prompts (remaining outputs U[1,256])"),
    "gpt3-13b-prefill-heavy": ("GPT-3 13B shape in bf16: 50 independent iterations, each 16 initiation requests with "
                               "prompts U[1024,2048] + 128 increment requests with contexts U[128,2048]"),
}

# ncu DRAM counters of the GEMM kernels (written when a capture of the current
# kernels is summarised; checked against the kernels' source hash).
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


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
    p.add_argument("--no-full-trace", action="store_true")
    p.add_argument("--no-request-level", action="store_true",
                   help="skip the padded request-level baseline on the same GPU")
    p.add_argument("--no-window", action="store_true",
                   help="skip the headline window, its serve loop and the whole trace (measure --configs only)")
    p.add_argument("--configs", default="tiny-fp32,gpt2-medium-mixed,gpt3-6.7b-decode,gpt3-13b-prefill-heavy",
                   help="comma-separated list of the other workloads to measure ('' for none)")
    p.add_argument("--prefill-heavy-iters", type=int, default=50)
    p.add_argument("--metrics", default="", help="write one JSON object per iteration of the full trace here")
    p.add_argument("--out", default="")
    return p.parse_args()


def source_sha(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_record(kernel: str):
    """The committed DRAM/algorithmic byte ratio of `kernel`, or (None, reason)."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)[kernel]
    except (OSError, KeyError, ValueError):
        return None, "no ncu capture of this kernel recorded"
    if source_sha(rec["sources"]) != rec["source_sha"]:
        return None, "the kernel changed since its ncu capture"
    return rec, None


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


def clock_device(local_rank):
    import torch
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    return vis.split(",")[local_rank].strip() if vis else str(torch.cuda.current_device())


# --------------------------------------------------------------------------- #
# model set-up on the GPU (weights drawn on the device)
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


def make_engine(cfg, ptrs, max_tokens, max_batch, kv_slots):
    import torch

    from iteration_level_scheduling_gb300 import native
    return native.Engine(cfg.n_layers, cfg.hidden, cfg.n_heads, cfg.ffn, cfg.vocab, cfg.max_pos,
                         native.DTYPE_BF16 if cfg.dtype == "bf16" else native.DTYPE_FP32, max_tokens, max_batch,
                         kv_slots, ptrs, torch.cuda.current_stream().cuda_stream)


def fill_kv_pool(eng, seed: int):
    """Seeded N(0,1) contents for every cached K/V slot (stands in for the
    contexts built by iterations that are not run)."""
    import torch
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


def release_gpu(*objs):
    import gc

    import torch
    for o in objs:
        if hasattr(o, "close"):
            o.close()
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


# --------------------------------------------------------------------------- #
# per-iteration work and roofline
# --------------------------------------------------------------------------- #
def iteration_work(n, ctx, cfg: synth.ModelConfig):
    """Algorithmic FLOPs and bytes of one iteration (per-iteration roofline):
    FLOPs of every linear layer, the LM head and causal attention; bytes of
    every weight read once, the embedding rows used and the K/V read."""
    n = np.asarray(n, np.int64)
    ctx = np.asarray(ctx, np.int64)
    R, B, H, F, V, L = int(n.sum()), len(n), cfg.hidden, cfg.ffn, cfg.vocab, cfg.n_layers
    es = 2 if cfg.dtype == "bf16" else 4
    pre = n > 1
    pairs = int((n[pre] * ctx[pre] + n[pre] * (n[pre] + 1) // 2).sum()) + int((ctx[~pre] + 1).sum())
    flops = 2.0 * R * L * (4 * H * H + 2 * H * F) + 2.0 * B * H * V + 4.0 * H * pairs * L
    w_bytes = es * (L * (4 * H * H + 2 * H * F) + V * H) + es * R * H  # + the position rows used
    kv_bytes = float((ctx + n).sum()) * L * 2 * H * es
    return dict(B=B, R=R, flops=flops, bytes=w_bytes + kv_bytes, kv_bytes=kv_bytes)


def roof_ms(w, peaks):
    return max(w["flops"] / (peaks["tc_sus"] * 1e12), w["bytes"] / (peaks["hbm"] * 1e9)) * 1000.0


def roofline_summary(work, it_ms, peaks):
    fr = [roof_ms(w, peaks) / t for w, t in zip(work, it_ms)]
    return {"mean_frac": float(np.mean(fr)), "aggregate_frac": sum(roof_ms(w, peaks) for w in work) / sum(it_ms),
            "iterations": len(it_ms)}, fr


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


# --------------------------------------------------------------------------- #
# device-resident plans
# --------------------------------------------------------------------------- #
def build_plans(eng, s, n_max=None, record=None):
    """Dry-run scheduler `s` (attached to `eng`) and pack every selected batch
    into a plan.  Returns (plans, [(n_input, ctx_len, n_req)])."""
    from iteration_level_scheduling_gb300 import native
    plans, shapes = [], []
    while n_max is None or len(plans) < n_max:
        st, b = s.next_raw()
        if st == 2:
            break
        if st != 1:
            continue
        words = native.check(native.lib.orca_plan_words(eng.handle, native.C.byref(b)), "orca_plan_words")
        buf = np.zeros(words, np.int32)
        native.check(native.lib.orca_plan_build(eng.handle, native.C.byref(b), buf.ctypes.data, words),
                     "orca_plan_build")
        n = np.ctypeslib.as_array(b.n_input, (b.n_req,)).copy()
        c = np.ctypeslib.as_array(b.ctx_len, (b.n_req,)).copy()
        plans.append(buf)
        shapes.append((n, c))
        if record is not None:
            record(s, b)
        s.complete(np.zeros(b.n_req, np.int32))
    return plans, shapes


class DevicePlans:
    """Every plan of a run copied to the device once (16-byte aligned each)."""

    def __init__(self, plans):
        import torch
        self.plans = plans
        self.offs = np.cumsum([0] + [((p.size + 63) // 64) * 64 for p in plans])
        host = np.zeros(int(self.offs[-1]), np.int32)
        for p, o in zip(plans, self.offs):
            host[o:o + p.size] = p
        self.dev = torch.from_numpy(host).cuda()
        self.base = self.dev.data_ptr()
        torch.cuda.synchronize()

    def run(self, eng, i):
        eng.run_planned(self.plans[i], self.base + 4 * int(self.offs[i]))


def timed_run(eng, dp, first, count):
    """Run plans first .. first+count-1 with an event after each; returns the
    per-iteration times (ms) and the launches issued."""
    import torch
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(count + 1)]
    l0 = eng.stats().launches
    torch.cuda.synchronize()
    evs[0].record()
    for j in range(count):
        dp.run(eng, first + j)
        evs[j + 1].record()
    torch.cuda.synchronize()
    eng.sync()
    return [evs[j].elapsed_time(evs[j + 1]) for j in range(count)], eng.stats().launches - l0


# --------------------------------------------------------------------------- #
# GEMM family roofline from the engine's per-launch events
# --------------------------------------------------------------------------- #
GEMM_KINDS = ("gemm_qkv", "gemm_o", "gemm_ffn1", "gemm_ffn2", "lm_head")


def gemm_roofline(recs, n_layers, peaks):
    """The linear layers as one kernel family.  Every record is one event-timed
    launch of the sampled layer (standing for n_layers launches per iteration)
    or of the LM head (once per iteration); bytes, flops and time are weighted
    by launches per iteration before the ratio is taken."""
    by_kind, tot = {}, dict(bytes=0.0, flops=0.0, ms=0.0, launches=0.0)
    for r in recs:
        if r["kind"] not in GEMM_KINDS:
            continue
        wgt = n_layers if r["layer"] >= 0 else 1
        d = by_kind.setdefault(r["kind"], dict(ms=0.0, bytes=0.0, flops=0.0, n=0, wgt=wgt))
        d["ms"] += r["ms"]
        d["bytes"] += r["bytes"]
        d["flops"] += r["flops"]
        d["n"] += 1
        tot["bytes"] += r["bytes"] * wgt
        tot["flops"] += r["flops"] * wgt
        tot["ms"] += r["ms"] * wgt
        tot["launches"] += wgt
    kinds = {k: {"launches_timed": d["n"], "launches_per_iteration": d["wgt"], "avg_us": 1000 * d["ms"] / d["n"],
                 "GB/s": d["bytes"] / (d["ms"] / 1000) / 1e9, "TFLOP/s": d["flops"] / (d["ms"] / 1000) / 1e12,
                 "frac_of_hbm": d["bytes"] / (d["ms"] / 1000) / 1e9 / peaks["hbm"]}
             for k, d in by_kind.items() if d["n"] and d["ms"]}
    return tot, kinds


def kernel_breakdown(recs, n_layers, steps):
    kinds = {}
    for r in recs:
        k = "gemm (all linear layers)" if r["kind"] in GEMM_KINDS else r["kind"]
        wgt = n_layers if r["layer"] >= 0 else 1
        d = kinds.setdefault(k, dict(ms=0.0, bytes=0.0, flops=0.0, n=0, est=0.0))
        d["ms"] += r["ms"]
        d["bytes"] += r["bytes"]
        d["flops"] += r["flops"]
        d["n"] += 1
        d["est"] += r["ms"] * wgt
    tot = sum(d["est"] for d in kinds.values()) or 1.0
    return {k: {"share_of_iteration": d["est"] / tot, "est_ms_per_iteration": d["est"] / steps,
                "launches_timed": d["n"], "avg_us": 1000 * d["ms"] / max(d["n"], 1),
                "GB/s": d["bytes"] / (d["ms"] / 1000) / 1e9 if d["ms"] else None,
                "TFLOP/s": d["flops"] / (d["ms"] / 1000) / 1e12 if d["ms"] else None}
            for k, d in sorted(kinds.items(), key=lambda kv: -kv[1]["est"])}


def kernel_breakdown_by_kind(recs, work, n_layers):
    """kernel_breakdown for decode-only and prompt-carrying iterations apart: the
    records split into iterations at each embedding launch (the first of an
    iteration), `work` giving each iteration's rows."""
    its, cur = [], None
    for r in recs:
        if r["kind"] == "embed":
            cur = []
            its.append(cur)
        if cur is not None:
            cur.append(r)
    out = {}
    for name, sel in (("decode_only", lambda w: w["R"] == w["B"]), ("with_prefill", lambda w: w["R"] > w["B"])):
        idx = [i for i, w in enumerate(work[:len(its)]) if sel(w)]
        if idx:
            out[name] = kernel_breakdown([r for i in idx for r in its[i]], n_layers, len(idx))
    return out


def per_kernel_pass(eng, dp, first, count):
    """The same plans again with CUDA events around every launch of one sampled
    layer per iteration and the per-iteration kernels (events between launches
    forgo their programmatic-launch overlap, so this pass is not the timed one)."""
    eng.timing(True)
    for j in range(count):
        dp.run(eng, first + j)
    eng.sync()
    recs = eng.timing_read()
    eng.timing(False)
    return recs


# --------------------------------------------------------------------------- #
# the CPU oracle (baseline / reference arm)
# --------------------------------------------------------------------------- #
class OracleRunner:
    """Times the oracle (float32 NumPy, or float64) on one iteration's batch at
    full width with ONE layer plus the final LayerNorm and LM head, and
    extrapolates to the model's depth: t = t_head + n_layers * t_layer."""

    def __init__(self, cfg: synth.ModelConfig, seed: int = 0, dtype=np.float32):
        from oracle import model as omodel
        self.om, self.cfg, self.dtype, self.seed = omodel, cfg, dtype, seed
        w = synth.make_weights(cfg.with_layers(1), seed)
        f = lambda a: np.asarray(a, dtype)
        self.w = {k: f(v) for k, v in w.items() if k != "layers"}
        self.w["layers"] = [{k: f(v) for k, v in L.items()} for L in w["layers"]]
        self.store = omodel.KVStore(1, cfg.hidden, dtype)

    def step(self, rids, ns, ctxs, toks):
        """Returns (extrapolated seconds for the whole iteration, requests, measured seconds)."""
        om, cfg = self.om, self.cfg
        items, p = [], 0
        for rid, n, c in zip(rids, ns, ctxs):
            tk = [t if t >= 0 else 0 for t in toks[p:p + n]]
            p += n
            if self.store.length(rid) != c:  # first sight of a request that entered with a cached context
                self.store.drop(rid)
                if c:
                    k, v = synth.kv_context(self.seed, rid, 0, c, cfg.hidden, cfg.dtype)
                    self.store.load(rid, 0, k, v)
            items.append(om.BatchItem(rid, tk, c))
        t0 = time.perf_counter()
        om.iteration(self.w, cfg.n_heads, items, self.store, hidden_only=True, dtype=self.dtype)
        t1 = time.perf_counter()
        x = np.random.default_rng(0).standard_normal((len(items), cfg.hidden)).astype(self.dtype)
        t2 = time.perf_counter()
        y = om.layer_norm(x, self.w["lnf_g"], self.w["lnf_b"], dtype=self.dtype)
        lg = y @ self.w["tok_emb"].T
        _ = [om.argmax_lowest(row) for row in lg]
        t3 = time.perf_counter()
        t_head = t3 - t2
        return t_head + cfg.n_layers * (t1 - t0), len(items), (t1 - t0) + t_head


def cpu_line(runner, batches, what):
    runner.step(*batches[0])  # first sight: loads contexts, warms BLAS
    ts = [runner.step(*b) for b in batches[1:]] if len(batches) > 1 else [runner.step(*batches[0])]
    t = sum(x[0] for x in ts)
    return {"value": sum(x[1] for x in ts) / t, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle", "dtype": np.dtype(runner.dtype).name,
            "extrapolated_ms_per_iteration": 1000 * t / len(ts),
            "measured_ms_per_sample": 1000 * sum(x[2] for x in ts) / len(ts),
            "sample": (f"{what}; per iteration 1 of {runner.cfg.n_layers} layers and the LM head timed at full batch "
                       f"width ({np.dtype(runner.dtype).name} NumPy oracle), extrapolated to "
                       f"{runner.cfg.n_layers} layers")}


def one_thread_sample(window_start: int):
    """tokens/s of the same oracle sample with one BLAS thread: a child process
    started with single-thread BLAS (the thread count is fixed when NumPy
    loads), timing the second of two window iterations; None if it fails."""
    code = ("import json, numpy as np, bench\n"
            f"b = bench.oracle_window_batches({window_start}, 2)\n"
            "r = bench.OracleRunner(bench.MODEL, 0, np.float32)\n"
            "r.step(*b[0])\n"
            "t, B, m = r.step(*b[1])\n"
            "print(json.dumps({'value': B / t, 'measured_ms_per_sample': 1000 * m}))\n")
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    try:
        out = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT, capture_output=True, text=True,
                             timeout=600)
        return json.loads(out.stdout.strip().splitlines()[-1]) if out.returncode == 0 else None
    except (subprocess.TimeoutExpired, ValueError, IndexError):
        return None


def oracle_window_batches(window_start: int, n: int):
    """Batches of the headline window, scheduled by the oracle's scheduler."""
    from oracle import sched as osched
    s = osched.Scheduler(MAX_BATCH, MAX_TOKENS, kv_slots=MAX_BATCH * KV_RESERVE, kv_reserve=KV_RESERVE)
    for sp in make_trace(0):
        s.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len, sp.ctx0)
    out, done = [], 0
    while len(out) < n and s.unfinished():
        batch = s.select()
        if not batch:
            s.idle()
            continue
        it = s.describe(batch)
        if done >= window_start:  # engine iterations, as the native window counts them (idle ticks excluded)
            out.append((it.rids, it.n_input, it.ctx, it.tokens))
        s.complete(batch, [0] * len(batch))
        done += 1
    return out


def make_trace(rank: int):
    return synth.poisson_trace(seed=rank, n=1000, rate=0.5, prompt_range=(32, 512), out_range=(1, 512),
                               vocab=MODEL.vocab)


def run_reference(args, rank, world):
    if rank != 0:
        return None
    cores = len(os.sched_getaffinity(0))
    batches = oracle_window_batches(args.window_start, args.warmup + args.steps)
    runner = OracleRunner(MODEL, 0, np.float32)
    t_start = time.perf_counter()
    for b in batches[:args.warmup]:
        runner.step(*b)
    ext, toks, meas = 0.0, 0, 0.0
    for b in batches[args.warmup:]:
        t, B, m = runner.step(*b)
        ext += t
        toks += B
        meas += m
    steps = len(batches) - args.warmup
    value = toks / ext
    # the same samples once in float64 (the precision every parity test uses)
    r64 = OracleRunner(MODEL, 0, np.float64)
    r64.step(*batches[args.warmup])
    t64, b64, _ = r64.step(*batches[args.warmup])
    sample = (f"each step: one iteration of the window at full batch width, 1 of {MODEL.n_layers} layers and the "
              f"LM head timed (float32 NumPy oracle; batches from the oracle's scheduler); tokens/s extrapolates "
              f"the layer to {MODEL.n_layers} layers")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": steps, "warmup": args.warmup, "ms_per_step": 1000 * meas / max(steps, 1),
            "extrapolated_ms_per_iteration": 1000 * ext / max(steps, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "window_start_iteration": args.window_start},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample,
                             "f64_value": b64 / t64},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": time.perf_counter() - t_start}
    return line


# --------------------------------------------------------------------------- #
# the headline window and the whole trace
# --------------------------------------------------------------------------- #
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


def window_scheduler(eng, trace, window_start):
    from iteration_level_scheduling_gb300 import native
    s = native.Scheduler(MAX_BATCH, MAX_TOKENS, kv_reserve=KV_RESERVE, engine=eng)
    for sp in trace:
        s.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len)
    advance(s, window_start)
    return s


def serve_loop_e2e(eng, s, warmup, steps, plan_words, world):
    """`steps` iterations through the public serve loop (orca_sched_run) after
    `warmup` of them; returns the e2e block."""
    import torch
    s.run(warmup)
    g0 = s.stats().generated
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    t0 = time.perf_counter()
    s.run(steps)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    tokens = s.stats().generated - g0
    return dt, tokens


def phases(work):
    """Ramp (before the batch first fills), steady, drain (after it last is full)."""
    full = [i for i, w in enumerate(work) if w["B"] == MAX_BATCH]
    if not full:
        return {"all": list(range(len(work)))}
    a, b = full[0], full[-1]
    return {"ramp": list(range(0, a)), "steady": list(range(a, b + 1)), "drain": list(range(b + 1, len(work)))}


def request_latency(arrival, out_len, ids_per_it, sel_clock, it_ms):
    """Per-request latency on the device timeline of a run whose iterations took
    it_ms back to back: from the start of the first iteration selected at or
    after the request's arrival (logical clock; sel_clock[i] is iteration i's,
    nondecreasing) to the end of the iteration that made its last token;
    queueing until the start of its own first iteration; and latency per output
    token.  Mean and 50/90/99th percentiles, in ms."""
    t = np.concatenate([[0.0], np.cumsum(np.asarray(it_ms, np.float64))])
    first, last = {}, {}
    for i, ids in enumerate(ids_per_it):
        for r in ids:
            first.setdefault(int(r), i)
            last[int(r)] = i
    sel = np.asarray(sel_clock)
    lat, queue, per_tok = [], [], []
    for r, a in arrival.items():
        if r not in last:
            continue
        k = int(np.searchsorted(sel, a, side="left"))
        lat.append(t[last[r] + 1] - t[k])
        queue.append(t[first[r]] - t[k])
        per_tok.append(lat[-1] / out_len[r])

    def pct(v):
        return {"mean": float(np.mean(v)), "p50": float(np.percentile(v, 50)), "p90": float(np.percentile(v, 90)),
                "p99": float(np.percentile(v, 99))}
    return {"requests": len(lat), "latency_ms": pct(lat), "queue_ms": pct(queue),
            "ms_per_output_token": pct(per_tok)}


def run_full_trace(args, eng, trace, cfg, peaks):
    import torch

    from iteration_level_scheduling_gb300 import native
    s = native.Scheduler(MAX_BATCH, MAX_TOKENS, kv_reserve=KV_RESERVE, engine=eng, token_feedback=True)
    for sp in trace:
        s.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len)
    meta = []

    def rec(sched, b):
        st = sched.stats()
        # (the clock has already advanced past this iteration's selection)
        meta.append(dict(clock=st.clock, waiting=st.waiting, kv_reserved=st.kv_reserved,
                         ids=np.ctypeslib.as_array(b.request_id, (b.n_req,)).copy()))

    t0 = time.perf_counter()
    plans, shapes = build_plans(eng, s, record=rec)
    host_plan_s = time.perf_counter() - t0
    s.close()
    work = [iteration_work(n, c, cfg) for n, c in shapes]
    dp = DevicePlans(plans)
    clocks = Clocks(clock_device(int(os.environ.get("LOCAL_RANK", "0"))))
    time.sleep(0.3)
    it_ms, launches = timed_run(eng, dp, 0, len(plans))
    clk = clocks.stop()
    tokens = sum(w["B"] for w in work)
    total_ms = sum(it_ms)
    roof, fr = roofline_summary(work, it_ms, peaks)
    by_phase = {}
    for name, idx in phases(work).items():
        if idx:
            by_phase[name] = {"iterations": len(idx), "mean_ms": float(np.mean([it_ms[i] for i in idx])),
                              "mean_batch": float(np.mean([work[i]["B"] for i in idx])),
                              "mean_frac": float(np.mean([fr[i] for i in idx])),
                              "aggregate_frac": sum(roof_ms(work[i], peaks) for i in idx) / sum(it_ms[i] for i in idx)}
    block = {"iterations": len(plans), "tokens": tokens, "value": tokens / (total_ms / 1000), "unit": "tokens/s",
             "ms_per_iteration": total_ms / len(plans), "total_s": total_ms / 1000, "gpu_launches": launches,
             "iteration_roofline": dict(roof, by_phase=by_phase, by_kind=split_by_prefill(work, it_ms, fr)),
             "slots_busy": tokens / (len(plans) * MAX_BATCH), "clocks": clk,
             "host_plan_build_us_per_iteration": 1e6 * host_plan_s / len(plans),
             "request_latency": request_latency({sp.rid: sp.arrival for sp in trace},
                                                {sp.rid: sp.out_len for sp in trace},
                                                [m["ids"] for m in meta], [m["clock"] - 1 for m in meta], it_ms)}
    if args.metrics:
        with open(args.metrics, "w") as f:
            for i, (w, m) in enumerate(zip(work, meta)):
                n, c = shapes[i]
                f.write(json.dumps({"iteration": i, "clock": m["clock"], "B": w["B"], "rows": w["R"],
                                    "initiation": int((c == 0).sum()), "increment": int((c > 0).sum()),
                                    "queue": m["waiting"], "kv_reserved": m["kv_reserved"],
                                    "kv_used": int((c + n).sum()), "ms": it_ms[i],
                                    "roofline_frac": fr[i]}) + "\n")
    del dp
    torch.cuda.synchronize()
    if not args.no_e2e:
        s2 = native.Scheduler(MAX_BATCH, MAX_TOKENS, kv_reserve=KV_RESERVE, engine=eng)
        for sp in trace:
            s2.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        s2.run()
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        st = s2.stats()
        s2.close()
        h2d = 4.0 * sum(p.size for p in plans)
        d2h = 4.0 * sum(w["B"] + 1 for w in work)
        block["e2e"] = {"value": st.generated / dt, "unit": "tokens/s", "iterations": int(st.iterations),
                        "ms_per_iteration": 1000 * dt / max(st.iterations, 1),
                        "host_overhead_us_per_iteration": 1000 * (dt * 1000 - total_ms) / max(st.iterations, 1),
                        "h2d_bytes_per_step": h2d / len(plans), "d2h_bytes_per_step": d2h / len(plans)}
    return block


# --------------------------------------------------------------------------- #
# the conventional baseline on the same GPU: request-level, padded + masked
# --------------------------------------------------------------------------- #
def run_request_level_padded(args, ptrs, cfg, peaks, trace):
    """The baseline the pages compare Orca with, on the same engine, model and
    trace: request-level batches ([0h-n0] "Request-Level vs Iteration-Level
    Scheduling": a batch forms only when the previous one has finished and runs
    until its longest member is done) executed as conventional padded + masked
    batches ([houmin] 3.1.2 "问题"): prompts padded to the longest of the batch,
    finished members kept in the batch as pad rows, increments attending over
    the batch's longest context with the rest masked (orca_plan_build_padded).
    Device-resident plans over `--steps` iterations from `--window-start` of its
    own schedule; tokens/s counts the real requests' tokens only."""
    import torch

    from iteration_level_scheduling_gb300 import native
    eng = make_engine(cfg, ptrs, MAX_BATCH * 512, MAX_BATCH, MAX_BATCH * KV_RESERVE)  # 64 prompts padded to <= 512
    fill_kv_pool(eng, 0)
    s = native.Scheduler(MAX_BATCH, MAX_TOKENS, kv_reserve=KV_RESERVE, mode=1, engine=eng)
    for sp in trace:
        s.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len)
    members, ctx, kv = [], {}, {}
    plans, work, real_tokens, rows = [], [], [], []
    n_it, done = args.warmup + args.steps, 0
    while len(plans) < n_it:
        st, b = s.next_raw()
        if st == 2:
            break
        if st != 1:
            continue
        B = b.n_req
        ids = np.ctypeslib.as_array(b.request_id, (B,)).tolist()
        n = np.ctypeslib.as_array(b.n_input, (B,)).tolist()
        c = np.ctypeslib.as_array(b.ctx_len, (B,)).tolist()
        ph = np.ctypeslib.as_array(b.phase, (B,)).tolist()
        if all(p == 0 for p in ph):  # a new batch
            members = ids
        for r, o in zip(ids, np.ctypeslib.as_array(b.kv_offset, (B,)).tolist()):
            kv[r] = o
        real = {r: i for i, r in enumerate(ids)}
        if done >= args.window_start:
            toks = np.ctypeslib.as_array(b.tokens, (sum(n),)).tolist()
            off = np.concatenate([[0], np.cumsum(n)]).tolist()
            d = dict(rid=[], ph=[], n=[], c=[], kv=[], tok=[])
            for r in members:
                i = real.get(r)
                ghost = i is None  # finished: a pad row after its own context
                d["rid"].append(r), d["ph"].append(1 if ghost else ph[i]), d["n"].append(1 if ghost else n[i])
                d["c"].append(ctx[r] if ghost else c[i]), d["kv"].append(kv[r])
                d["tok"].extend([0] if ghost else [t if t >= 0 else 0 for t in toks[off[i]:off[i + 1]]])
            desc = native.BatchDesc(d["rid"], d["ph"], d["n"], d["c"], d["kv"], d["tok"])
            buf = np.zeros(eng.plan_words(desc, padded=True), np.int32)
            eng.plan_build(desc, buf, padded=True)
            plans.append(buf)
            work.append(iteration_work(n, c, cfg))
            real_tokens.append(B)
            rows.append((max(d["n"]) * len(d["rid"]), sum(n)))
        for r in members:
            i = real.get(r)
            ctx[r] = (ctx[r] + 1) if i is None else c[i] + n[i]
        s.complete(np.zeros(B, np.int32))
        done += 1
    s.close()
    if len(plans) < n_it:
        raise RuntimeError("trace too short for the request-level window")
    dp = DevicePlans(plans)
    timed_run(eng, dp, 0, args.warmup)
    it_ms, launches = timed_run(eng, dp, args.warmup, args.steps)
    eng.close()
    del dp
    torch.cuda.synchronize()
    tot = sum(it_ms)
    tokens = sum(real_tokens[args.warmup:])
    padded = sum(r[0] for r in rows[args.warmup:])
    useful = sum(r[1] for r in rows[args.warmup:])
    return {"value": tokens / (tot / 1000), "unit": "tokens/s", "ms_per_iteration": tot / args.steps,
            "iterations_timed": args.steps, "window_start_iteration": args.window_start,
            "mean_real_batch": float(np.mean(real_tokens[args.warmup:])),
            "rows_computed_over_real_rows": padded / useful, "gpu_launches": launches,
            "scheduler": "request-level (a batch forms when the previous one has finished), padded + masked "
                         "batches (orca_plan_build_padded)"}


# --------------------------------------------------------------------------- #
# the other workloads
# --------------------------------------------------------------------------- #
def cfg_block(work, it_ms, peaks, launches, extra=None):
    roof, fr = roofline_summary(work, it_ms, peaks)
    total = sum(it_ms)
    tok = sum(w["B"] for w in work)
    out = {"value": tok / (total / 1000), "unit": "tokens/s", "ms_per_iteration": total / len(it_ms),
           "iterations_timed": len(it_ms), "gpu_launches": launches,
           "iteration_roofline": dict(roof, by_kind=split_by_prefill(work, it_ms, fr),
                                      bound=("tensor" if np.mean([w["flops"] / (peaks["tc_sus"] * 1e12) >
                                                                  w["bytes"] / (peaks["hbm"] * 1e9) for w in work])
                                             > 0.5 else "hbm"))}
    if extra:
        out.update(extra)
    return out


def run_tiny(args, peaks, do_cpu):
    """Tiny fp32 config through the public serve loop: iteration-level (50
    iterations) and request-level (90) on the pages' 8-request example."""
    import torch

    from iteration_level_scheduling_gb300 import native
    cfg = synth.TINY
    w = synth.make_weights(cfg, 0)
    keep = []

    def dev(a):
        t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
        keep.append(t)
        return t.data_ptr()

    ptrs = {"tok_emb": dev(w["tok_emb"]), "pos_emb": dev(w["pos_emb"]), "lnf_g": dev(w["lnf_g"]),
            "lnf_b": dev(w["lnf_b"]), "layers": [{k: dev(v) for k, v in L.items()} for L in w["layers"]]}
    out = {"workload": CFG_WORKLOADS["tiny-fp32"], "dtype": "f32"}
    for name, mode in (("iteration_level", 0), ("request_level", 1)):
        eng = make_engine(cfg, ptrs, 4096, 4, 4 * 128)
        best = None
        for _ in range(3):
            s = native.Scheduler(4, 4096, mode=mode, engine=eng)
            for sp in synth.tiny_requests(0):
                s.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            s.run()
            dt = time.perf_counter() - t0
            st = s.stats()
            s.close()
            best = dt if best is None else min(best, dt)
        out[name] = {"iterations": int(st.iterations), "generated": int(st.generated),
                     "e2e_tokens_per_s": st.generated / best, "ms_per_iteration": 1000 * best / st.iterations,
                     "slots_busy": st.generated / (st.iterations * 4)}
        eng.close()
    out["iteration_over_request_level"] = out["iteration_level"]["e2e_tokens_per_s"] / out["request_level"]["e2e_tokens_per_s"]
    if do_cpu:
        from oracle import model as omodel
        from oracle import sched as osched
        w64 = {k: np.asarray(v, np.float32) for k, v in w.items() if k != "layers"}
        w64["layers"] = [{k: np.asarray(v, np.float32) for k, v in L.items()} for L in w["layers"]]
        store = omodel.KVStore(cfg.n_layers, cfg.hidden, np.float32)

        def tok_fn(it):
            items = [omodel.BatchItem(r, it.tokens[o:o + n], c)
                     for r, n, c, o in zip(it.rids, it.n_input, it.ctx, it.offsets)]
            return omodel.iteration(w64, cfg.n_heads, items, store, dtype=np.float32).next_tokens

        t0 = time.perf_counter()
        s, recs = osched.run(synth.tiny_requests(0), 4, 4096, 4 * 128, token_fn=tok_fn)
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = {"value": s.generated_total / dt, "unit": "tokens/s",
                               "cores": len(os.sched_getaffinity(0)), "kind": "oracle", "dtype": "float32",
                               "sample": "the whole iteration-level trace (50 iterations, full depth)"}
    del keep
    return out


def run_gpt2_mixed(args, peaks, do_cpu):
    import torch

    from iteration_level_scheduling_gb300 import native
    cfg = synth.GPT2_MEDIUM
    keep, ptrs = gpu_weights(cfg, 0)
    reqs = synth.mixed_batch(0)
    rows = sum(len(r.prompt) for r in reqs)
    reserve = [r.ctx0 + len(r.prompt) + 8 for r in reqs]
    eng = make_engine(cfg, ptrs, rows, len(reqs), sum(reserve))
    offs = [eng.kv_alloc(r.rid, n) for r, n in zip(reqs, reserve)]
    fill_kv_pool(eng, 0)
    b = native.BatchDesc([r.rid for r in reqs], [1 if r.ctx0 else 0 for r in reqs], [len(r.prompt) for r in reqs],
                         [r.ctx0 for r in reqs], offs, [t for r in reqs for t in r.prompt])
    W, K = max(args.warmup, 3), max(args.steps, 20)
    plans = []
    for _ in range(W + K):  # the same iteration again and again (its K/V writes are idempotent)
        buf = np.zeros(eng.plan_words(b), np.int32)
        eng.plan_build(b, buf)
        plans.append(buf)
    dp = DevicePlans(plans)
    timed_run(eng, dp, 0, W)
    it_ms, launches = timed_run(eng, dp, W, K)
    w = iteration_work(b.n_input, b.ctx_len, cfg)
    out = cfg_block([w] * K, it_ms, peaks, launches, {"workload": CFG_WORKLOADS["gpt2-medium-mixed"],
                                                     "rows": int(rows), "requests": len(reqs)})
    out["kernels"] = kernel_breakdown(per_kernel_pass(eng, dp, W, min(K, cfg.n_layers)), cfg.n_layers,
                                      min(K, cfg.n_layers))
    release_gpu(eng)
    del dp, keep
    release_gpu()
    if do_cpu:
        runner = OracleRunner(cfg, 0, np.float32)
        batch = ([r.rid for r in reqs], [len(r.prompt) for r in reqs], [r.ctx0 for r in reqs],
                 [t for r in reqs for t in r.prompt])
        out["cpu_baseline"] = cpu_line(runner, [batch], "the mixed batch")
    return out


def run_gpt3_decode(args, peaks, do_cpu):
    from iteration_level_scheduling_gb300 import native
    cfg = synth.GPT3_6_7B
    B, reserve = 128, 1280
    keep, ptrs = gpu_weights(cfg, 0)
    eng = make_engine(cfg, ptrs, 4096, B, B * reserve)
    s = native.Scheduler(B, 4096, kv_reserve=reserve, engine=eng, token_feedback=True)
    specs = synth.decode_pool(0, n_running=B, ctx_range=(256, 1024), remaining_range=(1, 256), n_refill=4096,
                              refill_prompt=64, vocab=cfg.vocab)
    for sp in specs:
        s.submit(sp.rid, sp.arrival, sp.prompt, sp.out_len, sp.ctx0)
    fill_kv_pool(eng, 0)
    W, K = max(args.warmup, 3), 256
    plans, shapes = build_plans(eng, s, n_max=W + K)
    s.close()
    dp = DevicePlans(plans)
    timed_run(eng, dp, 0, W)
    it_ms, launches = timed_run(eng, dp, W, K)
    work = [iteration_work(n, c, cfg) for n, c in shapes[W:]]
    out = cfg_block(work, it_ms, peaks, launches, {"workload": CFG_WORKLOADS["gpt3-6.7b-decode"]})
    try:  # (a replayed plan must follow one of the same batch size)
        out["kernels"] = kernel_breakdown(per_kernel_pass(eng, dp, W, cfg.n_layers), cfg.n_layers, cfg.n_layers)
    except native.OrcaError as e:
        out["kernels"] = {"unavailable": str(e)}
    release_gpu(eng)
    del dp, keep
    release_gpu()
    if do_cpu:
        runner = OracleRunner(cfg, 0, np.float32)
        sp = specs[:B]
        batch = ([r.rid for r in sp], [1] * B, [r.ctx0 for r in sp], [r.prompt[0] for r in sp])
        out["cpu_baseline"] = cpu_line(runner, [batch], "the first iteration (128 increment requests)")
    return out


def run_gpt3_prefill_heavy(args, peaks, do_cpu, cfg, ptrs13):
    """`cfg` is the 13B shape at the depth of the weights `ptrs13` (40 layers
    unless --layers says otherwise, e.g. for a small profiler capture)."""
    from iteration_level_scheduling_gb300 import native
    n_it = max(1, args.prefill_heavy_iters)
    W = 3
    draws = [synth.prefill_heavy_batch(seed=i % n_it, vocab=cfg.vocab) for i in range(n_it)]
    need = [[r.ctx0 + len(r.prompt) + 50 for r in d] for d in draws]
    rows = [sum(len(r.prompt) for r in d) for d in draws]
    eng = make_engine(cfg, ptrs13, max(rows), max(len(d) for d in draws), max(sum(n) for n in need))
    fill_kv_pool(eng, 5)
    plans, work = [], []
    for j in range(W + n_it):  # the first W are warm-up copies of the first draws
        i = j % n_it
        d = draws[i]
        ids = [1_000_000 * (j + 1) + r.rid for r in d]
        offs = [eng.kv_alloc(rid, n) for rid, n in zip(ids, need[i])]
        b = native.BatchDesc(ids, [1 if r.ctx0 else 0 for r in d], [len(r.prompt) for r in d],
                             [r.ctx0 for r in d], offs, [t for r in d for t in r.prompt])
        buf = np.zeros(eng.plan_words(b), np.int32)
        eng.plan_build(b, buf)
        for rid in ids:
            eng.kv_free(rid)
        plans.append(buf)
        if j >= W:
            work.append(iteration_work(b.n_input, b.ctx_len, cfg))
    dp = DevicePlans(plans)
    timed_run(eng, dp, 0, W)
    it_ms, launches = timed_run(eng, dp, W, n_it)
    out = cfg_block(work, it_ms, peaks, launches, {"workload": CFG_WORKLOADS["gpt3-13b-prefill-heavy"],
                                                  "mean_rows": float(np.mean(rows)), "layers": cfg.n_layers})
    # the linear layers of one iteration, event-timed per launch (tensor-pipe bound)
    recs = per_kernel_pass(eng, dp, W, min(n_it, 3))
    out["kernels"] = kernel_breakdown(recs, cfg.n_layers, min(n_it, 3))
    tot, kinds = gemm_roofline(recs, cfg.n_layers, peaks)
    if tot["ms"]:
        ach = tot["flops"] / (tot["ms"] / 1000) / 1e12
        out["gemm"] = {"bound": "tensor", "achieved": ach, "peak": peaks["tc_sus"], "unit": "TFLOP/s",
                       "frac": ach / peaks["tc_sus"], "by_kind": kinds}
    release_gpu(eng)
    del dp
    release_gpu()
    if do_cpu:
        runner = OracleRunner(MODEL, 0, np.float32)
        d = draws[0]
        batch = ([r.rid for r in d], [len(r.prompt) for r in d], [r.ctx0 for r in d], [t for r in d for t in r.prompt])
        out["cpu_baseline"] = cpu_line(runner, [batch], "the first iteration (16 prompts + 128 increments)")
    return out


# --------------------------------------------------------------------------- #
# our arm
# --------------------------------------------------------------------------- #
def run_headline(args, eng, trace, cfg, peaks, world, local_rank):
    """The headline window (device-resident and through the serve loop) and the
    linear-layer roofline; returns the JSON line without the extra blocks."""
    import torch.distributed as dist

    # ---------------- the headline window, device-resident ------------------
    s = window_scheduler(eng, trace, args.window_start)
    s.set_token_feedback(True)  # from here on, increment inputs are the engine's own previous outputs
    n_it = args.warmup + args.steps
    plans, shapes = build_plans(eng, s, n_max=n_it)
    s.close()
    if len(plans) < n_it:
        raise RuntimeError("trace too short for the requested window")
    work = [iteration_work(n, c, cfg) for n, c in shapes]
    dp = DevicePlans(plans)
    timed_run(eng, dp, 0, args.warmup)
    clocks = Clocks(clock_device(local_rank))
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    it_ms, launches = timed_run(eng, dp, args.warmup, args.steps)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    elapsed_ms, tokens = reduce_replicas(sum(it_ms), sum(w["B"] for w in work[args.warmup:]), world, "cuda")
    value = tokens / (elapsed_ms / 1000.0)
    roof_it, fr = roofline_summary(work[args.warmup:], it_ms, peaks)

    # ---------------- the dominant kernel family: the linear layers --------
    recs = per_kernel_pass(eng, dp, args.warmup, args.steps)
    tot, gemm_kinds = gemm_roofline(recs, cfg.n_layers, peaks)
    t_hbm = tot["bytes"] / (peaks["hbm"] * 1e9)
    t_tc = tot["flops"] / (peaks["tc_sus"] * 1e12)
    if t_tc > t_hbm:
        ach = tot["flops"] / (tot["ms"] / 1000) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peaks["tc_sus"], "unit": "TFLOP/s"}
    else:
        ach = tot["bytes"] / (tot["ms"] / 1000) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm"], "unit": "GB/s"}
    per_launch = tot["bytes"] / tot["launches"]
    trec, why = traffic_record("gemm_decode")
    roof.update({"frac": roof["achieved"] / roof["peak"], "kernel": "linear layers (tcgen05 GEMM)",
                 "traffic": trec["dram_over_algorithmic"] * per_launch if trec else None,
                 "traffic_note": (f"ncu DRAM read+write over algorithmic bytes {trec['dram_over_algorithmic']:.3f} "
                                  f"({trec['workload']}), times this run's algorithmic bytes per launch")
                 if trec else why,
                 "peak_source": peaks["src"], "launches_per_iteration": tot["launches"] / args.steps,
                 "algorithmic_bytes_per_launch": per_launch,
                 "algorithmic_flops_per_launch": tot["flops"] / tot["launches"],
                 "ms_per_iteration": tot["ms"] / args.steps,
                 "weighting": "per-launch bytes and times weighted by launches per iteration "
                              f"({cfg.n_layers} per projection, 1 LM head)"})
    breakdown = kernel_breakdown(recs, cfg.n_layers, args.steps)
    breakdown_by_kind = kernel_breakdown_by_kind(recs, work[args.warmup:], cfg.n_layers)
    del dp

    # ---------------- the same window through the public serve loop --------
    e2e = None
    if not args.no_e2e:
        s2 = window_scheduler(eng, trace, args.window_start)
        dt, e2e_tokens = serve_loop_e2e(eng, s2, args.warmup, args.steps, None, world)
        s2.close()
        dt, e2e_tokens = reduce_replicas(dt, e2e_tokens, world, "cuda")
        h2d = 4.0 * sum(p.size for p in plans[args.warmup:]) / args.steps
        d2h = 4.0 * sum(w["B"] + 1 for w in work[args.warmup:]) / args.steps
        e2e = {"value": e2e_tokens / dt, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": 1000 * dt / args.steps, "api": "orca_sched_run (scheduler + orca_run_iteration)"}

    return {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "window_start_iteration": args.window_start, "layers": cfg.n_layers,
                   "replicas": world, "l2": "inputs larger than L2 (25.7 GB of weights streamed every iteration)"},
        "iteration_roofline": dict(roof_it, peaks={"hbm_GBs": peaks["hbm"], "bf16_TFLOPs_sustained": peaks["tc_sus"],
                                                   "source": peaks["src"]},
                                   mean_batch=float(np.mean([w["B"] for w in work[args.warmup:]])),
                                   mean_rows=float(np.mean([w["R"] for w in work[args.warmup:]])),
                                   by_kind=split_by_prefill(work[args.warmup:], it_ms, fr)),
        "roofline": roof, "kernels": breakdown, "kernels_by_kind": breakdown_by_kind, "gemm_by_kind": gemm_kinds,
        "gpu_launches": launches,
        "clocks": clk, "e2e": e2e,
    }


def run_orca(args, rank, world, local_rank):
    import torch

    torch.cuda.set_device(local_rank)
    cfg = MODEL.with_layers(args.layers)
    peaks = load_peaks()
    solo = world == 1
    keep, ptrs = gpu_weights(cfg, seed=rank)
    line = {"metric": METRIC, "unit": "tokens/s", "n_gpus": world, "dtype": "bf16", "data": "synthetic"}
    if not args.no_window:
        eng = make_engine(cfg, ptrs, MAX_TOKENS, MAX_BATCH, MAX_BATCH * KV_RESERVE)
        fill_kv_pool(eng, rank)
        trace = make_trace(rank)
        line = run_headline(args, eng, trace, cfg, peaks, world, local_rank)
        # ---------------- the whole trace (ramp, steady state, drain) ------
        if solo and not args.no_full_trace and cfg.n_layers == MODEL.n_layers:
            line["full_trace"] = run_full_trace(args, eng, trace, cfg, peaks)
        eng.close()
        release_gpu()
        # ---------------- the request-level baseline, padded + masked -------
        if solo and not args.no_request_level:
            rl = run_request_level_padded(args, ptrs, cfg, peaks, trace)
            rl["iteration_level_over_request_level"] = line["value"] / rl["value"]
            line["request_level"] = rl
        # ---------------- the CPU oracle on a bounded sample (rank 0, N=1) --
        if solo and not args.no_cpu:
            runner = OracleRunner(MODEL, 0, np.float32)
            line["cpu_baseline"] = cpu_line(runner, oracle_window_batches(args.window_start + args.warmup, 3),
                                            "2 window iterations")
            line["cpu_baseline"]["one_thread"] = one_thread_sample(args.window_start + args.warmup)

    # ---------------- the other workloads ------------------------------------
    if solo and args.configs:
        cfgs = {}
        names = [c for c in args.configs.split(",") if c]
        do_cpu = not args.no_cpu
        if "gpt3-13b-prefill-heavy" in names:
            cfgs["gpt3-13b-prefill-heavy"] = run_gpt3_prefill_heavy(args, peaks, do_cpu, cfg, ptrs)
        del keep
        release_gpu()
        if "gpt3-6.7b-decode" in names:
            cfgs["gpt3-6.7b-decode"] = run_gpt3_decode(args, peaks, do_cpu)
        if "gpt2-medium-mixed" in names:
            cfgs["gpt2-medium-mixed"] = run_gpt2_mixed(args, peaks, do_cpu)
        if "tiny-fp32" in names:
            cfgs["tiny-fp32"] = run_tiny(args, peaks, do_cpu)
        line["configs"] = cfgs
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
