"""Seeded synthetic inputs shared by the CUDA path's tests, the bench and the oracle.

This module only *draws* inputs: model weights, request traces and the
contents of pre-existing K/V caches.  It contains none of the method's
arithmetic (no layer norm, no attention, no scheduling), so the oracle and the
engine can both consume its output without sharing any computation.

All draws use ``numpy.random.Generator(PCG64(...))``.  The draw order for every
generator is fixed and documented below so a result can be reproduced from the
seed alone.  Values destined for bf16 storage are rounded to bf16
(round-to-nearest-even) here, once, so both sides see bit-identical numbers.
"""

from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np


# --------------------------------------------------------------------------- #
# model shapes
# --------------------------------------------------------------------------- #
@dataclasses.dataclass(frozen=True)
class ModelConfig:
    """Decoder-only GPT shape (pre-LN, learned positions, tied LM head)."""

    n_layers: int
    hidden: int
    n_heads: int
    ffn: int
    vocab: int
    max_pos: int
    dtype: str  # "fp32" or "bf16": storage type of matrices, embeddings and K/V

    @property
    def head_dim(self) -> int:
        return self.hidden // self.n_heads

    def with_layers(self, n_layers: int) -> "ModelConfig":
        return dataclasses.replace(self, n_layers=n_layers)

    def matrix_bytes(self) -> int:
        """Bytes of every weight matrix and both embeddings in storage type."""
        es = 2 if self.dtype == "bf16" else 4
        H, F = self.hidden, self.ffn
        per_layer = 3 * H * H + H * H + F * H + H * F
        return es * (self.n_layers * per_layer + self.vocab * H + self.max_pos * H)


# Tiny fp32 decoder: 2 layers, H=64, 4 heads, FFN 256, 128 positions, vocab 512.
TINY = ModelConfig(n_layers=2, hidden=64, n_heads=4, ffn=256, vocab=512, max_pos=128, dtype="fp32")
# GPT-2-medium shape in bf16 (the single mixed-batch microbench).
GPT2_MEDIUM = ModelConfig(n_layers=24, hidden=1024, n_heads=16, ffn=4096, vocab=50257, max_pos=4096, dtype="bf16")
# GPT-3 13B shape in bf16 (continuous-batching trace and prefill-heavy mix).
GPT3_13B = ModelConfig(n_layers=40, hidden=5120, n_heads=40, ffn=20480, vocab=50257, max_pos=4096, dtype="bf16")
# GPT-3 6.7B shape in bf16 (decode-dominated trace).
GPT3_6_7B = ModelConfig(n_layers=32, hidden=4096, n_heads=32, ffn=16384, vocab=50257, max_pos=4096, dtype="bf16")

CONFIGS = {"tiny": TINY, "gpt2-medium": GPT2_MEDIUM, "gpt3-13b": GPT3_13B, "gpt3-6.7b": GPT3_6_7B}


# --------------------------------------------------------------------------- #
# bf16 rounding of inputs
# --------------------------------------------------------------------------- #
def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32.

    Inputs here are finite normal draws, so NaN handling is not needed.
    """
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Upper 16 bits of float32 values that are already bf16-exact."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(list(key)))


def _normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    return (rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


# --------------------------------------------------------------------------- #
# weights
# --------------------------------------------------------------------------- #
LAYER_MATRICES = ("w_qkv", "w_o", "w_1", "w_2")
LAYER_VECTORS = ("b_qkv", "b_o", "b_1", "b_2", "ln1_g", "ln1_b", "ln2_g", "ln2_b")


def layer_shapes(cfg: ModelConfig) -> Dict[str, tuple]:
    H, F = cfg.hidden, cfg.ffn
    return {
        "w_qkv": (3 * H, H), "w_o": (H, H), "w_1": (F, H), "w_2": (H, F),
        "b_qkv": (3 * H,), "b_o": (H,), "b_1": (F,), "b_2": (H,),
        "ln1_g": (H,), "ln1_b": (H,), "ln2_g": (H,), "ln2_b": (H,),
    }


def make_weights(cfg: ModelConfig, seed: int = 0, random_affine: bool = False, std: float = 0.02) -> dict:
    """Random weights N(0, std) for every matrix and embedding.

    Matrices are stored output-major (``w[out, in]``), so ``y = x @ w.T``.
    Embeddings: ``tok_emb[V, H]`` (also the tied LM head), ``pos_emb[max_pos, H]``.

    Biases are 0 and LayerNorm gains 1 / shifts 0 unless ``random_affine``, in
    which case biases, gains-1 and shifts are N(0, std) so every fused epilogue
    term is exercised.  Matrices and embeddings are bf16-rounded when
    ``cfg.dtype == "bf16"``; biases and LayerNorm parameters stay float32.

    Draw order: stream ``(seed, 0)`` gives tok_emb then pos_emb; stream
    ``(seed, 1 + l)`` gives layer ``l``'s w_qkv, w_o, w_1, w_2 and then (only if
    ``random_affine``) its eight vectors in ``LAYER_VECTORS`` order; stream
    ``(seed, 100000)`` gives lnf_g-1 and lnf_b (only if ``random_affine``).
    """
    H, V, P = cfg.hidden, cfg.vocab, cfg.max_pos
    rnd = bf16_round if cfg.dtype == "bf16" else (lambda a: a)
    g = _rng(seed, 0)
    w = {"tok_emb": rnd(_normal(g, (V, H), std)), "pos_emb": rnd(_normal(g, (P, H), std)), "layers": []}
    shapes = layer_shapes(cfg)
    for l in range(cfg.n_layers):
        g = _rng(seed, 1 + l)
        layer = {name: rnd(_normal(g, shapes[name], std)) for name in LAYER_MATRICES}
        for name in LAYER_VECTORS:
            shape = shapes[name]
            if random_affine:
                v = _normal(g, shape, std)
                if name.endswith("_g"):
                    v = v + np.float32(1.0)
            else:
                v = np.ones(shape, np.float32) if name.endswith("_g") else np.zeros(shape, np.float32)
            layer[name] = v.astype(np.float32)
        w["layers"].append(layer)
    if random_affine:
        g = _rng(seed, 100000)
        w["lnf_g"] = (_normal(g, (H,), std) + np.float32(1.0)).astype(np.float32)
        w["lnf_b"] = _normal(g, (H,), std)
    else:
        w["lnf_g"] = np.ones((H,), np.float32)
        w["lnf_b"] = np.zeros((H,), np.float32)
    return w


# --------------------------------------------------------------------------- #
# requests and traces
# --------------------------------------------------------------------------- #
@dataclasses.dataclass
class RequestSpec:
    """One synthetic request.

    ``prompt`` are the input token ids.  ``out_len`` is the number of tokens the
    request generates (EOS is disabled, so this is fixed).  ``arrival`` is the
    arrival time in scheduler iterations.  A request that enters with an
    existing cached context (``ctx0 > 0``) has its K/V drawn by
    :func:`kv_context` and ``prompt`` holds exactly one token: the pending
    input of its next increment iteration.
    """

    rid: int
    arrival: float
    prompt: List[int]
    out_len: int
    ctx0: int = 0


def tiny_requests(seed: int = 0, vocab: int = 512) -> List[RequestSpec]:
    """8 requests, prompt lengths U[2,16], tokens U[0,vocab), all arriving at 0.

    Output lengths are the fixed list [5, 50, 8, 12, 40, 3, 30, 7].
    Draw order: 8 prompt lengths, then each prompt's tokens in request order.
    """
    outs = [5, 50, 8, 12, 40, 3, 30, 7]
    g = _rng(seed, 11)
    lens = g.integers(2, 16, size=8, endpoint=True)
    return [RequestSpec(i, 0.0, [int(t) for t in g.integers(0, vocab, size=int(L))], outs[i]) for i, L in enumerate(lens)]


def mixed_batch(seed: int = 0, vocab: int = 50257, prompt_lens=(128, 64, 256), n_incr: int = 29,
                ctx_range=(1, 1024)) -> List[RequestSpec]:
    """One mixed batch: initiation requests of the given prompt lengths followed by
    ``n_incr`` increment requests with cached contexts U[ctx_range].

    Draw order: the prompts' tokens in order, then the increment requests'
    context lengths, then their pending input tokens.
    """
    g = _rng(seed, 12)
    reqs = [RequestSpec(i, 0.0, [int(t) for t in g.integers(0, vocab, size=L)], 1) for i, L in enumerate(prompt_lens)]
    ctx = g.integers(ctx_range[0], ctx_range[1], size=n_incr, endpoint=True)
    toks = g.integers(0, vocab, size=n_incr)
    base = len(prompt_lens)
    reqs += [RequestSpec(base + j, 0.0, [int(toks[j])], 1, int(ctx[j])) for j in range(n_incr)]
    return reqs


def poisson_trace(seed: int = 0, n: int = 1000, rate: float = 0.5, prompt_range=(32, 512),
                  out_range=(1, 512), vocab: int = 50257, with_tokens: bool = True) -> List[RequestSpec]:
    """Continuous-batching trace: Poisson arrivals on the iteration clock.

    Inter-arrival gaps are Exp(rate) (rate in requests per iteration); prompt
    lengths U[prompt_range]; output lengths U[out_range].  Draw order: the n
    gaps, the n prompt lengths, the n output lengths, then the prompts' tokens
    in request order (skipped, and replaced by zeros, if ``with_tokens`` is
    false, which leaves every other draw unchanged).
    """
    g = _rng(seed, 13)
    gaps = g.exponential(1.0 / rate, size=n)
    arrival = np.cumsum(gaps)
    plen = g.integers(prompt_range[0], prompt_range[1], size=n, endpoint=True)
    olen = g.integers(out_range[0], out_range[1], size=n, endpoint=True)
    reqs = []
    for i in range(n):
        toks = [int(t) for t in g.integers(0, vocab, size=int(plen[i]))] if with_tokens else [0] * int(plen[i])
        reqs.append(RequestSpec(i, float(arrival[i]), toks, int(olen[i])))
    return reqs


def decode_pool(seed: int = 0, n_running: int = 128, ctx_range=(256, 1024), remaining_range=(1, 256),
                n_refill: int = 4096, refill_prompt: int = 64, vocab: int = 50257) -> List[RequestSpec]:
    """Decode-dominated workload: ``n_running`` requests already in the increment
    phase (contexts U[ctx_range], remaining outputs U[remaining_range]) plus a
    queue of refill requests (prompt ``refill_prompt`` tokens, outputs
    U[remaining_range]) that are admitted as running ones finish.

    Draw order: contexts, remaining lengths, pending tokens of the running
    requests; then refill output lengths, then refill prompt tokens.
    """
    g = _rng(seed, 14)
    ctx = g.integers(ctx_range[0], ctx_range[1], size=n_running, endpoint=True)
    rem = g.integers(remaining_range[0], remaining_range[1], size=n_running, endpoint=True)
    tok = g.integers(0, vocab, size=n_running)
    reqs = [RequestSpec(i, 0.0, [int(tok[i])], int(rem[i]), int(ctx[i])) for i in range(n_running)]
    rout = g.integers(remaining_range[0], remaining_range[1], size=n_refill, endpoint=True)
    for j in range(n_refill):
        reqs.append(RequestSpec(n_running + j, 0.0, [int(t) for t in g.integers(0, vocab, size=refill_prompt)], int(rout[j])))
    return reqs


def prefill_heavy_batch(seed: int = 0, n_init: int = 16, prompt_range=(1024, 2048), n_incr: int = 128,
                        ctx_range=(128, 2048), vocab: int = 50257) -> List[RequestSpec]:
    """One prefill-heavy iteration: ``n_init`` initiation requests with prompts
    U[prompt_range] plus ``n_incr`` increment requests with contexts U[ctx_range].

    Draw order: prompt lengths, prompt tokens in request order, contexts,
    pending tokens.
    """
    g = _rng(seed, 15)
    plen = g.integers(prompt_range[0], prompt_range[1], size=n_init, endpoint=True)
    reqs = [RequestSpec(i, 0.0, [int(t) for t in g.integers(0, vocab, size=int(plen[i]))], 1) for i in range(n_init)]
    ctx = g.integers(ctx_range[0], ctx_range[1], size=n_incr, endpoint=True)
    tok = g.integers(0, vocab, size=n_incr)
    reqs += [RequestSpec(n_init + j, 0.0, [int(tok[j])], 1, int(ctx[j])) for j in range(n_incr)]
    return reqs


# --------------------------------------------------------------------------- #
# cached K/V contents of requests that enter with an existing context
# --------------------------------------------------------------------------- #
def kv_context(seed: int, rid: int, layer: int, ctx: int, hidden: int, dtype: str = "bf16", std: float = 1.0):
    """K and V rows ``[ctx, hidden]`` (position-major, heads side by side) for one
    request and one layer, N(0, std), bf16-rounded for bf16 models.

    Stream ``(seed, 7, rid, layer)``: K first, then V.
    """
    g = _rng(seed, 7, rid, layer)
    k = _normal(g, (ctx, hidden), std)
    v = _normal(g, (ctx, hidden), std)
    if dtype == "bf16":
        k, v = bf16_round(k), bf16_round(v)
    return k, v
