"""One selectively batched iteration of a decoder-only GPT (oracle, float64).

What is computed ([houmin] 3.1.2 "方案"; [0h-n0] "Selective Batching";
[arcsin2] §3.2): the input rows of every request in the batch are stacked into
one ``[sum L, H]`` matrix with no batch dimension; the token-wise operations
(LayerNorm, the QKV / output / FFN projections, GeLU, residual adds) act on
that matrix as a whole; before attention the ``[sum L, 3H]`` projection is
split by request, attention runs per request over that request's own cached
K/V, and the per-request outputs are merged back into ``[sum L, H]``.  A
request with no cached K/V is in the initiation phase (all prompt tokens at
once); one with cached K/V is in the increment phase (one token) ([houmin]
3.1.2: the phase is read off whether the K/V manager holds K/V for it).  The
engine returns one output token per request ([houmin] 3.1.1 workflow step 4).

The pages list the block's operations (pre-projection, attention,
post-projection, FFN, LayerNorm, activation, residual; [houmin] 3.1.2 "思路")
but not their arrangement.  The reading taken is a GPT-2/3 block: pre-LN,
learned absolute positions, biases on every projection, exact (erf) GeLU,
LayerNorm with biased variance and eps = 1e-5, a final LayerNorm, an LM head
tied to the token embedding, dense causal attention, greedy argmax (lowest
index on ties).

Per layer, for request i with rows r = off[i] .. off[i+1]-1 and cached length
ctx[i], row r sits at position p = ctx[i] + (r - off[i]):

    h   = LN1(x)
    qkv = h W_qkv^T + b_qkv            q = qkv[:, :H], k = qkv[:, H:2H], v = qkv[:, 2H:]
    K_i[p] = k_r, V_i[p] = v_r         (written before attention)
    a_r (head j) = sum_{t<=p} softmax_t(q_r,j . K_i[t],j / sqrt(d)) V_i[t],j
    x  += a W_o^T + b_o
    x  += GeLU(LN2(x) W_1^T + b_1) W_2^T + b_2

and after the last layer ``y_i = LNf(x[off[i+1]-1])``, ``logits_i = y_i E^T``.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Sequence, Tuple

import numpy as np
from scipy.special import erf

LN_EPS = 1e-5


def layer_norm(x: np.ndarray, g: np.ndarray, b: np.ndarray, eps: float = LN_EPS, dtype=np.float64) -> np.ndarray:
    """Row-wise LayerNorm: (x - mean) / sqrt(biased var + eps) * g + b."""
    x = np.asarray(x, dtype)
    mean = x.mean(axis=-1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)
    return (x - mean) / np.sqrt(var + dtype(eps)) * np.asarray(g, dtype) + np.asarray(b, dtype)


def gelu(x: np.ndarray) -> np.ndarray:
    """Exact GeLU: x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2))."""
    return 0.5 * x * (1.0 + erf(x / math.sqrt(2.0)))


def softmax(s: np.ndarray, axis: int = -1) -> np.ndarray:
    m = np.max(s, axis=axis, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=axis, keepdims=True)


def argmax_lowest(v: np.ndarray) -> int:
    """Index of the maximum; the lowest index among equal maxima."""
    return int(np.argmax(v))


class KVStore:
    """Attention K/V manager: per request and per layer, the cached K and V
    rows ``[ctx, H]`` (position-major; head j is columns j*d .. (j+1)*d).

    ([0h-n0] "実装のポイント" item 2: an index table locating each request's
    K/V per layer.)  The oracle keys the cache by request id; where the rows
    live inside the engine's pool is checked separately (scheduler / K/V pool
    oracle), since the model's result does not depend on it.
    """

    def __init__(self, n_layers: int, hidden: int, dtype=np.float64):
        self.n_layers, self.hidden, self.dtype = n_layers, hidden, dtype
        self.k: Dict[Tuple[int, int], np.ndarray] = {}
        self.v: Dict[Tuple[int, int], np.ndarray] = {}

    def length(self, rid: int) -> int:
        a = self.k.get((rid, 0))
        return 0 if a is None else a.shape[0]

    def load(self, rid: int, layer: int, k: np.ndarray, v: np.ndarray) -> None:
        self.k[(rid, layer)] = np.asarray(k, self.dtype).copy()
        self.v[(rid, layer)] = np.asarray(v, self.dtype).copy()

    def write(self, rid: int, layer: int, pos: int, k_rows: np.ndarray, v_rows: np.ndarray) -> None:
        """Store rows at positions pos .. pos+n-1 (pos must equal the cached length)."""
        cur_k = self.k.get((rid, layer), np.zeros((0, self.hidden), self.dtype))
        cur_v = self.v.get((rid, layer), np.zeros((0, self.hidden), self.dtype))
        if cur_k.shape[0] != pos:
            raise ValueError(f"request {rid} layer {layer}: cache holds {cur_k.shape[0]} rows, writing at {pos}")
        self.k[(rid, layer)] = np.concatenate([cur_k, k_rows])
        self.v[(rid, layer)] = np.concatenate([cur_v, v_rows])

    def drop(self, rid: int) -> None:
        for l in range(self.n_layers):
            self.k.pop((rid, l), None)
            self.v.pop((rid, l), None)

    def copy(self) -> "KVStore":
        c = KVStore(self.n_layers, self.hidden, self.dtype)
        c.k = {key: a.copy() for key, a in self.k.items()}
        c.v = {key: a.copy() for key, a in self.v.items()}
        return c


@dataclasses.dataclass
class BatchItem:
    rid: int
    tokens: List[int]  # input rows of this iteration: the prompt (initiation) or one token (increment)
    ctx: int  # cached tokens before this iteration


@dataclasses.dataclass
class Result:
    hidden: np.ndarray  # [B, H]: LNf of each request's last row
    logits: np.ndarray  # [B, V]
    next_tokens: List[int]


def offsets(batch: Sequence[BatchItem]) -> List[int]:
    """Exclusive prefix sum of the per-request row counts (length B+1)."""
    off = [0]
    for it in batch:
        off.append(off[-1] + len(it.tokens))
    return off


def flatten(per_request_rows: Sequence[np.ndarray], dtype=np.float64) -> np.ndarray:
    """Selective batching's stacking: [(L_i, H)] -> (sum L_i, H), no batch dim."""
    return np.concatenate([np.asarray(r, dtype) for r in per_request_rows], axis=0)


def attention_one(q: np.ndarray, k: np.ndarray, v: np.ndarray, pos: np.ndarray, n_heads: int) -> np.ndarray:
    """Attention for one request: query rows at positions ``pos`` against the
    request's cached rows ``k, v`` [T, H]; row with position p sees keys 0..p."""
    n, H = q.shape
    d = H // n_heads
    T = k.shape[0]
    out = np.zeros((n, H), q.dtype)
    allowed = np.arange(T)[None, :] <= pos[:, None]
    for j in range(n_heads):
        sl = slice(j * d, (j + 1) * d)
        s = (q[:, sl] @ k[:, sl].T) / q.dtype.type(math.sqrt(d))
        s = np.where(allowed, s, -np.inf)
        out[:, sl] = softmax(s) @ v[:, sl]
    return out


def iteration(w: dict, n_heads: int, batch: Sequence[BatchItem], store: KVStore, hidden_only: bool = False,
              dtype=np.float64) -> Result:
    """One engine iteration over ``batch``; appends this iteration's K/V to ``store``.

    ``dtype`` is the arithmetic type: float64 (the default, used for every
    parity comparison) or float32, the precision the performance target names
    for timing this oracle as a CPU baseline."""
    f = lambda a: np.asarray(a, dtype)
    H = w["tok_emb"].shape[1]
    off = offsets(batch)
    tok = np.array([t for it in batch for t in it.tokens], dtype=np.int64)
    pos = np.array([it.ctx + j for it in batch for j in range(len(it.tokens))], dtype=np.int64)
    for it in batch:
        if store.length(it.rid) != it.ctx:
            raise ValueError(f"request {it.rid}: phase/context mismatch ({store.length(it.rid)} cached, ctx {it.ctx})")
    x = f(w["tok_emb"])[tok] + f(w["pos_emb"])[pos]
    for l, L in enumerate(w["layers"]):
        h = layer_norm(x, L["ln1_g"], L["ln1_b"], dtype=dtype)
        qkv = h @ f(L["w_qkv"]).T + f(L["b_qkv"])
        q, k, v = qkv[:, :H], qkv[:, H:2 * H], qkv[:, 2 * H:]
        a = np.zeros_like(q)
        for i, it in enumerate(batch):  # split ...
            rows = slice(off[i], off[i + 1])
            store.write(it.rid, l, it.ctx, k[rows], v[rows])
            a[rows] = attention_one(q[rows], store.k[(it.rid, l)], store.v[(it.rid, l)], pos[rows], n_heads)
        # ... merge: a is again one [sum L, H] matrix
        x = x + a @ f(L["w_o"]).T + f(L["b_o"])
        h2 = layer_norm(x, L["ln2_g"], L["ln2_b"], dtype=dtype)
        g1 = gelu(h2 @ f(L["w_1"]).T + f(L["b_1"]))
        x = x + g1 @ f(L["w_2"]).T + f(L["b_2"])
    last = [off[i + 1] - 1 for i in range(len(batch))]
    y = layer_norm(x[last], w["lnf_g"], w["lnf_b"], dtype=dtype)
    if hidden_only:
        return Result(y, np.zeros((len(batch), 0)), [])
    logits = y @ f(w["tok_emb"]).T
    return Result(y, logits, [argmax_lowest(r) for r in logits])
