"""The same iteration computed the padding + masking way (oracle).

[houmin] 3.1.2 "问题" and [arcsin2] §3.2: the conventional batched layer takes
one ``[B, L, H]`` tensor, so requests of different lengths (or different
cached lengths) must be padded to a common shape and masked.  The pages call
this wasteful, not wrong: it must give the same per-request result as
selective batching.  This module computes it that way, as an independent
check of :mod:`oracle.model`.

Shape: queries are padded to ``Lq = max n_i``, keys to ``Lk = max(ctx_i + n_i)``.
Query slot q of request b (valid when q < n_b) sits at position ctx_b + q and
may attend to key t when t <= ctx_b + q.  Padded query slots are given one
visible key (key 0) so their softmax is defined; their outputs are discarded.
"""

from __future__ import annotations

import math
from typing import Sequence

import numpy as np

from .model import BatchItem, KVStore, Result, argmax_lowest, gelu, layer_norm


def iteration(w: dict, n_heads: int, batch: Sequence[BatchItem], store: KVStore) -> Result:
    H = w["tok_emb"].shape[1]
    d = H // n_heads
    B = len(batch)
    Lq = max(len(it.tokens) for it in batch)
    Lk = max(it.ctx + len(it.tokens) for it in batch)
    n = np.array([len(it.tokens) for it in batch])
    ctx = np.array([it.ctx for it in batch])
    tok = np.zeros((B, Lq), np.int64)
    pos = np.zeros((B, Lq), np.int64)
    for b, it in enumerate(batch):
        tok[b, :n[b]] = it.tokens
        pos[b, :n[b]] = it.ctx + np.arange(n[b])
    valid_q = np.arange(Lq)[None, :] < n[:, None]  # [B, Lq]
    qpos = ctx[:, None] + np.arange(Lq)[None, :]
    mask = np.arange(Lk)[None, None, :] <= qpos[:, :, None]  # [B, Lq, Lk]
    mask = np.where(valid_q[:, :, None], mask, np.arange(Lk)[None, None, :] == 0)

    x = np.asarray(w["tok_emb"], np.float64)[tok] + np.asarray(w["pos_emb"], np.float64)[pos]  # [B, Lq, H]
    for l, L in enumerate(w["layers"]):
        h = layer_norm(x, L["ln1_g"], L["ln1_b"])
        qkv = h @ np.asarray(L["w_qkv"], np.float64).T + np.asarray(L["b_qkv"], np.float64)
        q, k, v = qkv[..., :H], qkv[..., H:2 * H], qkv[..., 2 * H:]
        K = np.zeros((B, Lk, H))
        Vv = np.zeros((B, Lk, H))
        for b, it in enumerate(batch):
            store.write(it.rid, l, it.ctx, k[b, :n[b]], v[b, :n[b]])
            T = it.ctx + n[b]
            K[b, :T] = store.k[(it.rid, l)]
            Vv[b, :T] = store.v[(it.rid, l)]
        a = np.zeros((B, Lq, H))
        for j in range(n_heads):
            sl = slice(j * d, (j + 1) * d)
            s = np.einsum("bqd,bkd->bqk", q[..., sl], K[..., sl]) / math.sqrt(d)
            s = np.where(mask, s, -np.inf)
            s = s - s.max(axis=-1, keepdims=True)
            p = np.exp(s)
            p = p / p.sum(axis=-1, keepdims=True)
            a[..., sl] = np.einsum("bqk,bkd->bqd", p, Vv[..., sl])
        x = x + a @ np.asarray(L["w_o"], np.float64).T + np.asarray(L["b_o"], np.float64)
        h2 = layer_norm(x, L["ln2_g"], L["ln2_b"])
        f = gelu(h2 @ np.asarray(L["w_1"], np.float64).T + np.asarray(L["b_1"], np.float64))
        x = x + f @ np.asarray(L["w_2"], np.float64).T + np.asarray(L["b_2"], np.float64)
    last = x[np.arange(B), n - 1]
    y = layer_norm(last, w["lnf_g"], w["lnf_b"])
    logits = y @ np.asarray(w["tok_emb"], np.float64).T
    return Result(y, logits, [argmax_lowest(r) for r in logits])
