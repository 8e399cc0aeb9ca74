"""Helpers of the GPU parity tests: upload seeded inputs, drive the engine
through the C ABI, and compare with the oracle.  PyTorch is used only to own
device memory."""

from __future__ import annotations

import numpy as np
import torch

from iteration_level_scheduling_gb300 import synth

DTYPE = {"fp32": 0, "bf16": 1}


class DevicePtr:
    """Zero-copy torch view of device memory owned by the engine."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None}


def to_dev(a: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def upload_weights(w: dict, cfg: synth.ModelConfig):
    """Returns (keep-alive list, pointer dict in orca_weights layout)."""
    keep = []

    def mat(a):
        t = to_dev(a, cfg.dtype)
        keep.append(t)
        return t.data_ptr()

    def vec(a):
        t = torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
        keep.append(t)
        return t.data_ptr()

    layers = []
    for L in w["layers"]:
        d = {k: mat(L[k]) for k in synth.LAYER_MATRICES}
        d.update({k: vec(L[k]) for k in synth.LAYER_VECTORS})
        layers.append(d)
    ptrs = {"tok_emb": mat(w["tok_emb"]), "pos_emb": mat(w["pos_emb"]), "lnf_g": vec(w["lnf_g"]),
            "lnf_b": vec(w["lnf_b"]), "layers": layers}
    return keep, ptrs


def make_engine(cfg: synth.ModelConfig, w: dict, max_tokens: int, max_batch: int, kv_slots: int,
                pack_weights: bool = True):
    from iteration_level_scheduling_gb300 import native
    keep, ptrs = upload_weights(w, cfg)
    eng = native.Engine(cfg.n_layers, cfg.hidden, cfg.n_heads, cfg.ffn, cfg.vocab, cfg.max_pos, DTYPE[cfg.dtype],
                        max_tokens, max_batch, kv_slots, ptrs, torch.cuda.current_stream().cuda_stream,
                        pack_weights=pack_weights)
    eng._keep = keep
    return eng


def kv_pool_tensor(eng) -> torch.Tensor:
    lay = eng.kv_layout()
    shape = (lay.n_layers, 2, lay.n_heads, lay.kv_slots, lay.head_dim)
    if lay.elem_bytes == 2:
        return torch.as_tensor(DevicePtr(lay.base, shape, "<i2"), device="cuda").view(torch.bfloat16)
    return torch.as_tensor(DevicePtr(lay.base, shape, "<f4"), device="cuda")


def load_context(eng, pool: torch.Tensor, cfg: synth.ModelConfig, seed: int, rid: int, kv_off: int, ctx: int,
                 store=None):
    """Write request rid's cached K/V (synth.kv_context) into the engine's pool
    (and, if given, the oracle's store)."""
    nh, d = cfg.n_heads, cfg.head_dim
    for l in range(cfg.n_layers):
        k, v = synth.kv_context(seed, rid, l, ctx, cfg.hidden, cfg.dtype)
        for which, a in ((0, k), (1, v)):
            t = to_dev(a, cfg.dtype).view(ctx, nh, d).permute(1, 0, 2)
            pool[l, which, :, kv_off:kv_off + ctx, :] = t
        if store is not None:
            store.load(rid, l, k, v)


def normwise(a: np.ndarray, ref: np.ndarray) -> float:
    return float(np.max(np.abs(np.asarray(a, np.float64) - ref)) / max(np.max(np.abs(ref)), 1e-30))


# Greedy-token agreement with the oracle: >= 99 % of the compared tokens.
MIN_AGREE = 0.99
# At GPT-3 widths (H 4096, 5120) with random N(0, 0.02) weights the logits of
# a row have many near-equal competitors, and rounding the GEMM operands to
# bf16 -- the engine's arithmetic -- flips 1.4 - 2.6 % of greedy tokens whose
# oracle margin lies within a few times the row's logit error (a CPU model of
# the same rounding points, compared with the float64 oracle, gives 97.4 % and
# 98.6 % on two 13B-width traces, and 100 % without the roundings).  There
# the tests allow up to 3 % of the tokens, at least one, to differ, and only
# as near-ties: the oracle's margin between its token and the engine's must
# be at most NEAR_TIE times that row's RMS logit error.  A kernel bug shows
# as a flip with a clear margin (error concentrated on a few logits) or as a
# flip rate above that floor.
MAX_NEAR_TIE_FLIPS = 0.03
NEAR_TIE = 6.0


def disagreements(got, gpu_logits, ref_logits, ref_tokens):
    """For every request whose greedy token differs from the oracle's: the
    oracle's own margin between its token and the engine's token, the
    engine's error on those two logits and the row's RMS logit error.  Empty
    when every token agrees."""
    out = []
    for i, (a, r) in enumerate(zip(list(got), list(ref_tokens))):
        if int(a) != int(r):
            margin = float(ref_logits[i, r] - ref_logits[i, a])
            err = float(max(abs(gpu_logits[i, r] - ref_logits[i, r]), abs(gpu_logits[i, a] - ref_logits[i, a])))
            rms = float(np.sqrt(np.mean((np.asarray(gpu_logits[i], np.float64) - ref_logits[i]) ** 2)))
            out.append(dict(row=i, gpu=int(a), ref=int(r), ref_margin=margin, logit_err=err, row_rms_err=rms))
    return out


def assert_agreement(agree: float, n: int, mismatches, wide: bool):
    """>= 99 % agreement; at GPT-3 widths the bf16 near-tie floor above."""
    if not wide:
        assert agree >= MIN_AGREE, (agree, n, mismatches)
        return
    assert len(mismatches) <= max(1, int(MAX_NEAR_TIE_FLIPS * n)), (agree, n, mismatches)
    for m in mismatches:
        assert m["ref_margin"] <= NEAR_TIE * m["row_rms_err"], m


# --------------------------------------------------------------------------- #
# full-depth checks on sampled requests: the oracle streams each layer's
# weights and each sampled request's cached K/V back from the device
# --------------------------------------------------------------------------- #
LAYER_KEYS = ("w_qkv", "w_o", "w_1", "w_2", "b_qkv", "b_o", "b_1", "b_2", "ln1_g", "ln1_b", "ln2_g", "ln2_b")


class DeviceLayers:
    """Iterates over the layers of device-resident weights (the keep list of
    bench.gpu_weights: 12 tensors per layer in LAYER_KEYS order), one layer's
    arrays on the host at a time."""

    def __init__(self, keep, n_layers):
        self.keep, self.n_layers = keep, n_layers

    def __iter__(self):
        for l in range(self.n_layers):
            yield {k: self.keep[12 * l + j].float().cpu().numpy() for j, k in enumerate(LAYER_KEYS)}

    def __len__(self):
        return self.n_layers


def device_weight_dict(keep, cfg):
    """The oracle's weight dict over bench.gpu_weights' tensors (layers streamed)."""
    L = cfg.n_layers
    assert len(keep) == 12 * L + 4
    tail = [t.float().cpu().numpy() for t in keep[12 * L:]]
    return {"tok_emb": tail[0], "pos_emb": tail[1], "lnf_g": tail[2], "lnf_b": tail[3],
            "layers": DeviceLayers(keep, L)}


class PoolStore:
    """The oracle's KVStore interface over the engine's pool: a request's cached
    rows of layer l are read from the device the first time they are needed
    and dropped once layer l + 1 has been written."""

    def __init__(self, pool, ctx_of, kv_off_of, n_layers, hidden):
        from oracle.model import KVStore
        self.inner = KVStore(n_layers, hidden)
        self.pool, self.ctx_of, self.kv_off_of = pool, ctx_of, kv_off_of
        self.k, self.v = self.inner.k, self.inner.v

    def _fetch(self, rid, l):
        if (rid, l) not in self.inner.k:
            c, o = self.ctx_of[rid], self.kv_off_of[rid]
            nh, d = self.pool.shape[2], self.pool.shape[4]
            k = self.pool[l, 0, :, o:o + c, :].permute(1, 0, 2).reshape(c, nh * d).float().cpu().numpy()
            v = self.pool[l, 1, :, o:o + c, :].permute(1, 0, 2).reshape(c, nh * d).float().cpu().numpy()
            self.inner.load(rid, l, k, v)

    def length(self, rid):
        return self.ctx_of[rid]

    def write(self, rid, layer, pos, k_rows, v_rows):
        self._fetch(rid, layer)
        self.inner.write(rid, layer, pos, k_rows, v_rows)
        if layer > 0:
            self.inner.k.pop((rid, layer - 1), None)
            self.inner.v.pop((rid, layer - 1), None)


def full_depth_check(eng, keep, cfg, batch, sample_idx):
    """Run `batch` (a native.BatchDesc) through the engine and recompute the
    requests at `sample_idx` with the oracle from the same device weights and
    K/V.  Returns normwise errors of the final-LN hidden rows and the logits,
    the greedy-token agreement, and the engine's argmax consistency."""
    from oracle.model import BatchItem, iteration
    got = eng.run_iteration(batch)
    hid = eng.last_hidden(batch.n_req)
    lg = eng.last_logits(batch.n_req)
    pool = kv_pool_tensor(eng)
    rid = batch.request_id.tolist()
    n = batch.n_input.tolist()
    ctx = batch.ctx_len.tolist()
    off = np.concatenate([[0], np.cumsum(n)]).tolist()
    toks = batch.tokens.tolist()
    items = [BatchItem(rid[i], toks[off[i]:off[i + 1]], ctx[i]) for i in sample_idx]
    store = PoolStore(pool, {rid[i]: ctx[i] for i in sample_idx},
                      {rid[i]: int(batch.kv_offset[i]) for i in sample_idx}, cfg.n_layers, cfg.hidden)
    ref = iteration(device_weight_dict(keep, cfg), cfg.n_heads, items, store)
    return dict(h=normwise(hid[sample_idx], ref.hidden), l=normwise(lg[sample_idx], ref.logits),
                agree=float(np.mean([got[i] == t for i, t in zip(sample_idx, ref.next_tokens)])),
                n=len(sample_idx), argmax_ok=got.tolist() == lg.argmax(1).tolist(),
                mismatches=disagreements(got[sample_idx], lg[sample_idx], ref.logits, ref.next_tokens))
