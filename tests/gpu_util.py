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
