"""ctypes binding of liborca.so (include/orca.h).

Argument marshalling only: every step of an iteration runs in the library's
CUDA kernels, and scheduling runs in its C++ scheduler.  Importing this module
loads the library and raises ``RuntimeError`` if it has not been built
(``python -m iteration_level_scheduling_gb300.build``); there is no fallback.
"""

from __future__ import annotations

import ctypes as C
import os
from typing import Dict, List, Optional, Sequence

import numpy as np

from .build import LIB

if not os.path.exists(LIB):
    raise RuntimeError(f"liborca.so is not built ({LIB}); run iteration_level_scheduling_gb300.build.build()")
lib = C.CDLL(LIB)

OK, ERR_INVALID, ERR_KV_FULL, ERR_CUDA, ERR_DEVICE_FLAG, ERR_NOT_FOUND, ERR_OOM, ERR_LIMIT = 0, -1, -2, -3, -4, -5, -6, -7
DTYPE_FP32, DTYPE_BF16 = 0, 1
KERNEL_KINDS = ["embed", "layernorm", "gemm_qkv", "kv_append", "attn_decode", "attn_prefill", "gemm_o",
                "gemm_ffn1", "gemm_ffn2", "lm_head", "argmax", "final_ln"]

EXPORTS = [
    "orca_strerror", "orca_engine_create", "orca_engine_destroy", "orca_kv_alloc", "orca_kv_free",
    "orca_kv_layout_get", "orca_run_iteration", "orca_plan_words", "orca_plan_build", "orca_run_planned",
    "orca_run_iteration_padded", "orca_plan_words_padded", "orca_plan_build_padded",
    "orca_engine_sync", "orca_get_last_hidden", "orca_get_last_logits", "orca_engine_stats_get",
    "orca_engine_timing", "orca_engine_timing_read", "orca_op_linear", "orca_op_attention", "orca_packed_weight_elems",
    "orca_pack_weight",
    "orca_attention_decode_noalloc", "orca_debug_expire_wait", "orca_sched_create", "orca_sched_destroy",
    "orca_sched_submit", "orca_sched_set_token_feedback", "orca_sched_next", "orca_sched_complete", "orca_sched_cancel",
    "orca_sched_stats_get", "orca_sched_request_get",
    "orca_sched_request_tokens", "orca_sched_run",
]


class OrcaError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {lib.orca_strerror(code).decode()} ({code})")


class ModelConfig(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("hidden", C.c_int32), ("n_heads", C.c_int32), ("ffn", C.c_int32),
                ("vocab", C.c_int32), ("max_pos", C.c_int32), ("dtype", C.c_int32), ("max_tokens", C.c_int32),
                ("max_batch", C.c_int32), ("kv_slots", C.c_int64), ("pack_weights", C.c_int32)]


class LayerWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("w_qkv", "w_o", "w_1", "w_2", "b_qkv", "b_o", "b_1", "b_2",
                                           "ln1_g", "ln1_b", "ln2_g", "ln2_b")]


class Weights(C.Structure):
    _fields_ = [("tok_emb", C.c_void_p), ("pos_emb", C.c_void_p), ("lnf_g", C.c_void_p), ("lnf_b", C.c_void_p),
                ("layers", C.POINTER(LayerWeights))]


class Batch(C.Structure):
    _fields_ = [("n_req", C.c_int32), ("request_id", C.POINTER(C.c_int64)), ("phase", C.POINTER(C.c_int32)),
                ("n_input", C.POINTER(C.c_int32)), ("ctx_len", C.POINTER(C.c_int32)),
                ("kv_offset", C.POINTER(C.c_int64)), ("tokens", C.POINTER(C.c_int32))]


class KVLayout(C.Structure):
    _fields_ = [("base", C.c_void_p), ("kv_slots", C.c_int64), ("n_layers", C.c_int32), ("n_heads", C.c_int32),
                ("head_dim", C.c_int32), ("elem_bytes", C.c_int32)]


class EngineStats(C.Structure):
    _fields_ = [("launches", C.c_int64), ("iterations", C.c_int64)]


class KernelTime(C.Structure):
    _fields_ = [("kind", C.c_int32), ("layer", C.c_int32), ("ms", C.c_float), ("bytes", C.c_double),
                ("flops", C.c_double)]


class SchedConfig(C.Structure):
    _fields_ = [("max_batch", C.c_int32), ("max_tokens", C.c_int32), ("kv_slots", C.c_int64),
                ("kv_reserve", C.c_int32), ("mode", C.c_int32), ("token_feedback", C.c_int32),
                ("chunked_prefill", C.c_int32), ("n_workers", C.c_int32)]


class SchedStats(C.Structure):
    _fields_ = [("clock", C.c_int64), ("iterations", C.c_int64), ("generated", C.c_int64), ("finished", C.c_int64),
                ("waiting", C.c_int64), ("running", C.c_int64), ("kv_reserved", C.c_int64), ("cancelled", C.c_int64)]


class RequestInfo(C.Structure):
    _fields_ = [("id", C.c_int64), ("kv_offset", C.c_int64), ("state", C.c_int32), ("ctx_len", C.c_int32),
                ("n_generated", C.c_int32), ("admitted_at", C.c_int64), ("finished_at", C.c_int64)]


P = C.c_void_p
_sig = {
    "orca_strerror": (C.c_char_p, [C.c_int]),
    "orca_engine_create": (C.c_int, [C.POINTER(ModelConfig), C.POINTER(Weights), P, C.POINTER(P)]),
    "orca_engine_destroy": (C.c_int, [P]),
    "orca_kv_alloc": (C.c_int, [P, C.c_int64, C.c_int32, C.POINTER(C.c_int64)]),
    "orca_kv_free": (C.c_int, [P, C.c_int64]),
    "orca_kv_layout_get": (C.c_int, [P, C.POINTER(KVLayout)]),
    "orca_run_iteration": (C.c_int, [P, C.POINTER(Batch), P]),
    "orca_plan_words": (C.c_int64, [P, C.POINTER(Batch)]),
    "orca_plan_build": (C.c_int, [P, C.POINTER(Batch), P, C.c_int64]),
    "orca_run_planned": (C.c_int, [P, P, P, P]),
    "orca_run_iteration_padded": (C.c_int, [P, C.POINTER(Batch), P]),
    "orca_plan_words_padded": (C.c_int64, [P, C.POINTER(Batch)]),
    "orca_plan_build_padded": (C.c_int, [P, C.POINTER(Batch), P, C.c_int64]),
    "orca_engine_sync": (C.c_int, [P]),
    "orca_get_last_hidden": (C.c_int, [P, P, C.c_int64]),
    "orca_get_last_logits": (C.c_int, [P, P, C.c_int64]),
    "orca_engine_stats_get": (C.c_int, [P, C.POINTER(EngineStats)]),
    "orca_engine_timing": (C.c_int, [P, C.c_int32]),
    "orca_engine_timing_read": (C.c_int, [P, C.POINTER(KernelTime), C.c_int32, C.POINTER(C.c_int32)]),
    "orca_op_linear": (C.c_int, [P, C.c_int32, P, P, C.c_int32, C.c_int32, C.c_int32, C.c_int32, P, C.c_int32, P, P,
                                 P, C.c_int32]),
    "orca_packed_weight_elems": (C.c_int64, [C.c_int32, C.c_int32]),
    "orca_pack_weight": (C.c_int, [P, P, C.c_int32, C.c_int32, P]),
    "orca_op_attention": (C.c_int, [P, C.c_int32, P, P, C.c_int64, C.c_int32, C.c_int32, C.c_int32, P, P, P, P]),
    "orca_attention_decode_noalloc": (C.c_int, [C.c_int32, P, P, C.c_int64, C.c_int32, C.c_int32, C.c_int32, P, P,
                                                P, P]),
    "orca_debug_expire_wait": (C.c_int, [P, C.c_int64]),
    "orca_sched_create": (C.c_int, [C.POINTER(SchedConfig), P, C.POINTER(P)]),
    "orca_sched_destroy": (C.c_int, [P]),
    "orca_sched_submit": (C.c_int, [P, C.c_int64, C.c_double, P, C.c_int32, C.c_int32, C.c_int32,
                                    C.POINTER(C.c_int64)]),
    "orca_sched_set_token_feedback": (C.c_int, [P, C.c_int32]),
    "orca_sched_next": (C.c_int, [P, C.POINTER(Batch), C.POINTER(C.c_int32)]),
    "orca_sched_complete": (C.c_int, [P, P]),
    "orca_sched_cancel": (C.c_int, [P, C.c_int64]),
    "orca_sched_stats_get": (C.c_int, [P, C.POINTER(SchedStats)]),
    "orca_sched_request_get": (C.c_int, [P, C.c_int64, C.POINTER(RequestInfo)]),
    "orca_sched_request_tokens": (C.c_int, [P, C.c_int64, P, C.c_int32, C.POINTER(C.c_int32)]),
    "orca_sched_run": (C.c_int, [P, C.c_int64]),
}
for _name, (_res, _args) in _sig.items():
    _f = getattr(lib, _name)
    _f.restype, _f.argtypes = _res, _args


def check(rc: int, what: str) -> int:
    if rc < 0:
        raise OrcaError(rc, what)
    return rc


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


class BatchDesc:
    """Host-side owner of the arrays an ``orca_batch`` points to."""

    def __init__(self, request_id, phase, n_input, ctx_len, kv_offset, tokens):
        self.request_id, self.kv_offset = _i64(request_id), _i64(kv_offset)
        self.phase, self.n_input, self.ctx_len, self.tokens = _i32(phase), _i32(n_input), _i32(ctx_len), _i32(tokens)
        self.c = Batch(len(self.request_id), self.request_id.ctypes.data_as(C.POINTER(C.c_int64)),
                       self.phase.ctypes.data_as(C.POINTER(C.c_int32)),
                       self.n_input.ctypes.data_as(C.POINTER(C.c_int32)),
                       self.ctx_len.ctypes.data_as(C.POINTER(C.c_int32)),
                       self.kv_offset.ctypes.data_as(C.POINTER(C.c_int64)),
                       self.tokens.ctypes.data_as(C.POINTER(C.c_int32)))

    @property
    def n_req(self) -> int:
        return len(self.request_id)

    @staticmethod
    def from_c(b: Batch) -> "BatchDesc":
        n = b.n_req
        rows = int(np.ctypeslib.as_array(b.n_input, (n,)).sum())
        return BatchDesc(np.ctypeslib.as_array(b.request_id, (n,)).copy(), np.ctypeslib.as_array(b.phase, (n,)).copy(),
                         np.ctypeslib.as_array(b.n_input, (n,)).copy(), np.ctypeslib.as_array(b.ctx_len, (n,)).copy(),
                         np.ctypeslib.as_array(b.kv_offset, (n,)).copy(), np.ctypeslib.as_array(b.tokens, (rows,)).copy())


class Engine:
    """One model on one GPU.  ``weights`` holds device pointers (ints) laid out
    as ``orca_weights``; the engine borrows them (keep the tensors alive)."""

    def __init__(self, n_layers, hidden, n_heads, ffn, vocab, max_pos, dtype, max_tokens, max_batch, kv_slots,
                 weights: Optional[dict] = None, stream: int = 0, pack_weights: bool = True):
        self.cfg = ModelConfig(n_layers, hidden, n_heads, ffn, vocab, max_pos, dtype, max_tokens, max_batch, kv_slots,
                               int(pack_weights))
        self._h = P()
        wp = None
        if weights is not None:
            self._layers = (LayerWeights * n_layers)(*[LayerWeights(**L) for L in weights["layers"]])
            self._w = Weights(weights["tok_emb"], weights["pos_emb"], weights["lnf_g"], weights["lnf_b"], self._layers)
            wp = C.byref(self._w)
        check(lib.orca_engine_create(C.byref(self.cfg), wp, P(stream), C.byref(self._h)), "orca_engine_create")

    def close(self):
        if self._h:
            lib.orca_engine_destroy(self._h)
            self._h = P()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    def kv_alloc(self, rid: int, n: int) -> int:
        off = C.c_int64()
        check(lib.orca_kv_alloc(self._h, rid, n, C.byref(off)), "orca_kv_alloc")
        return off.value

    def kv_free(self, rid: int):
        check(lib.orca_kv_free(self._h, rid), "orca_kv_free")

    def kv_layout(self) -> KVLayout:
        out = KVLayout()
        check(lib.orca_kv_layout_get(self._h, C.byref(out)), "orca_kv_layout_get")
        return out

    def run_iteration(self, batch: BatchDesc) -> np.ndarray:
        out = np.zeros(batch.n_req, np.int32)
        check(lib.orca_run_iteration(self._h, C.byref(batch.c), _ptr(out)), "orca_run_iteration")
        return out

    def plan_words(self, batch: BatchDesc, padded: bool = False) -> int:
        f = lib.orca_plan_words_padded if padded else lib.orca_plan_words
        return check(f(self._h, C.byref(batch.c)), "orca_plan_words")

    def plan_build(self, batch: BatchDesc, buf: np.ndarray, padded: bool = False) -> None:
        f = lib.orca_plan_build_padded if padded else lib.orca_plan_build
        check(f(self._h, C.byref(batch.c), _ptr(buf), buf.size), "orca_plan_build")

    def run_iteration_padded(self, batch: BatchDesc) -> np.ndarray:
        """The iteration as a conventional padded + masked batch (see orca.h)."""
        out = np.zeros(batch.n_req, np.int32)
        check(lib.orca_run_iteration_padded(self._h, C.byref(batch.c), _ptr(out)), "orca_run_iteration_padded")
        return out

    def run_planned(self, host_plan: np.ndarray, dev_plan_ptr: int, dev_out_ptr: int = 0) -> None:
        check(lib.orca_run_planned(self._h, _ptr(host_plan), P(dev_plan_ptr), P(dev_out_ptr or None)),
              "orca_run_planned")

    def sync(self):
        check(lib.orca_engine_sync(self._h), "orca_engine_sync")

    def last_hidden(self, n_req: int) -> np.ndarray:
        out = np.zeros((n_req, self.cfg.hidden), np.float32)
        check(lib.orca_get_last_hidden(self._h, _ptr(out), out.size), "orca_get_last_hidden")
        return out

    def last_logits(self, n_req: int) -> np.ndarray:
        out = np.zeros((n_req, self.cfg.vocab), np.float32)
        check(lib.orca_get_last_logits(self._h, _ptr(out), out.size), "orca_get_last_logits")
        return out

    def stats(self) -> EngineStats:
        s = EngineStats()
        check(lib.orca_engine_stats_get(self._h, C.byref(s)), "orca_engine_stats_get")
        return s

    def timing(self, enable: bool):
        check(lib.orca_engine_timing(self._h, int(enable)), "orca_engine_timing")

    def timing_read(self, cap: int = 1 << 16) -> List[dict]:
        buf = (KernelTime * cap)()
        n = C.c_int32()
        check(lib.orca_engine_timing_read(self._h, buf, cap, C.byref(n)), "orca_engine_timing_read")
        return [dict(kind=KERNEL_KINDS[buf[i].kind], layer=buf[i].layer, ms=buf[i].ms, bytes=buf[i].bytes,
                     flops=buf[i].flops) for i in range(n.value)]

    def op_linear(self, dtype: int, x: int, w: int, m: int, n: int, k: int, bias: int = 0, gelu: bool = False,
                  resid: int = 0, out_f32: int = 0, out_bf16: int = 0, ld_out: int = 0, sync: bool = True,
                  w_packed: bool = False):
        check(lib.orca_op_linear(self._h, dtype, P(x), P(w), int(w_packed), m, n, k, P(bias or None), int(gelu),
                                 P(resid or None), P(out_f32 or None), P(out_bf16 or None), ld_out or n),
              "orca_op_linear")
        if sync:
            self.sync()

    def debug_expire_wait(self, limit_ns: int) -> None:
        """Make a bounded device wait run out (see orca.h); asynchronous."""
        check(lib.orca_debug_expire_wait(self._h, int(limit_ns)), "orca_debug_expire_wait")

    @staticmethod
    def packed_weight_elems(n_out: int, k: int) -> int:
        return check(lib.orca_packed_weight_elems(n_out, k), "orca_packed_weight_elems")

    def pack_weight(self, w: int, n_out: int, k: int, out: int) -> None:
        check(lib.orca_pack_weight(self._h, P(w), n_out, k, P(out)), "orca_pack_weight")

    def op_attention(self, dtype: int, qkv: int, kv_layer: int, kv_slots: int, n_heads: int, head_dim: int,
                     n_input, ctx_len, kv_offset, out: int, sync: bool = True):
        n, c, o = _attn_host_arrays(n_input, ctx_len, kv_offset)
        check(lib.orca_op_attention(self._h, dtype, P(qkv), P(kv_layer), kv_slots, n_heads, head_dim, len(n),
                                    _ptr(n), _ptr(c), _ptr(o), P(out)), "orca_op_attention")
        if sync:
            self.sync()


def _attn_host_arrays(n_input, ctx_len, kv_offset):
    return _i32(n_input), _i32(ctx_len), _i64(kv_offset)


def attention_decode_noalloc(dtype: int, qkv: int, kv_layer: int, kv_slots: int, n_heads: int, head_dim: int,
                             ctx_len, kv_offset, out: int, stream: int = 0) -> None:
    """Decode attention without any device allocation (see orca.h); asynchronous."""
    c, o = _i32(ctx_len), _i64(kv_offset)
    check(lib.orca_attention_decode_noalloc(dtype, P(qkv), P(kv_layer), kv_slots, n_heads, head_dim, len(c), _ptr(c),
                                            _ptr(o), P(out), P(stream or None)), "orca_attention_decode_noalloc")


class Scheduler:
    """Iteration-level (mode 0) or request-level (mode 1) scheduler.  With
    ``engine=None`` it keeps its own host-side K/V pool and needs no GPU."""

    def __init__(self, max_batch: int, max_tokens: int, kv_slots: int = 0, kv_reserve: int = 0, mode: int = 0,
                 token_feedback: bool = False, engine: Optional[Engine] = None, chunked_prefill: bool = False,
                 n_workers: int = 1):
        self.cfg = SchedConfig(max_batch, max_tokens, kv_slots, kv_reserve, mode, int(token_feedback),
                               int(chunked_prefill), int(n_workers))
        self._h = P()
        self.engine = engine
        check(lib.orca_sched_create(C.byref(self.cfg), engine.handle if engine else None, C.byref(self._h)),
              "orca_sched_create")
        self._last = None

    def close(self):
        if self._h:
            lib.orca_sched_destroy(self._h)
            self._h = P()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def submit(self, rid: int, arrival: float, prompt: Sequence[int], out_len: int, ctx0: int = 0) -> int:
        p = _i32(prompt)
        off = C.c_int64(-1)
        check(lib.orca_sched_submit(self._h, rid, float(arrival), _ptr(p), len(p), out_len, ctx0, C.byref(off)),
              "orca_sched_submit")
        return off.value

    def set_token_feedback(self, enable: bool) -> None:
        check(lib.orca_sched_set_token_feedback(self._h, int(enable)), "orca_sched_set_token_feedback")

    def next(self):
        """Returns (status, BatchDesc or None); status 1 batch, 0 idle tick, 2 done, 3 wait for an open batch."""
        b = Batch()
        st = C.c_int32()
        check(lib.orca_sched_next(self._h, C.byref(b), C.byref(st)), "orca_sched_next")
        if st.value != 1:
            return st.value, None
        self._last = b
        return 1, BatchDesc.from_c(b)

    def next_raw(self):
        """Like next() but returns the scheduler-owned ctypes Batch (valid until the next call)."""
        b = Batch()
        st = C.c_int32()
        check(lib.orca_sched_next(self._h, C.byref(b), C.byref(st)), "orca_sched_next")
        return st.value, b

    def complete(self, next_tokens) -> None:
        t = _i32(next_tokens)
        check(lib.orca_sched_complete(self._h, _ptr(t)), "orca_sched_complete")

    def cancel(self, rid: int) -> None:
        check(lib.orca_sched_cancel(self._h, rid), "orca_sched_cancel")

    def stats(self) -> SchedStats:
        s = SchedStats()
        check(lib.orca_sched_stats_get(self._h, C.byref(s)), "orca_sched_stats_get")
        return s

    def request(self, rid: int) -> RequestInfo:
        r = RequestInfo()
        check(lib.orca_sched_request_get(self._h, rid, C.byref(r)), "orca_sched_request_get")
        return r

    def tokens(self, rid: int) -> np.ndarray:
        n = C.c_int32()
        check(lib.orca_sched_request_tokens(self._h, rid, None, 0, C.byref(n)), "orca_sched_request_tokens")
        out = np.zeros(n.value, np.int32)
        check(lib.orca_sched_request_tokens(self._h, rid, _ptr(out), n.value, C.byref(n)), "orca_sched_request_tokens")
        return out

    def run(self, max_iterations: int = 1 << 62) -> None:
        check(lib.orca_sched_run(self._h, max_iterations), "orca_sched_run")
