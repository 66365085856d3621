"""Thin ctypes binding of libmb.so (include/mb.h).

Argument marshalling only: every function here forwards to the C entry point
of the same name.  Pointers are plain integers (device addresses for device
buffers); objects with a ``data_ptr()`` method (torch tensors) are accepted
and reduced to that address.  A non-OK status raises ``MbError`` carrying the
library's message.  There is no fallback: if the library is missing, loading
fails loudly.
"""

from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Sequence

import numpy as np

from . import build as _build

MB_OK, MB_EINVAL, MB_ENOMEM, MB_ENOSPACE, MB_ECUDA, MB_EUNSUPPORTED, MB_EDEVICE = 0, -1, -2, -3, -4, -5, -6
STATUS_NAMES = {0: "MB_OK", -1: "MB_EINVAL", -2: "MB_ENOMEM", -3: "MB_ENOSPACE", -4: "MB_ECUDA",
                -5: "MB_EUNSUPPORTED", -6: "MB_EDEVICE"}
TIMED_KERNELS = ("rmsnorm_attn", "gemm_qkv", "rope_append", "attention", "attn_merge", "gemm_o",
                 "rmsnorm_ffn", "gemm_gate_up", "gemm_down")
BUF_XN, BUF_QKV, BUF_Q, BUF_O, BUF_H, BUF_HN, BUF_A = range(7)


class MbError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


c_int32_p = ctypes.POINTER(ctypes.c_int32)
c_int64_p = ctypes.POINTER(ctypes.c_int64)


class mb_layer_desc(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("rms_eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float), ("qk_norm", ctypes.c_int32), ("max_tokens", ctypes.c_int32)]


class mb_layer_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("g_attn", "w_qkv", "g_q", "g_k", "w_o", "g_ffn", "w_gate_up", "w_down")]


class mb_batch(ctypes.Structure):
    _fields_ = [("num_reqs", ctypes.c_int32), ("qo_indptr", c_int32_p), ("kv_len", c_int32_p),
                ("bt_indptr", c_int32_p), ("bt", c_int32_p)]


class mb_pack_cfg(ctypes.Structure):
    _fields_ = [("budget", ctypes.c_int32), ("max_seqs", ctypes.c_int32), ("chunk_cap", ctypes.c_int32)]


class mb_sched_batch(ctypes.Structure):
    _fields_ = [("batch", mb_batch), ("req_ids", c_int64_p)]


_LIB: Optional[ctypes.CDLL] = None
_VP = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SIGS = {
    "mb_layer_create": (_I32, [ctypes.POINTER(mb_layer_desc), ctypes.POINTER(mb_layer_weights), ctypes.POINTER(_VP)]),
    "mb_destroy": (_I32, [_VP]),
    "mb_kv_alloc": (_I32, [_VP, _I32, _VP, ctypes.POINTER(_VP)]),
    "mb_kv_layout": (_I32, [_VP, c_int64_p, ctypes.POINTER(_VP)]),
    "mb_kv_free": (_I32, [_VP]),
    "mb_step": (_I32, [_VP, _VP, ctypes.POINTER(mb_batch), _VP, _VP, _VP]),
    "mb_batch_validate": (_I32, [ctypes.POINTER(mb_batch), _I32, _I32]),
    "mb_device_status": (_I32, [_VP, _VP]),
    "mb_layer_buffer": (_I32, [_VP, _I32, ctypes.POINTER(_VP), c_int64_p]),
    "mb_layer_set_timing": (_I32, [_VP, _I32]),
    "mb_layer_timing": (_I32, [_VP, ctypes.POINTER(ctypes.c_double), _I32, c_int64_p]),
    "mb_layer_last_launches": (_I32, [_VP]),
    "mb_layer_last_upload_bytes": (_I64, [_VP]),
    "mb_gemm": (_I32, [_VP, _VP, _VP, _VP, _I32, _I32, _I32, _I32, _VP, _VP]),
    "mb_gemm_workspace_bytes": (_I64, []),
    "mb_gemm_noalloc": (_I32, [_VP, _VP, _VP, _VP, _I32, _I32, _I32, _I32, _VP]),
    "mb_gemm_set_split_wait": (_I32, [_I64, _I32]),
    "mb_stack_create": (_I32, [ctypes.POINTER(_VP), _I32, _I32, ctypes.POINTER(_VP)]),
    "mb_stack_step": (_I32, [_VP, ctypes.POINTER(_VP), ctypes.POINTER(mb_batch), _VP, _VP, _VP]),
    "mb_stack_last_launches": (_I32, [_VP]),
    "mb_stack_destroy": (_I32, [_VP]),
    "mb_sched_create": (_I32, [ctypes.POINTER(mb_pack_cfg), _I32, c_int32_p, ctypes.POINTER(_VP)]),
    "mb_sched_add": (_I32, [_VP, _I64, _I32, _I32]),
    "mb_sched_pack": (_I32, [_VP, ctypes.POINTER(mb_sched_batch)]),
    "mb_sched_finish": (_I32, [_VP, _I64]),
    "mb_sched_set_adaptive": (_I32, [_VP, _I32, _I32, _I32, _I32]),
    "mb_layer_set_decode_sms": (_I32, [_VP, _I32]),
    "mb_layer_set_gemm_sms": (_I32, [_VP, _I32]),
    "mb_layer_set_gemm_workspace": (_I32, [_VP, _VP]),
    "mb_sample_greedy": (_I32, [_VP, _I32, _VP, _I32, _I32, ctypes.c_float, _VP, _VP, _I32, _VP, _VP, _VP, _VP]),
    "mb_embed": (_I32, [_VP, _I32, _I32, _VP, _I32, _VP, _VP]),
    "mb_sched_counts": (_I32, [_VP, c_int32_p]),
    "mb_sched_save": (_I32, [_VP, c_int64_p, _I64, c_int64_p]),
    "mb_sched_load": (_I32, [c_int64_p, _I64, ctypes.POINTER(_VP)]),
    "mb_sched_destroy": (_I32, [_VP]),
    "mb_last_error": (ctypes.c_char_p, []),
}


def lib_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libmb.so (built by ``build.build()``); raise if it is missing."""
    global _LIB
    if _LIB is None:
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run mixed_prefill_decode_gb300.build.build() first")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def header_symbols() -> list:
    """Entry points declared in include/mb.h."""
    hdr = os.path.join(_build.INCLUDE, "mb.h")
    text = open(hdr).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s+\*?\s*(mb_[a-z_0-9]+)\s*\(", text, re.M)))


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    return int(x)


def _check(st: int) -> None:
    if st != MB_OK:
        msg = lib().mb_last_error()
        raise MbError(st, msg.decode() if msg else "")


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _as_i32p(a: np.ndarray):
    return a.ctypes.data_as(c_int32_p)


class Batch:
    """Host-side descriptor holder: keeps the int32 arrays alive."""

    def __init__(self, qo_indptr, kv_len, bt_indptr, bt):
        self.qo_indptr = _i32(qo_indptr)
        self.kv_len = _i32(kv_len)
        self.bt_indptr = _i32(bt_indptr)
        self.bt = _i32(bt) if len(bt) else np.zeros(1, np.int32)
        self.c = mb_batch(len(self.kv_len), _as_i32p(self.qo_indptr), _as_i32p(self.kv_len),
                          _as_i32p(self.bt_indptr), _as_i32p(self.bt))

    @classmethod
    def of(cls, b) -> "Batch":
        return cls(b.qo_indptr, b.kv_len, b.bt_indptr, b.bt)


# ----------------------------------------------------------------- layer
def mb_layer_create(desc: mb_layer_desc, weights: mb_layer_weights) -> int:
    h = _VP()
    _check(lib().mb_layer_create(ctypes.byref(desc), ctypes.byref(weights), ctypes.byref(h)))
    return h.value


def mb_destroy(layer: int) -> None:
    _check(lib().mb_destroy(layer))


def mb_kv_alloc(layer: int, num_pages: int, dev_buf=None) -> int:
    h = _VP()
    _check(lib().mb_kv_alloc(layer, num_pages, _ptr(dev_buf), ctypes.byref(h)))
    return h.value


def mb_kv_layout(kv: int):
    strides = (ctypes.c_int64 * 5)()
    base = _VP()
    _check(lib().mb_kv_layout(kv, strides, ctypes.byref(base)))
    return list(strides), base.value


def mb_kv_free(kv: int) -> None:
    _check(lib().mb_kv_free(kv))


def mb_step(layer: int, kv: int, batch: Batch, x_in, x_out, stream=None) -> None:
    _check(lib().mb_step(layer, kv, ctypes.byref(batch.c), _ptr(x_in), _ptr(x_out), _ptr(stream)))


def mb_batch_validate(batch: Batch, num_pages: int, max_tokens: int) -> None:
    _check(lib().mb_batch_validate(ctypes.byref(batch.c), num_pages, max_tokens))


def mb_device_status(layer: Optional[int], stream=None) -> None:
    _check(lib().mb_device_status(layer, _ptr(stream)))


def mb_layer_buffer(layer: int, which: int):
    p = _VP()
    n = ctypes.c_int64()
    _check(lib().mb_layer_buffer(layer, which, ctypes.byref(p), ctypes.byref(n)))
    return p.value, n.value


def mb_layer_set_timing(layer: int, enable: bool) -> None:
    _check(lib().mb_layer_set_timing(layer, 1 if enable else 0))


def mb_layer_set_decode_sms(layer: int, n: int) -> None:
    _check(lib().mb_layer_set_decode_sms(layer, n))


def mb_layer_set_gemm_sms(layer: int, n: int) -> None:
    _check(lib().mb_layer_set_gemm_sms(layer, n))


def mb_layer_set_gemm_workspace(layer: int, workspace=None) -> None:
    _check(lib().mb_layer_set_gemm_workspace(layer, _ptr(workspace)))


def mb_layer_timing(layer: int):
    ms = (ctypes.c_double * len(TIMED_KERNELS))()
    steps = ctypes.c_int64()
    _check(lib().mb_layer_timing(layer, ms, len(TIMED_KERNELS), ctypes.byref(steps)))
    return dict(zip(TIMED_KERNELS, list(ms))), steps.value


def mb_layer_last_launches(layer: int) -> int:
    return int(lib().mb_layer_last_launches(layer))


def mb_layer_last_upload_bytes(layer: int) -> int:
    return int(lib().mb_layer_last_upload_bytes(layer))


def mb_gemm(A, B, D, R, M: int, N: int, K: int, epilogue: int, workspace=None, stream=None) -> None:
    _check(lib().mb_gemm(_ptr(A), _ptr(B), _ptr(D), _ptr(R), M, N, K, epilogue, _ptr(workspace), _ptr(stream)))


def mb_gemm_noalloc(A, B, D, R, M: int, N: int, K: int, epilogue: int, stream=None) -> None:
    _check(lib().mb_gemm_noalloc(_ptr(A), _ptr(B), _ptr(D), _ptr(R), M, N, K, epilogue, _ptr(stream)))


def mb_gemm_set_split_wait(limit_ns: int, phantom_pieces: int = 0) -> None:
    _check(lib().mb_gemm_set_split_wait(int(limit_ns), int(phantom_pieces)))


def mb_gemm_workspace_bytes() -> int:
    return int(lib().mb_gemm_workspace_bytes())


# ----------------------------------------------------------------- stack
def mb_stack_create(layers: Sequence[int], use_graphs: bool = True) -> int:
    arr = (_VP * len(layers))(*layers)
    h = _VP()
    _check(lib().mb_stack_create(arr, len(layers), 1 if use_graphs else 0, ctypes.byref(h)))
    return h.value


def mb_stack_step(stack: int, kvs: Sequence[int], batch: Batch, x_in, x_out, stream=None) -> None:
    arr = (_VP * len(kvs))(*kvs)
    _check(lib().mb_stack_step(stack, arr, ctypes.byref(batch.c), _ptr(x_in), _ptr(x_out), _ptr(stream)))


def mb_stack_last_launches(stack: int) -> int:
    return int(lib().mb_stack_last_launches(stack))


def mb_stack_destroy(stack: int) -> None:
    _check(lib().mb_stack_destroy(stack))


# ----------------------------------------------------------- next tokens
def mb_sample_greedy(x, T: int, rows, n_rows: int, d: int, eps: float, g_final, w_lm, vocab: int, y_work, logits,
                     ids, stream=None) -> None:
    _check(lib().mb_sample_greedy(_ptr(x), T, _ptr(rows), n_rows, d, eps, _ptr(g_final), _ptr(w_lm), vocab,
                                  _ptr(y_work), _ptr(logits), _ptr(ids), stream))


def mb_embed(table, vocab: int, d: int, ids, n: int, out, stream=None) -> None:
    _check(lib().mb_embed(_ptr(table), vocab, d, _ptr(ids), n, _ptr(out), stream))


# ------------------------------------------------------------- scheduler
def mb_sched_create(budget: int, max_seqs: int, chunk_cap: int, free_order: Sequence[int]) -> int:
    fo = _i32(free_order)
    cfg = mb_pack_cfg(budget, max_seqs, chunk_cap)
    h = _VP()
    _check(lib().mb_sched_create(ctypes.byref(cfg), len(fo), _as_i32p(fo) if len(fo) else None, ctypes.byref(h)))
    return h.value


def mb_sched_add(s: int, req_id: int, prompt_len: int, computed: int = 0) -> None:
    _check(lib().mb_sched_add(s, req_id, prompt_len, computed))


def mb_sched_pack(s: int):
    """Returns (qo_indptr, kv_len, bt_indptr, bt, req_ids) as NumPy copies."""
    out = mb_sched_batch()
    _check(lib().mb_sched_pack(s, ctypes.byref(out)))
    n = out.batch.num_reqs
    qo = np.ctypeslib.as_array(out.batch.qo_indptr, shape=(n + 1,)).copy()
    kv = np.ctypeslib.as_array(out.batch.kv_len, shape=(n,)).copy() if n else np.zeros(0, np.int32)
    bti = np.ctypeslib.as_array(out.batch.bt_indptr, shape=(n + 1,)).copy()
    nb = int(bti[-1])
    bt = np.ctypeslib.as_array(out.batch.bt, shape=(nb,)).copy() if nb else np.zeros(0, np.int32)
    ids = np.ctypeslib.as_array(out.req_ids, shape=(n,)).copy() if n else np.zeros(0, np.int64)
    return qo, kv, bti, bt, ids


def mb_sched_finish(s: int, req_id: int) -> None:
    _check(lib().mb_sched_finish(s, req_id))


def mb_sched_set_adaptive(s: int, min_chunk: int, base_chunk: int = 512, max_chunk: int = 4096,
                          decode_pressure: int = 16) -> None:
    _check(lib().mb_sched_set_adaptive(s, min_chunk, base_chunk, max_chunk, decode_pressure))


def mb_sched_counts(s: int):
    c = (ctypes.c_int32 * 4)()
    _check(lib().mb_sched_counts(s, c))
    return tuple(c)


def mb_sched_save(s: int) -> np.ndarray:
    """The packer's state as int64 words (layout in include/mb.h)."""
    n = ctypes.c_int64()
    _check(lib().mb_sched_save(s, None, 0, ctypes.byref(n)))
    buf = np.zeros(max(1, n.value), dtype=np.int64)
    _check(lib().mb_sched_save(s, buf.ctypes.data_as(c_int64_p), n.value, ctypes.byref(n)))
    return buf[:n.value].copy()


def mb_sched_load(words) -> int:
    """A new scheduler from mb_sched_save's words."""
    w = np.ascontiguousarray(np.asarray(words, dtype=np.int64))
    h = _VP()
    _check(lib().mb_sched_load(w.ctypes.data_as(c_int64_p), len(w), ctypes.byref(h)))
    return h.value


def mb_sched_destroy(s: int) -> None:
    _check(lib().mb_sched_destroy(s))


# ------------------------------------------------------------ convenience
class Layer:
    """A layer handle plus its KV pool (weights stay owned by the caller)."""

    def __init__(self, shape: dict, weights: dict, max_tokens: int, num_pages: int, kv_buf=None):
        self.desc = mb_layer_desc(shape["d_model"], shape["n_q_heads"], shape["n_kv_heads"], shape["head_dim"],
                                  shape["d_ff"], shape["rms_eps"], shape["rope_theta"], shape["qk_norm"],
                                  max_tokens)
        self.w = mb_layer_weights(*[_ptr(weights.get(k)) for k in
                                    ("g_attn", "w_qkv", "g_q", "g_k", "w_o", "g_ffn", "w_gate_up", "w_down")])
        # the library holds raw device pointers: keep the caller's tensors
        # (weights, and a KV buffer it hands in) alive as long as the layer
        self._keep = weights
        self._kv_buf = kv_buf
        self.handle = mb_layer_create(self.desc, self.w)
        self.kv = mb_kv_alloc(self.handle, num_pages, kv_buf)

    def step(self, batch: Batch, x_in, x_out, stream=None) -> None:
        mb_step(self.handle, self.kv, batch, x_in, x_out, stream)

    def buffer(self, which: int):
        return mb_layer_buffer(self.handle, which)

    def close(self) -> None:
        if self.handle:
            mb_kv_free(self.kv)
            mb_destroy(self.handle)
            self.handle = None
