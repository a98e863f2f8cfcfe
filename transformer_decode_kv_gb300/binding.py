"""Thin ctypes binding of libllm (include/llm.h): argument marshalling only.

Every step of the decode path runs inside the library's CUDA kernels; this module only converts
Python/numpy/torch arguments into the C structs and pointers the C ABI takes. Importing it when
libllm.so has not been built raises an error: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Iterable, Optional, Sequence

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libllm.so")

F32, F16, BF16, Q8_0 = 0, 1, 2, 8
CTX_HOST_ONLY = 1
CTX_FUSED_STEP = 2
CTX_KV_SPLIT = 4


class HParams(C.Structure):
    _fields_ = [("n_layer", C.c_int32), ("n_embd", C.c_int32), ("n_head", C.c_int32),
                ("n_head_kv", C.c_int32), ("head_dim", C.c_int32), ("n_ff", C.c_int32),
                ("n_vocab", C.c_int32), ("rope_freq_base", C.c_float), ("rms_eps", C.c_float),
                ("rope_type", C.c_int32)]


class CParams(C.Structure):
    _fields_ = [("n_ctx", C.c_uint32), ("n_seq_max", C.c_uint32), ("n_batch", C.c_uint32),
                ("n_ubatch", C.c_uint32), ("type_k", C.c_int32), ("type_v", C.c_int32),
                ("stream", C.c_void_p), ("flags", C.c_uint32)]


class Batch(C.Structure):
    _fields_ = [("n_tokens", C.c_int32), ("token", C.POINTER(C.c_int32)),
                ("pos", C.POINTER(C.c_int32)), ("n_seq_id", C.POINTER(C.c_int32)),
                ("seq_id", C.POINTER(C.POINTER(C.c_int32))), ("logits", C.POINTER(C.c_int8))]


class SamplerParams(C.Structure):
    _fields_ = [("top_k", C.c_int32), ("top_p", C.c_float), ("min_p", C.c_float),
                ("temperature", C.c_float), ("repeat_penalty", C.c_float),
                ("penalty_tokens", C.POINTER(C.c_int32)), ("n_penalty_tokens", C.c_int32)]


class PerfData(C.Structure):
    _fields_ = [("n_decode_calls", C.c_int64), ("n_tokens", C.c_int64), ("n_ubatches", C.c_int64),
                ("n_graph_replays", C.c_int64), ("t_decode_ms", C.c_double),
                ("n_fused_steps", C.c_int64), ("n_defrags", C.c_int64),
                ("weight_device_bytes", C.c_int64)]


ABORT_CB = C.CFUNCTYPE(C.c_int, C.c_void_p)

# every symbol include/llm.h declares, with (restype, argtypes)
SIGNATURES = {
    "llm_cparams_default": (CParams, []),
    "llm_ctx_init": (C.c_void_p, [C.POINTER(HParams), C.POINTER(CParams)]),
    "llm_ctx_free": (None, [C.c_void_p]),
    "llm_load_weights": (C.c_int, [C.c_void_p, C.c_char_p, C.c_int32, C.POINTER(C.c_int64),
                                   C.c_void_p, C.c_size_t]),
    "llm_weights_ready": (C.c_int, [C.c_void_p]),
    "llm_decode": (C.c_int32, [C.c_void_p, Batch]),
    "llm_get_logits_ith": (C.POINTER(C.c_float), [C.c_void_p, C.c_int32]),
    "llm_get_argmax_ith": (C.c_int32, [C.c_void_p, C.c_int32]),
    "llm_n_outputs": (C.c_int32, [C.c_void_p]),
    "llm_seq_rm": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32, C.c_int32]),
    "llm_seq_pos_max": (C.c_int32, [C.c_void_p, C.c_int32]),
    "llm_seq_pos_min": (C.c_int32, [C.c_void_p, C.c_int32]),
    "llm_set_abort_callback": (None, [C.c_void_p, ABORT_CB, C.c_void_p]),
    "llm_n_ctx": (C.c_uint32, [C.c_void_p]),
    "llm_n_ctx_seq": (C.c_uint32, [C.c_void_p]),
    "llm_n_batch": (C.c_uint32, [C.c_void_p]),
    "llm_n_ubatch": (C.c_uint32, [C.c_void_p]),
    "llm_kv_used_cells": (C.c_int32, [C.c_void_p]),
    "llm_last_error": (C.c_char_p, [C.c_void_p]),
    "llm_perf": (None, [C.c_void_p, C.POINTER(PerfData)]),
    "llm_debug_last_slots": (C.c_int32, [C.c_void_p, C.POINTER(C.c_int32), C.c_int32]),
    "llm_debug_ubatch_mask": (C.c_int64, [C.c_void_p, C.c_int32, C.POINTER(C.c_uint8), C.c_int64,
                                          C.POINTER(C.c_int32)]),
    "llm_debug_capture": (C.c_int, [C.c_void_p, C.c_int]),
    "llm_debug_get_tensor": (C.c_int64, [C.c_void_p, C.c_char_p, C.c_int32,
                                         C.POINTER(C.c_float), C.c_int64]),
    "llm_debug_inject_fault": (C.c_int, [C.c_void_p, C.c_int32, C.c_int32]),
    "llm_debug_kv_raw": (C.c_int64, [C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_int64]),
    "llm_memory_update": (C.c_int, [C.c_void_p, C.c_int]),
    "llm_sample_ith": (C.c_int32, [C.c_void_p, C.c_int32, C.POINTER(SamplerParams), C.c_float]),
    "llm_debug_set_logits": (C.c_int, [C.c_void_p, C.c_int32, C.POINTER(C.c_float)]),
    "llm_debug_step_trace_enable": (C.c_int, [C.c_void_p, C.c_int]),
    "llm_debug_step_trace": (C.c_int64, [C.c_void_p, C.POINTER(C.c_uint64), C.c_int64,
                                         C.POINTER(C.c_int32), C.POINTER(C.c_int32)]),
    "llm_debug_kernel_timing": (C.c_int, [C.c_void_p, C.c_int]),
    "llm_gemm_bf16_noalloc": (C.c_int, [C.c_int32, C.c_void_p, C.c_int64, C.c_int64, C.c_void_p,
                                        C.c_int32, C.c_void_p, C.c_int32, C.c_int32]),
    "llm_debug_noalloc_scratch_poke": (C.c_int, [C.c_uint32]),
    "llm_debug_gemm_tn_f16_trace": (C.c_int64, [C.c_int32, C.c_void_p, C.c_int64, C.c_int64, C.c_void_p, C.c_int32,
                                              C.c_void_p, C.c_int32, C.c_int32, C.c_int32,
                                              C.POINTER(C.c_uint64), C.c_int64]),
    "llm_debug_gemm_tn_q8": (C.c_int, [C.c_int32, C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.c_void_p,
                                       C.c_int32, C.c_void_p, C.c_int32, C.c_int32, C.c_int32]),
    "llm_debug_gemm_tn_q8_trace": (C.c_int64, [C.c_int32, C.c_void_p, C.c_void_p, C.c_int64, C.c_int64,
                                             C.c_void_p, C.c_int32, C.c_void_p, C.c_int32, C.c_int32, C.c_int32,
                                             C.POINTER(C.c_uint64), C.c_int64]),
    "llm_debug_gemm_tn_f16": (C.c_int, [C.c_int32, C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.c_void_p,
                                        C.c_int32, C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_int32]),
    "llm_debug_gemm_bf16": (C.c_int, [C.c_int32, C.c_void_p, C.c_int64, C.c_int64, C.c_void_p,
                                      C.c_int32, C.c_void_p, C.c_int32, C.c_int32]),
    "llm_debug_kernel_stats": (C.c_int32, [C.c_void_p, C.c_int32, C.c_char_p, C.c_int32,
                                           C.POINTER(C.c_int64), C.POINTER(C.c_double),
                                           C.POINTER(C.c_double), C.POINTER(C.c_double)]),
}

_lib = None


def lib():
    """Load libllm.so (built by transformer_decode_kv_gb300.build); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m transformer_decode_kv_gb300.build`")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: np.ndarray, ct):
    return a.ctypes.data_as(C.POINTER(ct))


class LlmError(RuntimeError):
    pass


def debug_gemm_bf16(epi: int, W, X, Y, F: int = 0) -> int:
    """One tensor-core GEMM launch on torch CUDA tensors (W [rows][K] bf16, X [T][K] bf16)."""
    return lib().llm_debug_gemm_bf16(epi, C.c_void_p(W.data_ptr()), W.shape[0], W.shape[1],
                                     C.c_void_p(X.data_ptr()), X.shape[0], C.c_void_p(Y.data_ptr()),
                                     Y.stride(0), F)


def gemm_bf16_noalloc(epi: int, W, X, Y, F: int = 0) -> int:
    """The same GEMM through the entry point that allocates no device memory."""
    return lib().llm_gemm_bf16_noalloc(epi, C.c_void_p(W.data_ptr()), W.shape[0], W.shape[1],
                                       C.c_void_p(X.data_ptr()), X.shape[0],
                                       C.c_void_p(Y.data_ptr()), Y.stride(0), F)


def debug_gemm_tn_f16(epi: int, W, X, Y, F: int = 0, W_lo=None, splits: int = 1, one_cta: bool = False) -> int:
    """One token-major tensor-core GEMM launch on torch CUDA tensors (W [rows][K] f16, X [T][K] f16)."""
    M = W.shape[0] if epi != 2 else 0
    return lib().llm_debug_gemm_tn_f16(epi, C.c_void_p(W.data_ptr()),
                                       C.c_void_p(W_lo.data_ptr()) if W_lo is not None else None,
                                       M, W.shape[1], C.c_void_p(X.data_ptr()), X.shape[0],
                                       C.c_void_p(Y.data_ptr()), Y.stride(0), F, splits, int(one_cta))


def debug_gemm_tn_q8(epi: int, Wq, Ws, X, Y, F: int = 0, splits: int = 1) -> int:
    """The token-major GEMM over a Q8_0 weight (Wq int8 [rows][K], Ws f16 scales [rows][K / 32], X f16
    [T][K]) dequantised inside the kernel."""
    M = Wq.shape[0] if epi != 2 else 0
    return lib().llm_debug_gemm_tn_q8(epi, C.c_void_p(Wq.data_ptr()), C.c_void_p(Ws.data_ptr()), M, Wq.shape[1],
                                      C.c_void_p(X.data_ptr()), X.shape[0], C.c_void_p(Y.data_ptr()), Y.stride(0),
                                      F, splits)


def debug_gemm_tn_q8_trace(epi: int, Wq, Ws, X, Y, F: int = 0, splits: int = 1):
    """The Q8_0 token-major GEMM with its per-CTA counters: returns (status, [n_cta, 8] uint64)."""
    M = Wq.shape[0] if epi != 2 else 0
    cap = 8 * 8192
    out = np.zeros(cap, dtype=np.uint64)
    n = lib().llm_debug_gemm_tn_q8_trace(epi, C.c_void_p(Wq.data_ptr()), C.c_void_p(Ws.data_ptr()), M, Wq.shape[1],
                                         C.c_void_p(X.data_ptr()), X.shape[0], C.c_void_p(Y.data_ptr()), Y.stride(0),
                                         F, splits, out.ctypes.data_as(C.POINTER(C.c_uint64)), cap)
    return (0, out[:n].reshape(-1, 8)) if n > 0 else (int(n), None)


def debug_gemm_tn_f16_trace(epi: int, W, X, Y, F: int = 0, splits: int = 1):
    """The two-CTA token-major GEMM with its per-CTA timeline: returns (status, [n_cta, 8] uint64)."""
    M = W.shape[0] if epi != 2 else 0
    cap = 8 * 4096
    out = np.zeros(cap, dtype=np.uint64)
    n = lib().llm_debug_gemm_tn_f16_trace(epi, C.c_void_p(W.data_ptr()), M, W.shape[1], C.c_void_p(X.data_ptr()),
                                          X.shape[0], C.c_void_p(Y.data_ptr()), Y.stride(0), F, splits,
                                          out.ctypes.data_as(C.POINTER(C.c_uint64)), cap)
    return (0, out[:n].reshape(-1, 8)) if n > 0 else (int(n), None)


def debug_noalloc_scratch_poke(value: int) -> int:
    """Plant a value in the allocation-free GEMM's error word on the current device."""
    return lib().llm_debug_noalloc_scratch_poke(value)


class Context:
    """One llm_ctx: a model's weights, a unified KV cache and the decode state."""

    def __init__(self, hp, n_ctx: int, n_seq_max: int = 1, type_k: int = F16, type_v: int = F16,
                 n_batch: int = 2048, n_ubatch: int = 512, stream: Optional[int] = None,
                 host_only: bool = False, fused_step: bool = False, kv_unified: bool = True):
        L = lib()
        self._hp = HParams(hp.n_layer, hp.n_embd, hp.n_head, hp.n_head_kv, hp.head_dim, hp.n_ff,
                           hp.n_vocab, hp.rope_freq_base, hp.rms_eps, getattr(hp, "rope_type", 0))
        cp = L.llm_cparams_default()
        cp.n_ctx, cp.n_seq_max, cp.n_batch, cp.n_ubatch = n_ctx, n_seq_max, n_batch, n_ubatch
        cp.type_k, cp.type_v = type_k, type_v
        cp.stream = stream
        cp.flags = ((CTX_HOST_ONLY if host_only else 0) | (CTX_FUSED_STEP if fused_step else 0) |
                    (0 if kv_unified else CTX_KV_SPLIT))
        self.n_vocab = hp.n_vocab
        self.type_k = type_k
        self.ptr = L.llm_ctx_init(C.byref(self._hp), C.byref(cp))
        if not self.ptr:
            raise LlmError("llm_ctx_init failed: " + L.llm_last_error(None).decode())
        self._abort = None

    # ---- lifetime
    def free(self):
        if self.ptr:
            lib().llm_ctx_free(self.ptr)
            self.ptr = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass

    def last_error(self) -> str:
        return lib().llm_last_error(self.ptr).decode()

    # ---- weights
    def load_weight(self, name: str, wtype: int, shape: Sequence[int], data) -> int:
        """data: a torch tensor (host or CUDA) or numpy array holding the storage bytes."""
        ne = (C.c_int64 * 2)(int(shape[0]), int(shape[1]) if len(shape) > 1 else 1)
        if hasattr(data, "data_ptr"):
            t = data.contiguous()
            ptr, nbytes = t.data_ptr(), t.numel() * t.element_size()
            keep = t
        else:
            keep = np.ascontiguousarray(data)
            ptr, nbytes = keep.ctypes.data, keep.nbytes
        r = lib().llm_load_weights(self.ptr, name.encode(), wtype, ne, C.c_void_p(ptr), nbytes)
        del keep
        return r

    def load_all(self, tensors: Iterable) -> None:
        """Load (name, wtype, shape, storage) tuples; raise on the first failure."""
        for name, wt, shape, t in tensors:
            if self.load_weight(name, wt, shape, t) != 0:
                raise LlmError(f"load {name}: {self.last_error()}")
        if lib().llm_weights_ready(self.ptr) != 0:
            raise LlmError(self.last_error())

    def weights_ready(self) -> int:
        return lib().llm_weights_ready(self.ptr)

    # ---- decode
    def decode(self, tokens, pos=None, seq_ids=None, logits=None) -> int:
        """tokens: ints; pos: ints or None; seq_ids: list of lists (or ints) or None;
        logits: flags or None. Returns llm_decode's status."""
        tok = _i32(tokens)
        n = len(tok)
        keep = [tok]
        b = Batch()
        b.n_tokens = n
        b.token = _ptr(tok, C.c_int32)
        if pos is not None:
            p = _i32(pos); keep.append(p); b.pos = _ptr(p, C.c_int32)
        if seq_ids is not None:
            # one flat id array; row i's pointer is its start inside it
            if len(seq_ids) != n:
                raise ValueError("seq_ids needs one row per token")
            rows = [r if hasattr(r, "__len__") else (r,) for r in seq_ids]
            nsid = np.fromiter((len(r) for r in rows), dtype=np.int32, count=n)
            flat = np.fromiter((x for r in rows for x in r), dtype=np.int32, count=int(nsid.sum()))
            start = np.zeros(n, dtype=np.uint64)
            np.cumsum(nsid[:-1], out=start[1:])
            ptrs = np.ascontiguousarray(np.uint64(flat.ctypes.data) + np.uint64(4) * start)
            keep += [nsid, flat, ptrs]
            b.n_seq_id = _ptr(nsid, C.c_int32)
            b.seq_id = ptrs.ctypes.data_as(C.POINTER(C.POINTER(C.c_int32)))
        if logits is not None:
            lg = np.ascontiguousarray(np.asarray(logits, dtype=np.int8)); keep.append(lg)
            b.logits = _ptr(lg, C.c_int8)
        return lib().llm_decode(self.ptr, b)

    def get_logits_ith(self, i: int) -> Optional[np.ndarray]:
        p = lib().llm_get_logits_ith(self.ptr, i)
        if not p:
            return None
        return np.ctypeslib.as_array(p, shape=(self.n_vocab,)).copy()

    def sample_ith(self, i: int, top_k: int = 40, top_p: float = 1.0, min_p: float = 0.0,
                   temperature: float = 1.0, repeat_penalty: float = 1.0, penalty_tokens=(),
                   u: float = 0.0) -> int:
        """The device sampler chain over logits row i; u in [0, 1) is the uniform draw."""
        pen = np.asarray(list(penalty_tokens), dtype=np.int32)
        p = SamplerParams(top_k, top_p, min_p, temperature, repeat_penalty,
                          pen.ctypes.data_as(C.POINTER(C.c_int32)) if len(pen) else None, len(pen))
        return lib().llm_sample_ith(self.ptr, i, C.byref(p), u)

    def debug_set_logits(self, i: int, row) -> int:
        r = np.ascontiguousarray(row, dtype=np.float32)
        assert r.shape == (self.n_vocab,)
        return lib().llm_debug_set_logits(self.ptr, i, _ptr(r, C.c_float))

    def get_argmax_ith(self, i: int) -> int:
        return lib().llm_get_argmax_ith(self.ptr, i)

    @property
    def n_outputs(self) -> int:
        return lib().llm_n_outputs(self.ptr)

    # ---- memory
    def seq_rm(self, seq: int, p0: int, p1: int) -> int:
        return lib().llm_seq_rm(self.ptr, seq, p0, p1)

    def memory_update(self, optimize: bool = True) -> int:
        return lib().llm_memory_update(self.ptr, int(optimize))

    def seq_pos_max(self, s: int) -> int:
        return lib().llm_seq_pos_max(self.ptr, s)

    def seq_pos_min(self, s: int) -> int:
        return lib().llm_seq_pos_min(self.ptr, s)

    def set_abort_callback(self, fn):
        """fn() -> bool, or None to remove."""
        if fn is None:
            self._abort = None
            lib().llm_set_abort_callback(self.ptr, ABORT_CB(), None)
            return
        self._abort = ABORT_CB(lambda _ud: 1 if fn() else 0)
        lib().llm_set_abort_callback(self.ptr, self._abort, None)

    @property
    def n_ctx(self) -> int:
        return lib().llm_n_ctx(self.ptr)

    @property
    def n_ctx_seq(self) -> int:
        return lib().llm_n_ctx_seq(self.ptr)

    @property
    def n_batch(self) -> int:
        return lib().llm_n_batch(self.ptr)

    @property
    def n_ubatch(self) -> int:
        return lib().llm_n_ubatch(self.ptr)

    def kv_used_cells(self) -> int:
        return lib().llm_kv_used_cells(self.ptr)

    def perf(self) -> dict:
        d = PerfData()
        lib().llm_perf(self.ptr, C.byref(d))
        return {k: getattr(d, k) for k, _ in PerfData._fields_}

    # ---- debug hooks
    def last_slots(self) -> np.ndarray:
        n = lib().llm_debug_last_slots(self.ptr, None, 0)
        out = np.zeros(n, dtype=np.int32)
        lib().llm_debug_last_slots(self.ptr, _ptr(out, C.c_int32), n)
        return out

    def ubatch_mask(self, ub: int):
        nkv = C.c_int32(0)
        n = lib().llm_debug_ubatch_mask(self.ptr, ub, None, 0, C.byref(nkv))
        if n == 0 and nkv.value == 0:
            return None
        out = np.zeros(n, dtype=np.uint8)
        lib().llm_debug_ubatch_mask(self.ptr, ub, _ptr(out, C.c_uint8), n, C.byref(nkv))
        return out.reshape(-1, nkv.value).astype(bool) if nkv.value else out.reshape(0, 0)

    def debug_capture(self, enable: bool = True) -> int:
        return lib().llm_debug_capture(self.ptr, int(enable))

    def debug_tensor(self, name: str, layer: int = 0) -> Optional[np.ndarray]:
        n = lib().llm_debug_get_tensor(self.ptr, name.encode(), layer, None, 0)
        if n <= 0:
            return None
        out = np.zeros(n, dtype=np.float32)
        lib().llm_debug_get_tensor(self.ptr, name.encode(), layer, _ptr(out, C.c_float), n)
        return out

    def kv_cache(self, layer: int, which: int) -> Optional[np.ndarray]:
        """Layer `layer`'s K (which 0) or V (which 1) cache as stored, [n_head_kv][n_ctx][head_dim]
        (float32 or float16 elements). A Q8_0 cache comes back as its 34-byte blocks (fp16 scale,
        then 32 int8 quants), uint8 [n_head_kv][n_ctx][head_dim / 32 * 34]."""
        n = lib().llm_debug_kv_raw(self.ptr, layer, which, None, 0)
        if n <= 0:
            return None
        out = np.zeros(n, dtype=np.uint8)
        lib().llm_debug_kv_raw(self.ptr, layer, which, out.ctypes.data_as(C.c_void_p), n)
        Hkv, hd = self._hp.n_head_kv, self._hp.head_dim
        if self.type_k == Q8_0:
            nq = n // 34 * 32
            q = out[:nq].reshape(Hkv, -1, hd // 32, 32)
            s = out[nq:].reshape(Hkv, -1, hd // 32, 2)
            return np.concatenate([s, q], axis=3).reshape(Hkv, -1, hd // 32 * 34)
        es = 4 if n // (self._hp.n_head_kv * self._hp.head_dim) == 4 * self.n_ctx else 2
        v = out.view(np.float32 if es == 4 else np.float16)
        return v.reshape(self._hp.n_head_kv, -1, self._hp.head_dim)

    def kv_f16_copy(self, which: int) -> Optional[np.ndarray]:
        """Q8_0 caches: the f16 copy of the K (which 0) or V (which 1) quants that the last
        attention over query tiles of several tokens read, float16 [n_head_kv][n_ctx][head_dim]
        (cells below that ubatch's n_kv are valid)."""
        n = lib().llm_debug_kv_raw(self.ptr, 0, which + 2, None, 0)
        if n <= 0:
            return None
        out = np.zeros(n, dtype=np.uint8)
        lib().llm_debug_kv_raw(self.ptr, 0, which + 2, out.ctypes.data_as(C.c_void_p), n)
        return out.view(np.float16).reshape(self._hp.n_head_kv, -1, self._hp.head_dim)

    def step_trace_enable(self, enable: bool = True) -> int:
        return lib().llm_debug_step_trace_enable(self.ptr, int(enable))

    def step_trace(self) -> Optional[np.ndarray]:
        """The last traced one-token step as uint64 [blocks][slots][2] (start, end) ns stamps."""
        nb, ns = C.c_int32(0), C.c_int32(0)
        n = lib().llm_debug_step_trace(self.ptr, None, 0, C.byref(nb), C.byref(ns))
        if n <= 0:
            return None
        out = np.zeros(n, dtype=np.uint64)
        lib().llm_debug_step_trace(self.ptr, out.ctypes.data_as(C.POINTER(C.c_uint64)), n, None, None)
        return out.reshape(nb.value, ns.value, 2)

    def kernel_timing(self, enable: bool = True) -> int:
        return lib().llm_debug_kernel_timing(self.ptr, int(enable))

    def kernel_stats(self) -> dict:
        """{class name: {launches, ms, bytes, flops}} of the timed launches."""
        L = lib()
        n = L.llm_debug_kernel_stats(self.ptr, 0, None, 0, None, None, None, None)
        out = {}
        for i in range(n):
            name = C.create_string_buffer(64)
            la, ms, by, fl = C.c_int64(), C.c_double(), C.c_double(), C.c_double()
            L.llm_debug_kernel_stats(self.ptr, i, name, 64, C.byref(la), C.byref(ms), C.byref(by),
                                     C.byref(fl))
            out[name.value.decode()] = {"launches": la.value, "ms": ms.value, "bytes": by.value,
                                        "flops": fl.value}
        return out

    def inject_fault(self, kind: int, ub: int = 0) -> int:
        return lib().llm_debug_inject_fault(self.ptr, kind, ub)
