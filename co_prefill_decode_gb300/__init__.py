"""Python binding of libcf, the GB300 co-batched layer-step library.

Argument marshalling only: every step of the layer runs in the CUDA kernels
behind the C ABI declared in include/cf.h.  Tensors are passed as raw device
pointers (``tensor.data_ptr()``) and streams as ``torch.cuda.Stream``
handles; PyTorch only provides device memory and streams.  There is no CPU
fallback: importing works without a GPU, but every call needs the built
library (``python -m co_prefill_decode_gb300.build``) and a CUDA device.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcf.so")

CF_OK, CF_ERR_INVALID_ARG, CF_ERR_UNSUPPORTED, CF_ERR_CUDA, CF_ERR_TIMEOUT, CF_ERR_OOM, CF_ERR_DEVICE = range(7)
CF_EPI_NONE, CF_EPI_RESID_F32, CF_EPI_RESID_BF16, CF_EPI_SWIGLU = range(4)
PHASES = ("rmsnorm", "qkv", "decode", "prefill", "fork", "oproj", "rmsnorm2", "gateup", "down", "step",
          "fork_in", "fork_out")

# every symbol include/cf.h declares
EXPORTS = (
    "cf_device_sm_count", "cf_create", "cf_destroy", "cf_layer_step", "cf_decode_attn",
    "cf_prefill_attn", "cf_gemm", "cf_kv_append", "cf_get_error", "cf_engine_buffer",
    "cf_engine_decode_sms", "cf_set_decode_sms", "cf_set_profiling", "cf_get_phase_times",
    "cf_launch_count", "cf_rmsnorm", "cf_qkv", "cf_decode_attn_noalloc", "cf_calibrate_decode_sms",
    "cf_calibration_points", "cf_gemm_schedule", "cf_set_split_k", "cf_prefill_plan", "cf_decode_plan", "cf_selftest_timeout", "cf_set_prefill_pairing", "cf_set_graphs", "cf_graph_captures",
    "cf_latency_predict", "cf_latency_fit_line", "cf_latency_calibrate", "cf_waterfill_dispatch",
    "cf_waterfill_assign", "cf_prefill_attn_varlen", "cf_set_prefill_split", "cf_set_fork_mode",
)


class CfError(RuntimeError):
    def __init__(self, status: int, msg: str = ""):
        super().__init__(f"libcf status {status}: {msg}")
        self.status = status


class cf_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("ffn_dim", ctypes.c_int), ("page_size", ctypes.c_int),
                ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float), ("qk_norm", ctypes.c_int),
                ("max_tokens", ctypes.c_int), ("max_decode", ctypes.c_int), ("decode_sms", ctypes.c_int)]


class cf_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_qkv", "w_o", "w_gate", "w_up", "w_down", "g_attn", "g_ffn", "g_q", "g_k")]


class cf_kv_pool(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("num_pages", ctypes.c_int)]


class cf_batch(ctypes.Structure):
    _fields_ = [("n_decode", ctypes.c_int), ("dec_ctx", ctypes.c_void_p), ("dec_pages", ctypes.c_void_p),
                ("dec_stride", ctypes.c_int), ("prefill_len", ctypes.c_int), ("prefill_prefix", ctypes.c_int),
                ("pre_pages", ctypes.c_void_p), ("n_chunks", ctypes.c_int),
                ("chunk_len", ctypes.POINTER(ctypes.c_int)), ("chunk_prefix", ctypes.POINTER(ctypes.c_int)),
                ("chunk_pages", ctypes.c_void_p), ("chunk_stride", ctypes.c_int)]


class cf_latency_model(ctypes.Structure):
    _fields_ = [(n, ctypes.c_double) for n in
                ("gamma", "gamma0", "a_d", "a_d0", "a_p", "a_p0", "a_comm", "a_comm0", "alpha", "beta")]


class cf_rank_load(ctypes.Structure):
    _fields_ = [("n_prefill", ctypes.c_longlong), ("n_decode", ctypes.c_longlong), ("ctx_sum", ctypes.c_double)]


class cf_latency_parts(ctypes.Structure):
    _fields_ = [(n, ctypes.c_double) for n in ("t_iter", "t_gemm", "t_attn", "t_prefill", "t_decode")]


class cf_dispatch_state(ctypes.Structure):
    _fields_ = [("n_ranks", ctypes.c_int), ("n_decode", ctypes.POINTER(ctypes.c_longlong)),
                ("ctx_sum", ctypes.POINTER(ctypes.c_double)), ("n_prefill", ctypes.POINTER(ctypes.c_longlong)),
                ("n_chunks", ctypes.c_int), ("chunk_len", ctypes.POINTER(ctypes.c_longlong)),
                ("chunk_ctx", ctypes.POINTER(ctypes.c_longlong))]


class cf_dispatch_result(ctypes.Structure):
    _fields_ = [("n_target", ctypes.c_longlong), ("budget", ctypes.c_longlong), ("chunk", ctypes.c_longlong),
                ("feasible", ctypes.c_int), ("t_iter", ctypes.c_double)]


_lib: Optional[ctypes.CDLL] = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libcf.so (fails loudly if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise FileNotFoundError(f"{path} not built: run python -m co_prefill_decode_gb300.build")
    lib = ctypes.CDLL(path)
    P, I, L, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_float
    sig = {
        "cf_device_sm_count": (I, []),
        "cf_create": (I, [ctypes.POINTER(cf_config), ctypes.POINTER(cf_weights), ctypes.POINTER(P)]),
        "cf_destroy": (None, [P]),
        "cf_layer_step": (I, [P, ctypes.POINTER(cf_batch), P, P, ctypes.POINTER(cf_kv_pool), P]),
        "cf_decode_attn": (I, [P, P, L, ctypes.POINTER(cf_kv_pool), I, P, P, I, P, L, I, P]),
        "cf_prefill_attn": (I, [P, P, ctypes.POINTER(cf_kv_pool), I, I, P, P, I, P]),
        "cf_prefill_attn_varlen": (I, [P, P, ctypes.POINTER(cf_kv_pool), I, ctypes.POINTER(I), ctypes.POINTER(I),
                                       P, I, P, I, P]),
        "cf_gemm": (I, [P, P, I, P, I, P, I, I, I, I, I, P, P]),
        "cf_kv_append": (I, [P, P, P, I, P, ctypes.POINTER(cf_kv_pool), I, I, I, P]),
        "cf_get_error": (I, [P, ctypes.c_char_p, I]),
        "cf_engine_buffer": (P, [P, ctypes.c_char_p]),
        "cf_engine_decode_sms": (I, [P]),
        "cf_set_decode_sms": (I, [P, I]),
        "cf_set_profiling": (I, [P, I]),
        "cf_get_phase_times": (I, [P, ctypes.POINTER(F), I, ctypes.POINTER(I)]),
        "cf_launch_count": (L, [P]),
        "cf_rmsnorm": (I, [P, P, I, P, P, I, P]),
        "cf_calibrate_decode_sms": (I, [P, ctypes.POINTER(cf_batch), ctypes.POINTER(cf_kv_pool), F, P,
                                        ctypes.POINTER(I)]),
        "cf_calibration_points": (I, [P, ctypes.POINTER(I), ctypes.POINTER(F), I]),
        "cf_decode_attn_noalloc": (I, [I, I, I, I, P, L, ctypes.POINTER(cf_kv_pool), I, P, P, I, P, L, I, P]),
        "cf_qkv": (I, [P, ctypes.POINTER(cf_batch), P, ctypes.POINTER(cf_kv_pool), P, P]),
        "cf_gemm_schedule": (I, [I, I, I, I, I, I, ctypes.POINTER(I), ctypes.POINTER(I), ctypes.POINTER(I),
                                 ctypes.POINTER(I)]),
        "cf_set_split_k": (I, [P, I]),
        "cf_prefill_plan": (I, [I, P, P, I, I, I, I, I, ctypes.POINTER(I), P, P, ctypes.POINTER(I)]),
        "cf_decode_plan": (I, [I, P, I, I, I, ctypes.POINTER(I), ctypes.POINTER(I), ctypes.POINTER(L)]),
        "cf_selftest_timeout": (I, [P, ctypes.c_ulonglong, P]),
        "cf_set_prefill_pairing": (I, [P, I]),
        "cf_set_prefill_split": (I, [P, I]),
        "cf_set_graphs": (I, [P, I]),
        "cf_set_fork_mode": (I, [P, I]),
        "cf_graph_captures": (L, [P]),
        "cf_latency_predict": (I, [ctypes.POINTER(cf_latency_model), I, ctypes.POINTER(cf_rank_load), I,
                                   ctypes.POINTER(L), ctypes.POINTER(L), I, ctypes.POINTER(cf_latency_parts)]),
        "cf_latency_fit_line": (I, [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double), I,
                                    ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]),
        "cf_latency_calibrate": (I, [ctypes.POINTER(cf_latency_model), I] + [ctypes.POINTER(ctypes.c_double)] * 4
                                 + [ctypes.c_double, ctypes.c_double, ctypes.POINTER(ctypes.c_double)]),
        "cf_waterfill_dispatch": (I, [ctypes.POINTER(cf_latency_model), I, ctypes.c_double, L,
                                      ctypes.POINTER(cf_dispatch_state), L, L, ctypes.POINTER(cf_dispatch_result),
                                      ctypes.POINTER(L)]),
        "cf_waterfill_assign": (I, [ctypes.POINTER(L), I, L, L, ctypes.POINTER(L)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libcf takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libcf takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(lib, eng, status: int):
    if status != CF_OK:
        buf = ctypes.create_string_buffer(512)
        if eng:
            lib.cf_get_error(eng, buf, 512)
        raise CfError(status, buf.value.decode(errors="replace"))


def device_sm_count() -> int:
    return int(load_library().cf_device_sm_count())


def cf_gemm_schedule(M: int, N: int, K: int, epilogue: int = CF_EPI_NONE, ctas: int = 152,
                     split_mode: int = 0) -> dict:
    """Work split of a GEMM on `ctas` persistent CTAs (host only)."""
    lib = load_library()
    g, t, d, sp = ctypes.c_int(), ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(lib, None, lib.cf_gemm_schedule(M, N, K, epilogue, ctas, split_mode, ctypes.byref(g),
                                           ctypes.byref(t), ctypes.byref(d), ctypes.byref(sp)))
    return {"grid": g.value, "tiles": t.value, "dp_tiles": d.value, "split": sp.value}


def cf_prefill_plan(chunks, n_q_heads: int, n_kv_heads: int, sms: int = 152, split_mode: int = 0,
                    pairing_mode: int = 0) -> dict:
    """Work plan of one prefill launch over chunks [(len, prefix), ...] (host only)."""
    lib = load_library()
    n = len(chunks)
    lens = (ctypes.c_int * max(n, 1))(*[int(c[0]) for c in chunks])
    prefixes = (ctypes.c_int * max(n, 1))(*[int(c[1]) for c in chunks])
    splits = (ctypes.c_int * max(n, 1))()
    cut = (ctypes.c_int * max(n, 1))()
    kind, items = ctypes.c_int(), ctypes.c_int()
    _check(lib, None, lib.cf_prefill_plan(n, ctypes.cast(lens, ctypes.c_void_p), ctypes.cast(prefixes, ctypes.c_void_p),
                                          n_q_heads, n_kv_heads, sms, split_mode, pairing_mode, ctypes.byref(kind),
                                          ctypes.cast(splits, ctypes.c_void_p), ctypes.cast(cut, ctypes.c_void_p),
                                          ctypes.byref(items)))
    return {"kind": kind.value, "splits": list(splits)[:n], "cut_from": list(cut)[:n], "items": items.value}


def cf_decode_plan(n_keys, page_stride: int, n_kv_heads: int, plan_ctas: int = 152) -> dict:
    """Work plan of one decode launch over requests with n_keys keys each (host only)."""
    lib = load_library()
    n = len(n_keys)
    keys = (ctypes.c_int * max(n, 1))(*[int(k) for k in n_keys])
    chunk, items, mx = ctypes.c_int(), ctypes.c_int(), ctypes.c_longlong()
    _check(lib, None, lib.cf_decode_plan(n, ctypes.cast(keys, ctypes.c_void_p), page_stride, n_kv_heads, plan_ctas,
                                         ctypes.byref(chunk), ctypes.byref(items), ctypes.byref(mx)))
    return {"chunk": chunk.value, "items": items.value, "max_items": mx.value}


def make_config(shape, max_tokens: int, max_decode: int, decode_sms: int = 0, page_size: int = 16) -> cf_config:
    return cf_config(shape.hidden, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, shape.ffn_dim, page_size,
                     float(shape.rope_theta), float(shape.rms_eps), int(shape.qk_norm), max_tokens, max_decode,
                     decode_sms)


class Engine:
    """Owns a cf_engine and keeps the weight tensors alive."""

    def __init__(self, cfg: cf_config, weights: Dict[str, torch.Tensor]):
        self.lib = load_library()
        self.cfg = cfg
        self._w = dict(weights)
        w = cf_weights(*[_ptr(self._w.get(n)) for n in
                         ("w_qkv", "w_o", "w_gate", "w_up", "w_down", "g_attn", "g_ffn", "g_q", "g_k")])
        h = ctypes.c_void_p()
        st = self.lib.cf_create(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(h))
        if st != CF_OK:
            raise CfError(st, "cf_create")
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            self.lib.cf_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- C ABI wrappers (same names as the C entry points) ---------------------
    def cf_layer_step(self, batch: cf_batch, x_in: torch.Tensor, x_out: torch.Tensor, pool: cf_kv_pool,
                      stream=None):
        _check(self.lib, self.handle, self.lib.cf_layer_step(self.handle, ctypes.byref(batch), _ptr(x_in),
                                                             _ptr(x_out), ctypes.byref(pool), _stream(stream)))

    def cf_decode_attn(self, q, q_row_stride: int, pool: cf_kv_pool, n: int, n_keys, pages, page_stride: int,
                       out, out_row_stride: int, num_sms: int = 0, stream=None):
        _check(self.lib, self.handle, self.lib.cf_decode_attn(
            self.handle, _ptr(q), q_row_stride, ctypes.byref(pool), n, _ptr(n_keys), _ptr(pages), page_stride,
            _ptr(out), out_row_stride, num_sms, _stream(stream)))

    def cf_prefill_attn(self, q, pool: cf_kv_pool, l: int, prefix: int, pages, out, num_sms: int = 0,
                        stream=None):
        _check(self.lib, self.handle, self.lib.cf_prefill_attn(
            self.handle, _ptr(q), ctypes.byref(pool), l, prefix, _ptr(pages), _ptr(out), num_sms,
            _stream(stream)))

    def cf_prefill_attn_varlen(self, q, pool: cf_kv_pool, chunk_len, chunk_prefix, chunk_pages, out,
                               num_sms: int = 0, stream=None):
        """chunk_len / chunk_prefix: host int sequences; chunk_pages: device
        int32 [n_chunks, stride]."""
        n = len(chunk_len)
        ln = (ctypes.c_int * max(n, 1))(*[int(v) for v in chunk_len])
        pf = (ctypes.c_int * max(n, 1))(*[int(v) for v in chunk_prefix])
        _check(self.lib, self.handle, self.lib.cf_prefill_attn_varlen(
            self.handle, _ptr(q), ctypes.byref(pool), n, ln, pf, _ptr(chunk_pages), int(chunk_pages.shape[1]),
            _ptr(out), num_sms, _stream(stream)))

    def cf_gemm(self, A, B, C, epilogue: int = CF_EPI_NONE, aux=None, stream=None):
        M, K = A.shape
        N = C.shape[1]
        _check(self.lib, self.handle, self.lib.cf_gemm(
            self.handle, _ptr(A), A.stride(0), _ptr(B), B.stride(0), _ptr(C), C.stride(0), M, N, K, epilogue,
            _ptr(aux), _stream(stream)))

    def cf_kv_append(self, k, v, slots, pool: cf_kv_pool, stream=None):
        n, hkv, d = k.shape
        _check(self.lib, self.handle, self.lib.cf_kv_append(
            self.handle, _ptr(k), _ptr(v), n, _ptr(slots), ctypes.byref(pool), hkv, d, self.cfg.page_size,
            _stream(stream)))

    def cf_rmsnorm(self, x, gain, out, stream=None):
        _check(self.lib, self.handle, self.lib.cf_rmsnorm(
            self.handle, _ptr(x), int(x.dtype == torch.float32), _ptr(gain), _ptr(out), x.shape[0],
            _stream(stream)))

    def cf_qkv(self, batch: cf_batch, xn, pool: cf_kv_pool, q_out, stream=None):
        _check(self.lib, self.handle, self.lib.cf_qkv(self.handle, ctypes.byref(batch), _ptr(xn),
                                                      ctypes.byref(pool), _ptr(q_out), _stream(stream)))

    def cf_calibrate_decode_sms(self, batch: cf_batch, pool: cf_kv_pool, frac: float = 0.9, stream=None) -> int:
        out = ctypes.c_int()
        _check(self.lib, self.handle, self.lib.cf_calibrate_decode_sms(
            self.handle, ctypes.byref(batch), ctypes.byref(pool), frac, _stream(stream), ctypes.byref(out)))
        return out.value

    def cf_calibration_points(self):
        n = self.lib.cf_calibration_points(self.handle, None, None, 0)
        sms = (ctypes.c_int * max(n, 1))()
        ms = (ctypes.c_float * max(n, 1))()
        self.lib.cf_calibration_points(self.handle, sms, ms, n)
        return [(sms[i], ms[i]) for i in range(n)]

    def cf_get_error(self):
        buf = ctypes.create_string_buffer(512)
        st = self.lib.cf_get_error(self.handle, buf, 512)
        return st, buf.value.decode(errors="replace")

    def cf_engine_buffer(self, name: str) -> int:
        return int(self.lib.cf_engine_buffer(self.handle, name.encode()) or 0)

    def cf_engine_decode_sms(self) -> int:
        return int(self.lib.cf_engine_decode_sms(self.handle))

    def cf_set_decode_sms(self, n: int):
        _check(self.lib, self.handle, self.lib.cf_set_decode_sms(self.handle, n))

    def cf_set_graphs(self, on: bool):
        _check(self.lib, self.handle, self.lib.cf_set_graphs(self.handle, int(on)))

    def cf_set_fork_mode(self, mode: int):
        """0: concurrent work-conserving attention fork; 1: serial (decode, then prefill, each on all SMs)."""
        _check(self.lib, self.handle, self.lib.cf_set_fork_mode(self.handle, int(mode)))

    def cf_graph_captures(self) -> int:
        return int(self.lib.cf_graph_captures(self.handle))

    def cf_set_prefill_pairing(self, mode: int):
        """0: automatic, 1: single query tiles, 2: tile pairs, 3: head pairs (even GQA groups)."""
        _check(self.lib, self.handle, self.lib.cf_set_prefill_pairing(self.handle, int(mode)))

    def cf_set_prefill_split(self, mode: int):
        _check(self.lib, self.handle, self.lib.cf_set_prefill_split(self.handle, int(mode)))

    def cf_selftest_timeout(self, wait_ns: int, stream=None):
        _check(self.lib, self.handle, self.lib.cf_selftest_timeout(self.handle, int(wait_ns), _stream(stream)))

    def cf_set_split_k(self, mode: int):
        """0: automatic, 1: whole tiles only (batch-invariant rows), n >= 2: n k-chunks."""
        _check(self.lib, self.handle, self.lib.cf_set_split_k(self.handle, int(mode)))

    def cf_set_profiling(self, on: bool):
        _check(self.lib, self.handle, self.lib.cf_set_profiling(self.handle, int(on)))

    def cf_get_phase_times(self):
        ms = (ctypes.c_float * len(PHASES))()
        steps = ctypes.c_int()
        _check(self.lib, self.handle, self.lib.cf_get_phase_times(self.handle, ms, len(PHASES), ctypes.byref(steps)))
        return dict(zip(PHASES, list(ms))), steps.value

    def cf_launch_count(self) -> int:
        return int(self.lib.cf_launch_count(self.handle))

    # -- views of workspace tensors (read-only use in tests) ---------------------
    def buffer(self, name: str, rows: int) -> torch.Tensor:
        """A zero-copy torch view of a workspace tensor of the last step."""
        c = self.cfg
        width = {"xn": c.hidden, "q": c.n_q_heads * c.head_dim, "attn": c.n_q_heads * c.head_dim,
                 "h": c.hidden, "hn": c.hidden, "act": c.ffn_dim}[name]
        ptr = self.cf_engine_buffer(name)
        if not ptr:
            raise CfError(CF_ERR_INVALID_ARG, f"no buffer {name}")
        if name == "h":
            return torch.as_tensor(_DeviceArray(ptr, (rows, width), "<f4"), device="cuda")
        return torch.as_tensor(_DeviceArray(ptr, (rows, width), "<i2"), device="cuda").view(torch.bfloat16)


class _DeviceArray:
    """__cuda_array_interface__ wrapper of a raw device pointer."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"data": (int(ptr), False), "shape": tuple(shape),
                                         "typestr": typestr, "version": 3, "strides": None}


def cf_decode_attn_noalloc(n_q_heads: int, n_kv_heads: int, head_dim: int, page_size: int, q,
                           q_row_stride: int, pool: cf_kv_pool, n: int, n_keys, pages, page_stride: int, out,
                           out_row_stride: int, num_sms: int = 0, stream=None):
    """Decode attention with no engine and no allocation (scratch lives in a
    fixed array inside the library); see include/cf.h."""
    lib = load_library()
    st = lib.cf_decode_attn_noalloc(n_q_heads, n_kv_heads, head_dim, page_size, _ptr(q), q_row_stride,
                                    ctypes.byref(pool), n, _ptr(n_keys), _ptr(pages), page_stride, _ptr(out),
                                    out_row_stride, num_sms, _stream(stream))
    if st != CF_OK:
        raise CfError(st, "cf_decode_attn_noalloc")


def pool_of(k_pool: torch.Tensor, v_pool: torch.Tensor) -> cf_kv_pool:
    return cf_kv_pool(_ptr(k_pool), _ptr(v_pool), int(k_pool.shape[0]))


def batch_of(n_decode: int, dec_ctx, dec_pages, prefill_len: int, prefill_prefix: int, pre_pages,
             chunks=None) -> cf_batch:
    """The batch of one step.  One prefill chunk: prefill_len / prefill_prefix /
    pre_pages.  Several: chunks = (lengths, prefixes, device int32 page table
    [n_chunks, stride]) with prefill_len 0."""
    stride = int(dec_pages.shape[1]) if dec_pages is not None and dec_pages.dim() == 2 else 1
    b = cf_batch(n_decode, _ptr(dec_ctx) if n_decode else None, _ptr(dec_pages) if n_decode else None, stride,
                 prefill_len, prefill_prefix, _ptr(pre_pages) if prefill_len else None)
    if chunks is not None:
        lens, prefixes, pages = chunks
        n = len(lens)
        b._chunk_arrays = ((ctypes.c_int * max(n, 1))(*[int(v) for v in lens]),
                           (ctypes.c_int * max(n, 1))(*[int(v) for v in prefixes]), pages)
        b.n_chunks = n
        b.chunk_len = b._chunk_arrays[0]
        b.chunk_prefix = b._chunk_arrays[1]
        b.chunk_pages = _ptr(pages)
        b.chunk_stride = int(pages.shape[1])
    return b


# ---------------------------------------------------------------------------
# Iteration-latency estimator (host code in libcf; no GPU needed)
# ---------------------------------------------------------------------------
def _doubles(v):
    v = [float(x) for x in v]
    return (ctypes.c_double * max(len(v), 1))(*v), len(v)


def cf_latency_predict(model: cf_latency_model, ranks, chunks=(), n_layers: int = 1) -> Dict[str, float]:
    """ranks: [(n_prefill, n_decode, ctx_sum)] per rank; chunks: [(l_i, c_i)].
    Returns t_iter, t_gemm, t_attn, t_prefill, t_decode."""
    lib = load_library()
    rk = (cf_rank_load * max(len(ranks), 1))(*[cf_rank_load(int(a), int(b), float(c)) for a, b, c in ranks])
    cl = (ctypes.c_longlong * max(len(chunks), 1))(*[int(l) for l, _ in chunks])
    cc = (ctypes.c_longlong * max(len(chunks), 1))(*[int(c) for _, c in chunks])
    out = cf_latency_parts()
    _check(lib, None, lib.cf_latency_predict(ctypes.byref(model), len(ranks), rk, len(chunks), cl, cc,
                                             int(n_layers), ctypes.byref(out)))
    return {n: getattr(out, n) for n, _ in cf_latency_parts._fields_}


def cf_latency_fit_line(x, y):
    """Least-squares (slope, intercept) of y on x."""
    lib = load_library()
    xa, n = _doubles(x)
    ya, m = _doubles(y)
    if n != m:
        raise ValueError("x and y differ in length")
    slope, icpt = ctypes.c_double(), ctypes.c_double()
    _check(lib, None, lib.cf_latency_fit_line(xa, ya, n, ctypes.byref(slope), ctypes.byref(icpt)))
    return slope.value, icpt.value


def cf_latency_calibrate(model: cf_latency_model, t_gemm, t_prefill, t_decode, t_meas,
                         f_max: float = 3.0, step: float = 0.01) -> float:
    """Sets model.alpha / model.beta from co-batched profiles; returns the MAPE (%)."""
    lib = load_library()
    arrs = [_doubles(v) for v in (t_gemm, t_prefill, t_decode, t_meas)]
    n = arrs[0][1]
    if any(a[1] != n for a in arrs):
        raise ValueError("profiles differ in length")
    err = ctypes.c_double()
    _check(lib, None, lib.cf_latency_calibrate(ctypes.byref(model), n, *[a[0] for a in arrs], float(f_max),
                                               float(step), ctypes.byref(err)))
    return err.value


def _longs(v):
    v = [int(x) for x in v]
    return (ctypes.c_longlong * max(len(v), 1))(*v)


def cf_waterfill_dispatch(model: cf_latency_model, n_layers: int, tbt_slo: float, quantum: int, n_decode,
                          ctx_sum, n_prefill, chunks=(), request=None) -> Dict[str, object]:
    """Algorithm 2 over len(n_decode) ranks.  chunks: scheduled [(l_j, c_j)];
    request: (m_i, c_i) or None (budget only).  Returns n_target, budget,
    chunk, feasible, t_iter and assign (A_i per rank)."""
    lib = load_library()
    n = len(n_decode)
    if len(ctx_sum) != n or len(n_prefill) != n:
        raise ValueError("per-rank lists differ in length")
    nd, cs, npf = _longs(n_decode), _doubles(ctx_sum)[0], _longs(n_prefill)
    cl, cc = _longs([l for l, _ in chunks]), _longs([c for _, c in chunks])
    st = cf_dispatch_state(n, nd, cs, npf, len(chunks), cl, cc)
    out = cf_dispatch_result()
    give = (ctypes.c_longlong * max(n, 1))()
    m_i, c_i = (-1, 0) if request is None else (int(request[0]), int(request[1]))
    _check(lib, None, lib.cf_waterfill_dispatch(ctypes.byref(model), int(n_layers), float(tbt_slo), int(quantum),
                                                ctypes.byref(st), m_i, c_i, ctypes.byref(out), give))
    res = {n_: getattr(out, n_) for n_, _ in cf_dispatch_result._fields_}
    res["feasible"] = bool(res["feasible"])
    res["assign"] = [int(give[r]) for r in range(n)]
    return res


def cf_waterfill_assign(loads, tokens: int, n_target: int):
    """WaterfillAssign alone: tokens per rank."""
    lib = load_library()
    n = len(loads)
    give = (ctypes.c_longlong * max(n, 1))()
    _check(lib, None, lib.cf_waterfill_assign(_longs(loads), n, int(tokens), int(n_target), give))
    return [int(give[r]) for r in range(n)]
