"""ctypes binding of liboscar.so: the names and arguments of include/oscar.h.

Argument marshalling only: every step of the serving path runs in the CUDA
library. Tensors are passed by device pointer; the CUDA stream is torch's
current stream unless one is given. If the library is missing, loading fails
loudly (there is no fallback).
"""

from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "liboscar.so")
HEADER = os.path.join(ROOT, "include", "oscar.h")

OK = 0
STATUS = {
    0: "OK", -1: "INVALID_ARG", -2: "NOT_LOADED", -3: "OUT_OF_RANGE", -4: "CUDA",
    -5: "UNSUPPORTED", -6: "NOT_BOUND",
}
FLAG_BAD_PAGE_ID = 1
FLAG_BAD_STATE = 2
FLAG_TIMEOUT = 4
PAGE_BLOCK_BYTES = 1536  # group size 32


def page_block_bytes(group_size: int = 32) -> int:
    """Bytes of one (page, KV head) block of the INT2 pool (include/oscar.h)."""
    return 1024 + 128 * (128 // group_size)


class OscarError(RuntimeError):
    def __init__(self, status, msg=""):
        super().__init__("oscar status %d (%s)%s" % (status, STATUS.get(status, "?"),
                                                     ": " + msg if msg else ""))
        self.status = status


class OscarConfig(ctypes.Structure):
    _fields_ = [
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("group_size", ctypes.c_int32),
        ("sink", ctypes.c_int32),
        ("recent", ctypes.c_int32),
        ("max_batch", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("fold_rv", ctypes.c_int32),
        ("num_splits", ctypes.c_int32),
    ]


class SeqState(ctypes.Structure):
    _fields_ = [("seq_len", ctypes.c_int32), ("int2_end", ctypes.c_int32),
                ("window_row", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_P = ctypes.c_void_p
_SIGS = {
    "oscar_version": (ctypes.c_int, []),
    "oscar_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "oscar_check_config": (ctypes.c_int, [ctypes.POINTER(OscarConfig)]),
    "oscar_cache_bytes": (ctypes.c_int, [ctypes.POINTER(OscarConfig), ctypes.c_int64,
                                         ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_size_t)]),
    "oscar_create": (ctypes.c_int, [ctypes.POINTER(OscarConfig), ctypes.POINTER(_P)]),
    "oscar_destroy": (None, [_P]),
    "oscar_bind_cache": (ctypes.c_int, [_P, _P, ctypes.c_int64, _P]),
    "oscar_load_rotations": (ctypes.c_int, [_P, _P, _P, _P, _P]),
    "oscar_quant_append": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.c_int32, ctypes.c_int32, _P]),
    "oscar_quant_append_traced": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.c_int32, ctypes.c_int32,
                                                 _P, ctypes.c_int32, _P]),
    "oscar_decode_attn": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.c_int32, _P]),
    "oscar_decode_attn_timed": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.c_int32, _P, _P, _P]),
    "oscar_decode_attn_shared_prefix": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_int32, _P, ctypes.c_int32, _P]),
    "oscar_decode_step": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, ctypes.c_int32, _P]),
    "oscar_decode_step_host": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, ctypes.c_int32, _P]),
    "oscar_calibration_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int32, ctypes.c_int32]),
    "oscar_calibration_covariances": (ctypes.c_int, [_P, _P, _P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                     ctypes.c_float, _P, _P, _P, ctypes.c_size_t, _P]),
    "oscar_quant_append_timed": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.c_int32, ctypes.c_int32, _P,
                                                _P, _P]),
    "oscar_decode_splits": (ctypes.c_int, [_P, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]),
    "oscar_error_flags": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int32]),
    "oscar_last_error": (ctypes.c_char_p, [_P]),
    "oscar_decode_attn_noalloc": (ctypes.c_int, [ctypes.POINTER(OscarConfig), _P, _P, _P, _P, ctypes.c_int32,
                                                 _P, ctypes.c_int64, _P, _P, _P, _P, _P, _P]),
}

_lib = None


def header_functions():
    """Names of the functions declared in include/oscar.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(oscar_\w+)\s*\(", text, re.M)))


def lib():
    """The loaded liboscar.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OscarError(-4, "liboscar.so is not built; run `python -m bit_rotated_kv_oscar_gb300.build` "
                                 "(or __graft_entry__.build())")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(status, ctx=None):
    if status != OK:
        msg = ""
        if ctx is not None:
            msg = (lib().oscar_last_error(ctx) or b"").decode()
        raise OscarError(status, msg)


def make_config(num_q_heads, num_kv_heads, sink, recent, max_batch, max_pages_per_seq,
                softmax_scale=0.0, fold_rv=0, num_splits=0, head_dim=128, page_size=16,
                group_size=32) -> OscarConfig:
    return OscarConfig(num_q_heads, num_kv_heads, head_dim, page_size, group_size, sink, recent,
                       max_batch, max_pages_per_seq, softmax_scale, fold_rv, num_splits)


def check_config(cfg: OscarConfig) -> int:
    return lib().oscar_check_config(ctypes.byref(cfg))


def calibration_covariances(q, k, v, softmax_scale: float = 0.0, stream=None):
    """C_Q, C_S (device float32 [Hkv, 128, 128]) of calibration activations q
    [N, Hq, 128], k, v [N, Hkv, 128] (device bf16), computed by the library."""
    import torch

    n, hq, _ = q.shape
    hkv = k.shape[1]
    c_q = torch.empty(hkv, 128, 128, dtype=torch.float32, device=q.device)
    c_s = torch.empty_like(c_q)
    nbytes = lib().oscar_calibration_workspace_bytes(n, hq)
    ws = torch.empty(max(nbytes, 4) // 4, dtype=torch.float32, device=q.device)
    _check(lib().oscar_calibration_covariances(_ptr(q), _ptr(k), _ptr(v), n, hq, hkv, softmax_scale, _ptr(c_q),
                                               _ptr(c_s), _ptr(ws), nbytes, _stream(stream)))
    return c_q, c_s


def cache_bytes(cfg: OscarConfig, num_pages: int):
    pb, wb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().oscar_cache_bytes(ctypes.byref(cfg), num_pages, ctypes.byref(pb), ctypes.byref(wb)))
    return pb.value, wb.value


def _ptr(t):
    """Device pointer of a tensor; the library reads dense row-major buffers only."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("liboscar takes contiguous tensors (got strides %s)" % (tuple(t.stride()),))
    return ctypes.c_void_p(t.data_ptr())


def _event(ev):
    """Raw cudaEvent_t of a torch.cuda.Event (recorded once so that it exists)."""
    if ev is None:
        return None
    if not ev.cuda_event:
        ev.record()
    return ctypes.c_void_p(ev.cuda_event)


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


NOALLOC_SCRATCH_BYTES = 32 << 20


def decode_attn_noalloc(cfg, q, page_table, state, o, batch, pool, num_pages, window, r_k, r_v, clip_v,
                        err_flags=None, stream=None):
    """oscar_decode_attn_noalloc: decode attention without a context and without any
    device allocation (device tensors in, device output out)."""
    _check(lib().oscar_decode_attn_noalloc(ctypes.byref(cfg), _ptr(q), _ptr(page_table), _ptr(state),
                                           _ptr(o), batch, _ptr(pool), num_pages, _ptr(window),
                                           _ptr(r_k), _ptr(r_v), _ptr(clip_v), _ptr(err_flags),
                                           _stream(stream)))


class Context:
    """One oscar_ctx: a layer's rotations, its bound cache and workspace."""

    def __init__(self, cfg: OscarConfig):
        self.cfg = cfg
        h = ctypes.c_void_p()
        _check(lib().oscar_create(ctypes.byref(cfg), ctypes.byref(h)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            lib().oscar_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def bind_cache(self, pool, num_pages, window):
        _check(lib().oscar_bind_cache(self.handle, _ptr(pool), num_pages, _ptr(window)), self.handle)

    def load_rotations(self, r_k, r_v, clip_k, clip_v):
        """Host float32 numpy arrays [Hkv,128,128] and [Hkv]."""
        import numpy as np
        arrs = [np.ascontiguousarray(a, dtype=np.float32) for a in (r_k, r_v, clip_k, clip_v)]
        ptrs = [a.ctypes.data_as(ctypes.c_void_p) for a in arrs]
        _check(lib().oscar_load_rotations(self.handle, *ptrs), self.handle)

    def quant_append(self, page_table, state, k, v, batch, n_new, stream=None):
        _check(lib().oscar_quant_append(self.handle, _ptr(page_table), _ptr(state), _ptr(k), _ptr(v),
                                        batch, n_new, _stream(stream)), self.handle)

    def quant_append_traced(self, page_table, state, k, v, batch, n_new, trace, trace_positions,
                            stream=None):
        _check(lib().oscar_quant_append_traced(self.handle, _ptr(page_table), _ptr(state), _ptr(k),
                                               _ptr(v), batch, n_new, _ptr(trace), trace_positions,
                                               _stream(stream)), self.handle)

    def decode_attn_timed(self, q, page_table, state, o, batch, ev_before, ev_after, stream=None):
        """decode_attn that records torch.cuda.Event ev_before / ev_after around its
        split-K attention kernel (for measurement)."""
        _check(lib().oscar_decode_attn_timed(self.handle, _ptr(q), _ptr(page_table), _ptr(state), _ptr(o),
                                             batch, _stream(stream), _event(ev_before), _event(ev_after)),
               self.handle)

    def quant_append_timed(self, page_table, state, k, v, batch, n_new, ev_before, ev_after, stream=None):
        """quant_append that records torch.cuda.Event ev_before / ev_after around its
        main kernel (the tensor-core kernel of a long append)."""
        _check(lib().oscar_quant_append_timed(self.handle, _ptr(page_table), _ptr(state), _ptr(k), _ptr(v),
                                              batch, n_new, _stream(stream), _event(ev_before),
                                              _event(ev_after)), self.handle)

    def decode_attn(self, q, page_table, state, o, batch, stream=None):
        _check(lib().oscar_decode_attn(self.handle, _ptr(q), _ptr(page_table), _ptr(state), _ptr(o),
                                       batch, _stream(stream)), self.handle)

    def decode_attn_shared_prefix(self, q, page_table, state, prefix_tokens, o, batch, stream=None):
        """decode_attn for requests whose first prefix_tokens positions map to the
        same pages: the shared range is read once per pack of requests."""
        _check(lib().oscar_decode_attn_shared_prefix(self.handle, _ptr(q), _ptr(page_table), _ptr(state),
                                                     prefix_tokens, _ptr(o), batch, _stream(stream)), self.handle)

    def decode_step(self, page_table, state, q, k, v, o, batch, stream=None):
        """oscar_decode_step: one new token per request (k, v [batch][Hkv][128])
        appended and one decode query (q) over the cache that then holds it, in the
        decode call's launches."""
        _check(lib().oscar_decode_step(self.handle, _ptr(page_table), _ptr(state), _ptr(q), _ptr(k), _ptr(v),
                                       _ptr(o), batch, _stream(stream)), self.handle)

    def decode_step_host(self, page_table, state, h_qkv, d_qkv, o, h_o, batch, stream=None):
        """oscar_decode_step_host: one new token per request and one decode query,
        inputs from host memory h_qkv (bf16 q, k, v back to back) through the device
        staging buffer d_qkv, output o (device) copied to host memory h_o."""
        _check(lib().oscar_decode_step_host(self.handle, _ptr(page_table), _ptr(state), _ptr(h_qkv), _ptr(d_qkv),
                                            _ptr(o), _ptr(h_o), batch, _stream(stream)), self.handle)

    def decode_splits(self, batch):
        s = ctypes.c_int32()
        _check(lib().oscar_decode_splits(self.handle, batch, ctypes.byref(s)), self.handle)
        return s.value

    def error_flags(self, clear=True):
        f = ctypes.c_uint32()
        _check(lib().oscar_error_flags(self.handle, ctypes.byref(f), 1 if clear else 0), self.handle)
        return f.value

    def last_error(self):
        return (lib().oscar_last_error(self.handle) or b"").decode()
