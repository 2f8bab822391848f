"""Python binding of the h3attn C ABI (``include/h3attn.h``), via ctypes.

Argument marshalling only: every function here converts Python arguments
(torch tensors, nested span lists, streams) into the plain pointers and sizes
of the C call of the same name, calls it, and raises ``H3AttnError`` on a
non-OK status.  All computation happens in the library's CUDA kernels; there
is no fallback.  If the library is missing, loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_double, c_float, c_int32, c_int64, c_uint64, c_void_p

import numpy as np

from . import build as _build

H3ATTN_OK, H3ATTN_EINVAL, H3ATTN_EUNSUPPORTED, H3ATTN_ENOMEM, H3ATTN_ECUDA, H3ATTN_ETIMEOUT = range(6)
STATUS_NAMES = ["OK", "EINVAL", "EUNSUPPORTED", "ENOMEM", "ECUDA", "ETIMEOUT"]


class H3AttnError(RuntimeError):
    def __init__(self, status: int, fn: str, msg: str):
        self.status = status
        name = STATUS_NAMES[status] if 0 <= status < len(STATUS_NAMES) else str(status)
        super().__init__(f"{fn}: H3ATTN_{name}: {msg}")


class h3attn_span(ctypes.Structure):
    _fields_ = [("n_t", c_int32), ("n_h", c_int32), ("n_w", c_int32),
                ("start", c_double * 3), ("step", c_double * 3)]


class h3attn_doc(ctypes.Structure):
    _fields_ = [("spans", POINTER(h3attn_span)), ("n_spans", c_int32)]


class h3attn_plan_opts(ctypes.Structure):
    _fields_ = [("num_heads", c_int32), ("head_dim", c_int32), ("rope_dims", c_int32),
                ("rope_base", c_double)]


_SIGS = {
    "h3attn_plan_create": [POINTER(h3attn_doc), c_int32, POINTER(h3attn_plan_opts), c_void_p,
                           POINTER(c_void_p)],
    "h3attn_plan_destroy": [c_void_p],
    "h3attn_plan_info": [c_void_p, POINTER(c_int64), POINTER(c_int32), POINTER(c_int32),
                         POINTER(c_int32)],
    "h3attn_plan_copy_cu_seqlens": [c_void_p, c_void_p],
    "h3attn_plan_copy_positions": [c_void_p, c_void_p],
    "h3attn_plan_copy_rope_table": [c_void_p, c_void_p],
    "h3attn_qk_prologue": [c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_void_p, c_int64,
                           c_void_p, c_void_p, c_int64, c_float, c_void_p],
    "h3attn_forward": [c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_int64,
                       c_float, c_void_p, c_void_p],
    "h3attn_forward_fused_q": [c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_int64,
                               c_void_p, c_int64, c_float, c_float, c_void_p, c_void_p],
    "h3attn_fp8_quantize": [c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_void_p, c_void_p,
                            c_void_p, c_void_p, c_void_p, c_void_p],
    "h3attn_plan_fp8_v_keys": [c_void_p, POINTER(c_int64)],
    "h3attn_plan_forward_kernels": [c_void_p, POINTER(c_int32)],
    "h3attn_qk_prologue_fp8": [c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_void_p, c_int64,
                               c_float, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p],
    "h3attn_work_list_host": [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_int64, c_void_p,
                              POINTER(c_int64), POINTER(c_int32)],
    "h3attn_forward_fp8": [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                           c_int64, c_float, c_void_p, c_void_p],
    "h3attn_forward_noalloc": [c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_int64,
                               c_void_p, c_int64, c_float, c_void_p, c_void_p],
    "h3attn_get_device_error": [c_void_p, c_void_p],
    "h3attn_selftest_bounded_wait": [c_uint64, c_void_p],
}

_lib = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Loads libh3attn.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with packed_varlen_non_gb300.build.build()")
        lib = ctypes.CDLL(path)
        for name, args in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = c_int32
        lib.h3attn_last_error.argtypes = []
        lib.h3attn_last_error.restype = c_char_p
        _lib = lib
    return _lib


def h3attn_last_error() -> str:
    return load().h3attn_last_error().decode()


def _check(status: int, fn: str):
    if status != H3ATTN_OK:
        raise H3AttnError(status, fn, h3attn_last_error())


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _row_stride(t, given):
    if given is not None:
        return int(given)
    if isinstance(t, int):
        raise ValueError("a row stride is required when passing raw pointers")
    return int(t.stride(0))


# ------------------------------------------------------------------ plan ----

def h3attn_plan_create(docs, num_heads: int, rope_base: float = 10000.0, head_dim: int = 128,
                       rope_dims: int = 96, stream=None) -> int:
    """docs: list of documents, each a list of spans (n_t, n_h, n_w, start3, step3).
    Returns the opaque plan handle (an int)."""
    span_arrays = []
    cdocs = (h3attn_doc * max(1, len(docs)))()
    for i, d in enumerate(docs):
        arr = (h3attn_span * max(1, len(d)))()
        for j, (n_t, n_h, n_w, start, step) in enumerate(d):
            arr[j].n_t, arr[j].n_h, arr[j].n_w = int(n_t), int(n_h), int(n_w)
            for a in range(3):
                arr[j].start[a] = float(start[a])
                arr[j].step[a] = float(step[a])
        span_arrays.append(arr)
        cdocs[i].spans = ctypes.cast(arr, POINTER(h3attn_span))
        cdocs[i].n_spans = len(d)
    opts = h3attn_plan_opts(int(num_heads), int(head_dim), int(rope_dims), float(rope_base))
    out = c_void_p()
    st = _stream(stream) if stream is not False else None
    _check(load().h3attn_plan_create(cdocs, len(docs), ctypes.byref(opts), st, ctypes.byref(out)),
           "h3attn_plan_create")
    return out.value


def h3attn_plan_destroy(plan):
    _check(load().h3attn_plan_destroy(plan), "h3attn_plan_destroy")


def h3attn_plan_info(plan) -> dict:
    S, nd, ml, nh = c_int64(), c_int32(), c_int32(), c_int32()
    _check(load().h3attn_plan_info(plan, ctypes.byref(S), ctypes.byref(nd), ctypes.byref(ml),
                                   ctypes.byref(nh)), "h3attn_plan_info")
    return {"S": S.value, "n_docs": nd.value, "max_seqlen": ml.value, "num_heads": nh.value}


def h3attn_plan_copy_cu_seqlens(plan) -> np.ndarray:
    info = h3attn_plan_info(plan)
    out = np.zeros(info["n_docs"] + 1, dtype=np.int32)
    _check(load().h3attn_plan_copy_cu_seqlens(plan, out.ctypes.data), "h3attn_plan_copy_cu_seqlens")
    return out


def h3attn_plan_copy_positions(plan) -> np.ndarray:
    info = h3attn_plan_info(plan)
    out = np.zeros((info["S"], 3), dtype=np.float64)
    _check(load().h3attn_plan_copy_positions(plan, out.ctypes.data), "h3attn_plan_copy_positions")
    return out


def h3attn_plan_copy_rope_table(plan) -> np.ndarray:
    info = h3attn_plan_info(plan)
    out = np.zeros((info["S"], 48, 2), dtype=np.float32)
    _check(load().h3attn_plan_copy_rope_table(plan, out.ctypes.data), "h3attn_plan_copy_rope_table")
    return out


# --------------------------------------------------------------- compute ----

def h3attn_qk_prologue(plan, q_in, k_in, q_out, k_out, gain_q, gain_k, eps: float = 1e-6,
                       in_row_stride=None, out_row_stride=None, gain_head_stride: int = 0,
                       stream=None):
    """Tensors: bf16 [S, H, 128]-shaped views (row stride taken from dim 0)
    or raw device pointers with explicit strides; gains fp32 on the device.
    q_in = q_out = None processes k only (for h3attn_forward_fused_q)."""
    for pair in ((q_in, k_in, in_row_stride), (q_out, k_out, out_row_stride)):
        if (pair[2] is None and pair[0] is not None and not isinstance(pair[0], int)
                and pair[0].stride(0) != pair[1].stride(0)):
            raise ValueError("q and k must share one row stride on each side")
    _check(load().h3attn_qk_prologue(plan, _ptr(q_in), _ptr(k_in), _row_stride(k_in, in_row_stride),
                                     _ptr(q_out), _ptr(k_out), _row_stride(k_out, out_row_stride),
                                     _ptr(gain_q), _ptr(gain_k), int(gain_head_stride), float(eps),
                                     _stream(stream)), "h3attn_qk_prologue")


def h3attn_forward(plan, q, k, v, o, softmax_scale: float, lse=None, qkv_row_stride=None,
                   o_row_stride=None, stream=None):
    if qkv_row_stride is None and not isinstance(q, int):
        strides = {int(x.stride(0)) for x in (q, k, v)}
        if len(strides) != 1:
            raise ValueError(f"q, k and v must share one row stride (got {sorted(strides)})")
    _check(load().h3attn_forward(plan, _ptr(q), _ptr(k), _ptr(v), _row_stride(q, qkv_row_stride),
                                 _ptr(o), _row_stride(o, o_row_stride), float(softmax_scale),
                                 _ptr(lse), _stream(stream)), "h3attn_forward")


def h3attn_forward_fused_q(plan, q_raw, k, v, o, gain_q, softmax_scale: float, eps: float = 1e-6,
                           lse=None, qkv_row_stride=None, o_row_stride=None, gain_head_stride: int = 0,
                           stream=None):
    """Forward with the Q prologue fused in: q_raw holds raw queries, k is
    already k-hat (see include/h3attn.h)."""
    if qkv_row_stride is None and not isinstance(q_raw, int):
        strides = {int(x.stride(0)) for x in (q_raw, k, v)}
        if len(strides) != 1:
            raise ValueError(f"q, k and v must share one row stride (got {sorted(strides)})")
    _check(load().h3attn_forward_fused_q(plan, _ptr(q_raw), _ptr(k), _ptr(v), _row_stride(q_raw, qkv_row_stride),
                                         _ptr(o), _row_stride(o, o_row_stride), _ptr(gain_q),
                                         int(gain_head_stride), float(eps), float(softmax_scale), _ptr(lse),
                                         _stream(stream)), "h3attn_forward_fused_q")


def h3attn_fp8_quantize(plan, q_hat, k_hat, v, q8, k8, v8t, sq, sk, sv, qkv_row_stride=None, stream=None):
    """FP8 quantisation of q-hat, k-hat, v (see include/h3attn.h for layouts)."""
    if qkv_row_stride is None and not isinstance(q_hat, int):
        strides = {int(x.stride(0)) for x in (q_hat, k_hat, v)}
        if len(strides) != 1:
            raise ValueError(f"q, k and v must share one row stride (got {sorted(strides)})")
    _check(load().h3attn_fp8_quantize(plan, _ptr(q_hat), _ptr(k_hat), _ptr(v), _row_stride(q_hat, qkv_row_stride),
                                      _ptr(q8), _ptr(k8), _ptr(v8t), _ptr(sq), _ptr(sk), _ptr(sv), _stream(stream)),
           "h3attn_fp8_quantize")


def h3attn_qk_prologue_fp8(plan, q_in, k_in, v, gain_q, gain_k, eps: float, q8, k8, v8t, sq, sk, sv,
                           gain_head_stride: int = 0, qkv_row_stride=None, stream=None):
    """The q/k prologue fused with the FP8 quantisation (see include/h3attn.h)."""
    if qkv_row_stride is None and not isinstance(q_in, int):
        strides = {int(x.stride(0)) for x in (q_in, k_in, v)}
        if len(strides) != 1:
            raise ValueError(f"q, k and v must share one row stride (got {sorted(strides)})")
    _check(load().h3attn_qk_prologue_fp8(plan, _ptr(q_in), _ptr(k_in), _ptr(v), _row_stride(q_in, qkv_row_stride),
                                         _ptr(gain_q), _ptr(gain_k), int(gain_head_stride), float(eps), _ptr(q8),
                                         _ptr(k8), _ptr(v8t), _ptr(sq), _ptr(sk), _ptr(sv), _stream(stream)),
           "h3attn_qk_prologue_fp8")


def h3attn_plan_forward_kernels(plan) -> int:
    n = c_int32()
    _check(load().h3attn_plan_forward_kernels(plan, ctypes.byref(n)), "h3attn_plan_forward_kernels")
    return n.value


def h3attn_work_list_host(cu_seqlens, num_heads: int, n_pairs: int):
    """The forward's work list for a layout, built on the host (no GPU needed).
    Returns (units int32 [n, 8], unit_off int32 [pairs + 1]); the fields of a
    unit are those of the C call."""
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    n_docs = int(cu.size) - 1
    n, used = c_int64(), c_int32()
    lib = load()
    _check(lib.h3attn_work_list_host(cu.ctypes.data, n_docs, int(num_heads), int(n_pairs), None, 0, None,
                                     ctypes.byref(n), ctypes.byref(used)), "h3attn_work_list_host")
    units = np.zeros((n.value, 8), dtype=np.int32)
    off = np.zeros(used.value + 1, dtype=np.int32)
    _check(lib.h3attn_work_list_host(cu.ctypes.data, n_docs, int(num_heads), int(n_pairs), units.ctypes.data,
                                     n.value, off.ctypes.data, ctypes.byref(n), ctypes.byref(used)),
           "h3attn_work_list_host")
    return units, off


def h3attn_plan_fp8_v_keys(plan) -> int:
    n = c_int64()
    _check(load().h3attn_plan_fp8_v_keys(plan, ctypes.byref(n)), "h3attn_plan_fp8_v_keys")
    return n.value


def h3attn_forward_fp8(plan, q8, k8, v8t, sq, sk, sv, o, softmax_scale: float, lse=None, o_row_stride=None,
                       stream=None):
    _check(load().h3attn_forward_fp8(plan, _ptr(q8), _ptr(k8), _ptr(v8t), _ptr(sq), _ptr(sk), _ptr(sv), _ptr(o),
                                     _row_stride(o, o_row_stride), float(softmax_scale), _ptr(lse),
                                     _stream(stream)), "h3attn_forward_fp8")


def h3attn_forward_noalloc(cu_seqlens, num_heads: int, q, k, v, o, softmax_scale: float, lse=None,
                           qkv_row_stride=None, o_row_stride=None, stream=None):
    """The allocation-free forward: cu_seqlens is a host int32 sequence
    [n_docs + 1]; no plan and no device allocation (see include/h3attn.h)."""
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    if qkv_row_stride is None and not isinstance(q, int):
        strides = {int(x.stride(0)) for x in (q, k, v)}
        if len(strides) != 1:
            raise ValueError(f"q, k and v must share one row stride (got {sorted(strides)})")
    _check(load().h3attn_forward_noalloc(cu.ctypes.data, cu.size - 1, int(num_heads), _ptr(q), _ptr(k),
                                         _ptr(v), _row_stride(q, qkv_row_stride), _ptr(o),
                                         _row_stride(o, o_row_stride), float(softmax_scale), _ptr(lse),
                                         _stream(stream)), "h3attn_forward_noalloc")


def h3attn_get_device_error(plan, stream=None):
    _check(load().h3attn_get_device_error(plan, _stream(stream)), "h3attn_get_device_error")


def h3attn_selftest_bounded_wait(timeout_ns: int, stream=None) -> int:
    """Returns the raw status (ETIMEOUT is the expected outcome)."""
    return int(load().h3attn_selftest_bounded_wait(int(timeout_ns), _stream(stream)))


class Plan:
    """Owns a plan handle; a context manager around create/destroy."""

    def __init__(self, docs, num_heads, rope_base=10000.0, stream=None):
        self.handle = h3attn_plan_create(docs, num_heads, rope_base, stream=stream)
        self.info = h3attn_plan_info(self.handle)

    def close(self):
        if self.handle:
            h3attn_plan_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
