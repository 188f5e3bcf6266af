"""CPU oracle for the grouped-expert MoE FFN layer (ctypes binding of moe_oracle.cpp).

TEST INFRASTRUCTURE ONLY: imported by tests, the smoke check and the benchmark's
CPU-baseline leg, never by the library. Inputs are numpy arrays or CPU torch tensors;
outputs are numpy arrays. See moe_oracle.cpp for the definition it computes.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from .build import build

_lib = None


class _Layer(C.Structure):
    _fields_ = [("E", C.c_int), ("k", C.c_int), ("H", C.c_int), ("I", C.c_int), ("Is", C.c_int),
                ("w_gate", C.c_void_p), ("w_up", C.c_void_p), ("w_down", C.c_void_p),
                ("s_gate", C.c_void_p), ("s_up", C.c_void_p), ("s_down", C.c_void_p),
                ("sh_gate", C.c_void_p), ("sh_up", C.c_void_p), ("sh_down", C.c_void_p),
                ("sh_s_gate", C.c_void_p), ("sh_s_up", C.c_void_p), ("sh_s_down", C.c_void_p)]


class _LayerNvfp4(C.Structure):
    _fields_ = [("E", C.c_int), ("k", C.c_int), ("H", C.c_int), ("I", C.c_int), ("Is", C.c_int),
                ("w_gate", C.c_void_p), ("w_up", C.c_void_p), ("w_down", C.c_void_p),
                ("b_gate", C.c_void_p), ("b_up", C.c_void_p), ("b_down", C.c_void_p),
                ("g_gate", C.c_void_p), ("g_up", C.c_void_p), ("g_down", C.c_void_p),
                ("sh_gate", C.c_void_p), ("sh_up", C.c_void_p), ("sh_down", C.c_void_p),
                ("sh_b_gate", C.c_void_p), ("sh_b_up", C.c_void_p), ("sh_b_down", C.c_void_p),
                ("sh_g", C.c_void_p)]


class _Taps(C.Structure):
    _fields_ = [("qx", C.c_void_p), ("sx", C.c_void_p), ("acc_gu", C.c_void_p),
                ("hq", C.c_void_p), ("sh", C.c_void_p), ("acc_d", C.c_void_p)]


def lib():
    """The oracle's shared library: built from moe_oracle.cpp, or the build named by the
    environment variable MOE_ORACLE_LIB (the mutation test loads deliberately broken copies
    that way)."""
    global _lib
    if _lib is None:
        _lib = C.CDLL(os.environ.get("MOE_ORACLE_LIB") or build())
        for name in ("oracle_route", "oracle_quant_rows", "oracle_permute", "oracle_forward",
                     "oracle_dense", "oracle_router_logits", "oracle_rmsnorm_residual",
                     "oracle_forward_nvfp4"):
            getattr(_lib, name).restype = C.c_int
        for name in ("oracle_e2m1_value", "oracle_e4m3_value"):
            getattr(_lib, name).restype = C.c_double
            getattr(_lib, name).argtypes = [C.c_int]
    return _lib


def _np(a, dtype):
    """Contiguous numpy copy/view of a numpy array or CPU torch tensor."""
    if hasattr(a, "detach"):
        import torch
        a = a.detach().cpu()
        if a.dtype == torch.bfloat16:
            a = a.view(torch.int16)
        a = a.numpy()
    return np.ascontiguousarray(a).view(dtype) if np.dtype(dtype).itemsize == a.dtype.itemsize \
        else np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return a.ctypes.data_as(C.c_void_p) if a is not None else None


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count())


def route(logits, k: int):
    lg = _np(logits, np.float32)
    T, E = lg.shape
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    rc = lib().oracle_route(_p(lg), T, E, k, _p(idx), _p(w))
    if rc:
        raise ValueError(f"oracle_route rc={rc}")
    return idx, w


def quant_rows(x_bf16):
    x = _np(x_bf16, np.uint16)
    T, H = x.shape
    q = np.zeros((T, H), np.int8)
    s = np.zeros((T,), np.float32)
    lib().oracle_quant_rows(_p(x), T, H, _p(q), _p(s))
    return q, s


def permute(idx, E: int):
    ix = _np(idx, np.int32)
    T, k = ix.shape
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(T * k, np.int32)
    rc = lib().oracle_permute(_p(ix), T, k, E, _p(counts), _p(offsets), _p(perm))
    if rc:
        raise ValueError(f"oracle_permute rc={rc}")
    return counts, offsets, perm


class Layer:
    """Host copies of one layer's quantised weights, held for the oracle calls."""

    def __init__(self, W: dict, E: int, k: int, H: int, I: int, Is: int):
        self.E, self.k, self.H, self.I, self.Is = E, k, H, I, Is
        self.arrs = {}
        for key in ("w_gate", "w_up", "w_down"):
            self.arrs[key] = _np(W[key], np.int8)
        for key in ("s_gate", "s_up", "s_down"):
            self.arrs[key] = _np(W[key], np.float32)
        if Is > 0:
            for key in ("sh_gate", "sh_up", "sh_down"):
                self.arrs[key] = _np(W[key], np.int8)
            for key in ("sh_s_gate", "sh_s_up", "sh_s_down"):
                self.arrs[key] = _np(W[key], np.float32)
        self.c = _Layer(E, k, H, I, Is, *[_p(self.arrs.get(f)) for f, _ in _Layer._fields_[5:]])


def forward(layer: Layer, x_bf16, idx, w, taps: bool = False, nthreads: int | None = None):
    """Whole layer. Returns y (float64 [T,H]) and, with taps=True, a dict of intermediates
    indexed by (token, slot); slot k is the shared expert."""
    x = _np(x_bf16, np.uint16)
    ix = _np(idx, np.int32)
    ww = _np(w, np.float32)
    T, H = x.shape
    k = layer.k
    S = k + (1 if layer.Is > 0 else 0)
    Imax = max(layer.I, layer.Is)
    y = np.zeros((T, H), np.float64)
    t = None
    tp = None
    if taps:
        t = dict(qx=np.zeros((T, H), np.int8), sx=np.zeros(T, np.float32),
                 acc_gu=np.zeros((T, S, 2, Imax), np.int32), hq=np.zeros((T, S, Imax), np.int8),
                 sh=np.zeros((T, S), np.float32), acc_d=np.zeros((T, S, H), np.int32))
        tp = _Taps(*[_p(t[f]) for f, _ in _Taps._fields_])
    n = nthreads or default_threads()
    rc = lib().oracle_forward(C.byref(layer.c), _p(x), T, _p(ix), _p(ww), _p(y),
                              C.byref(tp) if tp is not None else None, n)
    if rc:
        raise ValueError(f"oracle_forward rc={rc}")
    return (y, t) if taps else y


def dense(layer: Layer, x_bf16, idx, w, nthreads: int | None = None):
    x = _np(x_bf16, np.uint16)
    ix = _np(idx, np.int32)
    ww = _np(w, np.float32)
    T, H = x.shape
    y = np.zeros((T, H), np.float64)
    rc = lib().oracle_dense(C.byref(layer.c), _p(x), T, _p(ix), _p(ww), _p(y),
                            nthreads or default_threads())
    if rc:
        raise ValueError(f"oracle_dense rc={rc}")
    return y


def router_logits(x_bf16, w_router, nthreads: int | None = None):
    x = _np(x_bf16, np.uint16)
    wr = _np(w_router, np.float32)
    T, H = x.shape
    E = wr.shape[1]
    out = np.zeros((T, E), np.float64)
    lib().oracle_router_logits(_p(x), _p(wr), T, H, E, _p(out), nthreads or default_threads())
    return out


def rmsnorm_residual(x_bf16, y=None):
    """Stacked-prefill layer input. Returns (x after the residual update, x_in) as uint16
    bf16 bit arrays; y (float64/float32 [T,H]) may be None."""
    x = _np(x_bf16, np.uint16).copy()
    T, H = x.shape
    yy = None if y is None else np.ascontiguousarray(np.asarray(y, np.float64))
    x_in = np.zeros_like(x)
    lib().oracle_rmsnorm_residual(_p(x), _p(yy), _p(x_in), T, H)
    return x, x_in


def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(int(code))


def e4m3_value(byte: int) -> float:
    return lib().oracle_e4m3_value(int(byte))


class LayerNvfp4:
    """Host copies of one layer's NVFP4 expert weights (see synth.make_weights_nvfp4)."""

    def __init__(self, W: dict, E: int, k: int, H: int, I: int, Is: int):
        self.E, self.k, self.H, self.I, self.Is = E, k, H, I, Is
        self.arrs = {}
        for key in ("w_gate", "w_up", "w_down", "b_gate", "b_up", "b_down"):
            self.arrs[key] = _np(W[key], np.uint8)
        for key in ("g_gate", "g_up", "g_down"):
            self.arrs[key] = _np(W[key], np.float32)
        if Is > 0:
            for key in ("sh_gate", "sh_up", "sh_down", "sh_b_gate", "sh_b_up", "sh_b_down"):
                self.arrs[key] = _np(W[key], np.uint8)
            self.arrs["sh_g"] = _np(W["sh_g"], np.float32)
        self.c = _LayerNvfp4(E, k, H, I, Is,
                             *[_p(self.arrs.get(f)) for f, _ in _LayerNvfp4._fields_[5:]])


def forward_nvfp4(layer: LayerNvfp4, x_bf16, idx, w, taps: bool = False,
                  nthreads: int | None = None):
    """The layer with NVFP4 expert weights. Returns y (float64 [T,H]) and, with taps=True,
    the intermediates; acc_gu and acc_d are the exact sums of q * e2m1 * e4m3 (float64)."""
    x = _np(x_bf16, np.uint16)
    ix = _np(idx, np.int32)
    ww = _np(w, np.float32)
    T, H = x.shape
    k = layer.k
    S = k + (1 if layer.Is > 0 else 0)
    Imax = max(layer.I, layer.Is)
    y = np.zeros((T, H), np.float64)
    t = None
    tp = None
    if taps:
        t = dict(qx=np.zeros((T, H), np.int8), sx=np.zeros(T, np.float32),
                 acc_gu=np.zeros((T, S, 2, Imax), np.float64), hq=np.zeros((T, S, Imax), np.int8),
                 sh=np.zeros((T, S), np.float32), acc_d=np.zeros((T, S, H), np.float64))
        tp = _Taps(*[_p(t[f]) for f, _ in _Taps._fields_])
    rc = lib().oracle_forward_nvfp4(C.byref(layer.c), _p(x), T, _p(ix), _p(ww), _p(y),
                                    C.byref(tp) if tp is not None else None,
                                    nthreads or default_threads())
    if rc:
        raise ValueError(f"oracle_forward_nvfp4 rc={rc}")
    return (y, t) if taps else y
