"""Python binding of libmoe (include/moe.h): the grouped-expert MoE FFN layer on GB300.

Argument marshalling only: every step of the layer runs in the CUDA kernels of libmoe.so.
The functions keep the C names; tensors are torch CUDA tensors (their data pointers are
passed), streams default to torch's current stream. A nonzero status raises MoeError.
There is no CPU fallback: if libmoe.so has not been built, importing the library raises.
"""
from __future__ import annotations

import ctypes as C
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "moe.h")

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_OOM",
          4: "MOE_ERR_CAPACITY", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_TIMEOUT", 7: "MOE_ERR_DEVICE",
          8: "MOE_ERR_NO_DEVICE"}
MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_OOM = 0, 1, 2, 3
MOE_ERR_CAPACITY, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE, MOE_ERR_NO_DEVICE = 4, 5, 6, 7, 8

TAP_COUNTS, TAP_OFFSETS, TAP_PERM, TAP_QX, TAP_SX, TAP_ACC_GU, TAP_HQ, TAP_SH, TAP_ACC_D = range(9)
TAP_ACC_GU_F64, TAP_ACC_D_F64 = 9, 10  # NVFP4 weights: fp64 accumulators


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} ({status_string(status)})")


class Weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in (
        "w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down",
        "sh_gate", "sh_up", "sh_down", "sh_s_gate", "sh_s_up", "sh_s_down")]


class WeightsNvfp4(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in (
        "w_gate", "w_up", "w_down", "b_gate", "b_up", "b_down", "g_gate", "g_up", "g_down",
        "sh_gate", "sh_up", "sh_down", "sh_b_gate", "sh_b_up", "sh_b_down", "sh_g")]


_lib = None


def lib() -> C.CDLL:
    """The loaded libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libmoe.so not built ({LIB_PATH}); run "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = C.CDLL(LIB_PATH)
        vp, i32, sz = C.c_void_p, C.c_int, C.c_size_t
        sig = {
            "moe_plan": ([i32, i32, i32, i32, i32, i32, C.POINTER(vp)], i32),
            "moe_plan_destroy": ([vp], i32),
            "moe_plan_set_decode_rows": ([vp, i32], i32),
            "moe_pack_weights": ([vp, C.POINTER(Weights), vp, C.POINTER(vp)], i32),
            "moe_pack_weights_nvfp4": ([vp, C.POINTER(WeightsNvfp4), vp, C.POINTER(vp)], i32),
            "moe_packed_destroy": ([vp], i32),
            "moe_route": ([vp, vp, i32, vp, vp, vp], i32),
            "moe_forward": ([vp, vp, vp, i32, vp, vp, vp, vp], i32),
            "moe_route_forward": ([vp, vp, vp, i32, vp, vp, vp, vp, vp], i32),
            "moe_get_error": ([vp], i32),
            "moe_clear_error": ([vp], i32),
            "moe_selftest_wait_timeout": ([vp, vp], i32),
            "moe_status_string": ([i32], C.c_char_p),
            "moe_debug_enable": ([vp, i32], i32),
            "moe_debug_tap_bytes": ([vp, i32], sz),
            "moe_debug_tap": ([vp, i32, vp, sz], i32),
            "moe_profile_enable": ([vp, i32], i32),
            "moe_profile_read": ([vp, i32, C.POINTER(C.c_float), C.POINTER(C.c_int)], i32),
            "moe_router_logits": ([vp, vp, i32, i32, i32, vp, vp], i32),
            "moe_router_pack": ([vp, i32, i32, vp, vp], i32),
            "moe_router_logits_packed": ([vp, vp, i32, i32, i32, vp, vp], i32),
            "moe_residual_add": ([vp, vp, i32, i32, vp], i32),
            "moe_rmsnorm_residual": ([vp, vp, vp, i32, i32, vp], i32),
            "moe_forward_decode_static": ([i32, i32, i32, i32, i32, C.POINTER(Weights), vp, i32,
                                           vp, vp, vp, vp, vp], i32),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def header_symbols() -> list[str]:
    """Entry points declared in include/moe.h."""
    src = open(HEADER).read()
    return re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)


def status_string(s: int) -> str:
    return lib().moe_status_string(s).decode()


def _check(st: int, where: str):
    if st != MOE_OK:
        raise MoeError(st, where)


def _ptr(t):
    """Device address of a tensor argument (None and raw integer addresses pass through).
    The kernels read row-major contiguous device memory, so a strided view or a host tensor
    is refused here instead of being read with the wrong layout or from the wrong memory."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError(f"tensor argument of shape {tuple(t.shape)} is not contiguous")
    if not t.is_cuda:
        raise ValueError(f"tensor argument of shape {tuple(t.shape)} is on {t.device}, not CUDA")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---- C entry points (same names) -----------------------------------------------------

def moe_plan(E: int, top_k: int, H: int, I: int, I_shared: int, max_tokens: int) -> int:
    h = C.c_void_p()
    _check(lib().moe_plan(E, top_k, H, I, I_shared, max_tokens, C.byref(h)), "moe_plan")
    return h.value


def moe_plan_destroy(plan: int):
    _check(lib().moe_plan_destroy(plan), "moe_plan_destroy")


def moe_plan_set_decode_rows(plan: int, rows: int):
    """T <= rows runs the weight-streaming decode kernels, larger T the grouped GEMMs."""
    _check(lib().moe_plan_set_decode_rows(plan, rows), "moe_plan_set_decode_rows")


def make_weights_struct(W: dict) -> Weights:
    return Weights(*[_ptr(W.get(n)) for n, _ in Weights._fields_])


def moe_pack_weights(plan: int, W: dict, stream=None) -> int:
    h = C.c_void_p()
    ws = make_weights_struct(W)
    _check(lib().moe_pack_weights(plan, C.byref(ws), _stream(stream), C.byref(h)),
           "moe_pack_weights")
    return h.value


def moe_pack_weights_nvfp4(plan: int, W: dict, stream=None) -> int:
    """Register NVFP4 expert weights (uint8 codes and E4M3 block scales, fp32 matrix scales;
    the keys of moe_weights_nvfp4). The tensors are read in place: keep them alive."""
    h = C.c_void_p()
    ws = WeightsNvfp4(*[_ptr(W.get(n)) for n, _ in WeightsNvfp4._fields_])
    _check(lib().moe_pack_weights_nvfp4(plan, C.byref(ws), _stream(stream), C.byref(h)),
           "moe_pack_weights_nvfp4")
    return h.value


def moe_packed_destroy(packed: int):
    _check(lib().moe_packed_destroy(packed), "moe_packed_destroy")


def moe_route(plan: int, logits, idx, w, stream=None):
    T = logits.shape[0]
    _check(lib().moe_route(plan, _ptr(logits), T, _ptr(idx), _ptr(w), _stream(stream)),
           "moe_route")


def moe_forward(plan: int, packed: int, x, idx, w, y, stream=None):
    T = x.shape[0]
    _check(lib().moe_forward(plan, packed, _ptr(x), T, _ptr(idx), _ptr(w), _ptr(y),
                             _stream(stream)), "moe_forward")


def moe_route_forward(plan: int, packed: int, x, logits, idx, w, y, stream=None):
    """Routing (written to idx, w) and the layer (y) in one call; the routing runs inside
    the forward's first kernel."""
    T = x.shape[0]
    _check(lib().moe_route_forward(plan, packed, _ptr(x), T, _ptr(logits), _ptr(idx), _ptr(w),
                                   _ptr(y), _stream(stream)), "moe_route_forward")


def moe_get_error(plan: int) -> int:
    return lib().moe_get_error(plan)


def moe_clear_error(plan: int):
    _check(lib().moe_clear_error(plan), "moe_clear_error")


def moe_selftest_wait_timeout(plan: int, stream=None):
    """Queue the bounded-wait self-test: the plan's error word becomes MOE_ERR_TIMEOUT."""
    _check(lib().moe_selftest_wait_timeout(plan, _stream(stream)), "moe_selftest_wait_timeout")


def moe_debug_enable(plan: int, on: bool = True):
    _check(lib().moe_debug_enable(plan, 1 if on else 0), "moe_debug_enable")


def moe_debug_tap(plan: int, which: int):
    """Host copy (numpy) of one intermediate of the last moe_forward."""
    import numpy as np
    n = lib().moe_debug_tap_bytes(plan, which)
    dt = {TAP_QX: np.int8, TAP_HQ: np.int8, TAP_SX: np.float32, TAP_SH: np.float32,
          TAP_ACC_GU_F64: np.float64, TAP_ACC_D_F64: np.float64}.get(which, np.int32)
    out = np.zeros(n // np.dtype(dt).itemsize, dt)
    _check(lib().moe_debug_tap(plan, which, out.ctypes.data, n), "moe_debug_tap")
    return out


def moe_profile_enable(plan: int, on: bool = True):
    _check(lib().moe_profile_enable(plan, 1 if on else 0), "moe_profile_enable")


def moe_profile_read(plan: int, path: int):
    """(per-stage summed device ms over the forwards since the last read, number of calls);
    path 0 = prefill, 1 = decode."""
    ms = (C.c_float * 4)()
    calls = C.c_int()
    _check(lib().moe_profile_read(plan, path, ms, C.byref(calls)), "moe_profile_read")
    return list(ms), calls.value


def moe_router_logits(x, w_router, logits, stream=None):
    T, H = x.shape
    E = w_router.shape[1]
    _check(lib().moe_router_logits(_ptr(x), _ptr(w_router), T, H, E, _ptr(logits),
                                   _stream(stream)), "moe_router_logits")


def moe_router_pack(w_router, packed=None, stream=None):
    """bf16 [3E, H] three-part split of the fp32 router weight [H, E] (blocks of 16 experts,
    each block hi, mid, lo rows) for moe_router_logits_packed."""
    H, E = w_router.shape
    if packed is None:
        packed = torch.empty((3 * E, H), dtype=torch.bfloat16, device=w_router.device)
    _check(lib().moe_router_pack(_ptr(w_router), H, E, _ptr(packed), _stream(stream)),
           "moe_router_pack")
    return packed


def moe_router_logits_packed(x, packed, logits, stream=None):
    T, H = x.shape
    E = packed.shape[0] // 3
    _check(lib().moe_router_logits_packed(_ptr(x), _ptr(packed), T, H, E, _ptr(logits),
                                          _stream(stream)), "moe_router_logits_packed")


def moe_residual_add(x, y, stream=None):
    T, H = x.shape
    _check(lib().moe_residual_add(_ptr(x), _ptr(y), T, H, _stream(stream)), "moe_residual_add")


def moe_rmsnorm_residual(x, y, x_in, stream=None):
    """x <- bf16(x + y) when y is not None, then x_in <- bf16(x / rms(x))."""
    T, H = x.shape
    _check(lib().moe_rmsnorm_residual(_ptr(x), _ptr(y), _ptr(x_in), T, H, _stream(stream)),
           "moe_rmsnorm_residual")


# ---- convenience wrapper ---------------------------------------------------------------

class MoELayer:
    """One plan plus one packed weight set; keeps the caller's weight tensors alive. The
    weight format follows the dict's keys: NVFP4 when it holds block scales (b_gate)."""

    def __init__(self, E, top_k, H, I, I_shared, max_tokens, weights: dict, stream=None):
        self.E, self.k, self.H, self.I, self.Is = E, top_k, H, I, I_shared
        self.plan = moe_plan(E, top_k, H, I, I_shared, max_tokens)
        self.weights = weights
        self.nvfp4 = "b_gate" in weights
        pack = moe_pack_weights_nvfp4 if self.nvfp4 else moe_pack_weights
        self.packed = pack(self.plan, weights, stream)

    def route(self, logits, stream=None):
        T = logits.shape[0]
        idx = torch.empty((T, self.k), dtype=torch.int32, device=logits.device)
        w = torch.empty((T, self.k), dtype=torch.float32, device=logits.device)
        moe_route(self.plan, logits, idx, w, stream)
        return idx, w

    def forward(self, x, idx, w, y=None, stream=None):
        if y is None:
            y = torch.empty((x.shape[0], self.H), dtype=torch.float32, device=x.device)
        moe_forward(self.plan, self.packed, x, idx, w, y, stream)
        return y

    def close(self):
        if self.packed:
            moe_packed_destroy(self.packed)
            self.packed = None
        if self.plan:
            moe_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
