"""Python binding of libtg.so: an exact ternary weight apply for one GB300 GPU.

Argument marshalling only. Every function here has the name of the C entry
point it calls (include/tg.h) and does nothing but convert arguments: numpy
arrays for the host packer, device pointers (torch CUDA tensors, or plain
integers) and a CUDA stream for the compute calls. All computation runs in the
library's CUDA kernels; there is no CPU fallback. If libtg.so is missing the
import of this module still works, but every call raises.
"""

from __future__ import annotations

import ctypes as C
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtg.so")

TG_OK = 0
TG_ERR_ARG = -1
TG_ERR_SHAPE = -2
TG_ERR_VALUE = -3
TG_ERR_BOUND = -4
TG_ERR_WORKSPACE = -5
TG_ERR_CUDA = -6
TG_ERR_DEVICE = -7

TG_TERNARY_I8 = 1
TG_TERNARY_LNS8 = 2
TG_PLANES8 = 3
TG_BINARY_Q1 = 4

TG_GROUP = 128
TG_MAX_M = 64
TG_MAX_K = 1024
TG_NOALLOC_SCRATCH_BYTES = 4 * 1024 * 1024
TG_FLAG_CONST_WEIGHTS = 1
TG_FLAG_LNS8_STATE_SET = 2
TG_FLAG_X_INT64 = 4
TG_FLAG_LNS8_PURE_LNS = 8

# Every symbol include/tg.h declares.
EXPORTS = (
    "tg_status_string",
    "tg_layout_init",
    "tg_packed_bytes",
    "tg_pack_weights",
    "tg_gemv_i8",
    "tg_gemv_lns8_phase",
    "tg_lmhead_workspace_bytes",
    "tg_lmhead_argmax_topk",
    "tg_lmhead_argmax_topk_noalloc",
    "tg_device_error",
)


class tg_layout(C.Structure):
    _fields_ = [
        ("kind", C.c_int32), ("version", C.c_int32),
        ("N", C.c_int64), ("K", C.c_int64), ("G", C.c_int64), ("tiles", C.c_int64),
        ("mask_off", C.c_int64), ("mask_bytes", C.c_int64),
        ("scale_off", C.c_int64), ("scale_bytes", C.c_int64),
        ("aux_off", C.c_int64), ("aux_bytes", C.c_int64),
        ("aux2_off", C.c_int64), ("aux2_bytes", C.c_int64),
        ("total_bytes", C.c_int64), ("max_abs_scale", C.c_int64),
        ("flags", C.c_int64),
        ("frac", C.c_int64),
        ("wait_limit", C.c_int64),
        ("reserved", C.c_int64 * 1),
    ]


class TgError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {tg_status_string(status)} ({status})")


_lib = None


def lib():
    """The loaded libtg.so. Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libtg.so is not built ({LIB_PATH}); run bit_decode_gemv_gb300.build.build()")
        L = C.CDLL(LIB_PATH)
        p, i64, i32, sz = C.c_void_p, C.c_int64, C.c_int32, C.c_size_t
        lp = C.POINTER(tg_layout)
        L.tg_status_string.argtypes = [C.c_int]
        L.tg_status_string.restype = C.c_char_p
        L.tg_layout_init.argtypes = [C.c_int, i64, i64, lp]
        L.tg_packed_bytes.argtypes = [C.c_int, i64, i64]
        L.tg_packed_bytes.restype = sz
        L.tg_pack_weights.argtypes = [C.c_int, i64, i64, p, p, p, sz, lp]
        L.tg_gemv_i8.argtypes = [lp, p, p, i64, p, p]
        L.tg_gemv_lns8_phase.argtypes = [lp, p, p, p, p, p, p]
        L.tg_lmhead_workspace_bytes.argtypes = [lp, i32]
        L.tg_lmhead_workspace_bytes.restype = sz
        L.tg_lmhead_argmax_topk.argtypes = [lp, p, p, i32, p, p, p, p, p, p, sz, p]
        L.tg_lmhead_argmax_topk_noalloc.argtypes = [lp, p, p, i32, p, p, p, p, p, p]
        L.tg_device_error.argtypes = [p, C.POINTER(i32)]
        for name in ("tg_layout_init", "tg_pack_weights", "tg_gemv_i8", "tg_gemv_lns8_phase",
                     "tg_lmhead_argmax_topk", "tg_lmhead_argmax_topk_noalloc", "tg_device_error"):
            getattr(L, name).restype = C.c_int
        _lib = L
    return _lib


def _check(status: int, where: str):
    if status != TG_OK:
        raise TgError(status, where)


def _ptr(t):
    """Device (or host) address of a torch tensor, an int, or None."""
    if t is None:
        return None
    if type(t) is int:
        return t
    try:
        return t.data_ptr()   # (the common case first: this runs once per argument of every call)
    except AttributeError:
        if isinstance(t, int):
            return int(t)
        raise TypeError(f"expected a tensor or an address, got {type(t).__name__}") from None


def _stream(stream):
    """cudaStream_t handle: a torch.cuda.Stream, a raw int, or None (torch's current stream)."""
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def tg_status_string(status: int) -> str:
    return lib().tg_status_string(int(status)).decode()


def tg_layout_init(kind: int, N: int, K: int) -> tg_layout:
    L = tg_layout()
    _check(lib().tg_layout_init(kind, N, K, C.byref(L)), "tg_layout_init")
    return L


def tg_packed_bytes(kind: int, N: int, K: int) -> int:
    return int(lib().tg_packed_bytes(kind, N, K))


def tg_pack_weights(kind: int, trits: np.ndarray, scales: np.ndarray):
    """Pack host weights; returns (uint8 host blob, tg_layout).

    trits: int8 [N][K] (ternary kinds; -1/+1 for TG_BINARY_Q1) or [8][N][K] (TG_PLANES8).
    scales: int32 [N][K/128] (TG_TERNARY_I8, TG_BINARY_Q1), uint8 [N][K/128] (TG_TERNARY_LNS8),
    int32 [N] (TG_PLANES8).
    """
    trits = np.ascontiguousarray(trits, dtype=np.int8)
    sdt = np.uint8 if kind == TG_TERNARY_LNS8 else np.int32
    scales = np.ascontiguousarray(scales, dtype=sdt)
    if kind == TG_PLANES8:
        if trits.ndim != 3 or trits.shape[0] != 8:
            raise ValueError("planes must be [8][N][K]")
        N, K = trits.shape[1], trits.shape[2]
    else:
        if trits.ndim != 2:
            raise ValueError("trits must be [N][K]")
        N, K = trits.shape
    nbytes = tg_packed_bytes(kind, N, K)
    if nbytes == 0:
        raise TgError(TG_ERR_SHAPE, "tg_packed_bytes")
    need = N if kind == TG_PLANES8 else N * (K // TG_GROUP)
    if scales.size != need:
        raise TgError(TG_ERR_SHAPE, "tg_pack_weights: scales size")
    out = np.empty(nbytes, dtype=np.uint8)
    L = tg_layout()
    _check(lib().tg_pack_weights(kind, N, K, trits.ctypes.data_as(C.c_void_p),
                                 scales.ctypes.data_as(C.c_void_p), out.ctypes.data_as(C.c_void_p),
                                 nbytes, C.byref(L)), "tg_pack_weights")
    return out, L


_FAST_UNSET = object()
_fast_mod = _FAST_UNSET


def _fast():
    """The compiled call path to tg_gemv_i8 (csrc/tgpy.c), or None if it was not built."""
    global _fast_mod
    if _fast_mod is _FAST_UNSET:
        lib()   # the same libtg.so, loaded first
        try:
            from . import _tgpy
            _fast_mod = _tgpy
        except ImportError:
            _fast_mod = None
    return _fast_mod


def tg_gemv_i8(layout: tg_layout, w, x, M: int, y, stream=None) -> None:
    f = _fast_mod if _fast_mod is not _FAST_UNSET else _fast()
    if f is not None:
        st = f.gemv_i8(C.addressof(layout), _ptr(w) or 0, _ptr(x) or 0, int(M), _ptr(y) or 0, _stream(stream) or 0)
    else:
        st = lib().tg_gemv_i8(C.byref(layout), _ptr(w), _ptr(x), int(M), _ptr(y), _stream(stream))
    _check(st, "tg_gemv_i8")


def tg_gemv_lns8_phase(layout: tg_layout, w, xa, A, S=None, stream=None, F=None) -> None:
    """F: device fp64 [8] phase constants, or None for the built-in 2^((p-2)/8)
    (the C argument between xa and A)."""
    _check(lib().tg_gemv_lns8_phase(C.byref(layout), _ptr(w), _ptr(xa), _ptr(F), _ptr(A), _ptr(S),
                                    _stream(stream)), "tg_gemv_lns8_phase")


def tg_lmhead_workspace_bytes(layout: tg_layout, k: int) -> int:
    return int(lib().tg_lmhead_workspace_bytes(C.byref(layout), int(k)))


def tg_lmhead_argmax_topk(layout: tg_layout, w, x, k: int, logits, argmax, ids, scores, ncand,
                          ws, ws_bytes: int, stream=None) -> None:
    _check(lib().tg_lmhead_argmax_topk(C.byref(layout), _ptr(w), _ptr(x), int(k), _ptr(logits),
                                       _ptr(argmax), _ptr(ids), _ptr(scores), _ptr(ncand), _ptr(ws),
                                       int(ws_bytes), _stream(stream)), "tg_lmhead_argmax_topk")


def tg_lmhead_argmax_topk_noalloc(layout: tg_layout, w, x, k: int, logits, argmax, ids, scores,
                                  ncand, stream=None) -> None:
    """tg_lmhead_argmax_topk on the library's own fixed scratch, for callers that
    cannot allocate device memory (see include/tg.h for the limit and the sharing rules)."""
    _check(lib().tg_lmhead_argmax_topk_noalloc(C.byref(layout), _ptr(w), _ptr(x), int(k),
                                               _ptr(logits), _ptr(argmax), _ptr(ids), _ptr(scores),
                                               _ptr(ncand), _stream(stream)),
           "tg_lmhead_argmax_topk_noalloc")


def tg_device_error(stream=None) -> int:
    code = C.c_int32(0)
    _check(lib().tg_device_error(_stream(stream), C.byref(code)), "tg_device_error")
    return int(code.value)
