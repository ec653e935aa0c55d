"""CPU oracle for the exact ternary weight apply (numpy wrappers over oracle.c).

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product package
never imports it and shares no code with it; both take their inputs from the
seeded generators in ``workloads.py``.

Each wrapper calls the plain C definition in ``oracle.c``; the citation of the
passage each one follows is on the C function. Pins that tie these functions to
what the pages and the mathematics fix are in ``tests/test_oracle_pins.py``.
"""

from __future__ import annotations

import ctypes as C

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(_build.build())
        i64, p = C.c_int64, C.c_void_p
        sigs = {
            "oracle_gemv_i8": [i64, i64, i64, p, p, p, p],
            "oracle_gemv_i8_masked": [i64, i64, i64, p, p, p, p],
            "oracle_gemv_i8_stateset": [i64, i64, i64, p, p, p, p],
            "oracle_gemv_i8_frac": [i64, i64, i64, p, p, p, C.c_int, p],
            "oracle_gemv_q1": [i64, i64, i64, p, p, p, C.c_int, p],
            "oracle_gemv_x64": [i64, i64, i64, p, p, p, C.c_int, p],
            "oracle_lns8_purelns": [i64, i64, p, p, p, C.c_int, p, p, p],
            "oracle_lns_tables": [C.c_int, p, p, p],
            "oracle_lns8_direct": [i64, i64, p, p, p, p],
            "oracle_lns8_histogram": [i64, i64, p, p, p, p],
            "oracle_lns8_tile64": [i64, i64, p, p, p, p],
            "oracle_lns8_stateset": [i64, i64, p, p, p, p],
            "oracle_lns8_materialise": [i64, p, p, p],
            "oracle_lns8_materialise_hi": [i64, p, p, p],
            "oracle_lns8_decode_fp64": [i64, i64, p, p, p, p, p],
            "oracle_lmhead_logits": [i64, i64, p, p, p, p],
            "oracle_topk": [i64, p, i64, p, p],
            "oracle_lmhead_two_stage": [i64, i64, p, p, p, i64, p, p, p, p, p],
            "oracle_planes_of_weight": [C.c_int32, p],
        }
        for name, args in sigs.items():
            fn = getattr(_lib, name)
            fn.argtypes = args
            fn.restype = C.c_int
        _lib.oracle_argmax.argtypes = [i64, p]
        _lib.oracle_argmax.restype = i64
        _lib.oracle_lns8_F.argtypes = [p]
        _lib.oracle_lns8_F.restype = None
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(C.c_void_p)


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"{name}: invalid argument")


# ----------------------------------------------------------------------------
# Ternary GEMV
# ----------------------------------------------------------------------------

def _gemv(fn_name, t, d, x):
    t, pt = _c(t, np.int8)
    d, pd = _c(d, np.int32)
    x = np.atleast_2d(x)
    x, px = _c(x, np.int8)
    N, K = t.shape
    M = x.shape[0]
    if x.shape[1] != K or d.shape != (N, K // 128):
        raise ValueError("shape mismatch")
    y = np.zeros((M, N), dtype=np.int64)
    _check(getattr(lib(), fn_name)(M, N, K, pt, pd, px, y.ctypes.data_as(C.c_void_p)), fn_name)
    return y


def gemv_i8(t, d, x):
    """y[m][r] = sum_g d[r,g] * sum_{i in g} t[r,i] x[m,i]  -> int64 [M][N]."""
    return _gemv("oracle_gemv_i8", t, d, x)


def gemv_i8_frac(t, d, x, frac):
    """y[m][r] = sum_g arshift(d[r,g] * sum_{i in g} t[r,i] x[m,i], frac) -> int64 [M][N]
    (integer engine §4.2 with the per-group floor)."""
    t, pt = _c(t, np.int8)
    d, pd = _c(d, np.int32)
    x = np.atleast_2d(x)
    x, px = _c(x, np.int8)
    N, K = t.shape
    M = x.shape[0]
    if x.shape[1] != K or d.shape != (N, K // 128):
        raise ValueError("shape mismatch")
    y = np.zeros((M, N), dtype=np.int64)
    _check(lib().oracle_gemv_i8_frac(M, N, K, pt, pd, px, int(frac), y.ctypes.data_as(C.c_void_p)),
           "oracle_gemv_i8_frac")
    return y


def gemv_x64(t, d, x, frac=0):
    """int64 fixed-point activations (integer engine §4.4, exact modulo 2^64 as
    its §5 states): y[m][r] = sum_g arshift(d[r,g] * sum_{i in g} t[r,i] x[m,i],
    frac) with every sum and product wrapping modulo 2^64. t in {-1,0,1}."""
    t, pt = _c(t, np.int8)
    d, pd = _c(d, np.int32)
    x = np.atleast_2d(x)
    x, px = _c(x, np.int64)
    N, K = t.shape
    M = x.shape[0]
    if x.shape[1] != K or d.shape != (N, K // 128):
        raise ValueError("shape mismatch")
    y = np.zeros((M, N), dtype=np.int64)
    _check(lib().oracle_gemv_x64(M, N, K, pt, pd, px, int(frac), y.ctypes.data_as(C.c_void_p)),
           "oracle_gemv_x64")
    return y


def gemv_q1(bits, d, x, frac=0):
    """Q1_0 (integer engine §4.1): bits [N][K] in {0,1} for sign -1/+1;
    y[m][r] = sum_g arshift((2 pos_sum - block_total) * d[r,g], frac)."""
    b, pb = _c(bits, np.uint8)
    d, pd = _c(d, np.int32)
    x = np.atleast_2d(x)
    x, px = _c(x, np.int8)
    N, K = b.shape
    M = x.shape[0]
    if x.shape[1] != K or d.shape != (N, K // 128):
        raise ValueError("shape mismatch")
    y = np.zeros((M, N), dtype=np.int64)
    _check(lib().oracle_gemv_q1(M, N, K, pb, pd, px, int(frac), y.ctypes.data_as(C.c_void_p)),
           "oracle_gemv_q1")
    return y


def gemv_i8_masked(t, d, x):
    return _gemv("oracle_gemv_i8_masked", t, d, x)


def gemv_i8_stateset(t, d, x):
    return _gemv("oracle_gemv_i8_stateset", t, d, x)


# ----------------------------------------------------------------------------
# LNS8 eight-phase path
# ----------------------------------------------------------------------------

def _lns8(fn_name, t, dcode, xa):
    t, pt = _c(t, np.int8)
    dcode, pd = _c(dcode, np.uint8)
    xa, px = _c(xa, np.uint8)
    N, K = t.shape
    if xa.shape != (K,) or dcode.shape != (N, K // 128):
        raise ValueError("shape mismatch")
    A = np.zeros((N, 8), dtype=np.int64)
    _check(getattr(lib(), fn_name)(N, K, pt, pd, px, A.ctypes.data_as(C.c_void_p)), fn_name)
    return A


def lns8_direct(t, dcode, xa):
    """A[r][p] by direct eight-phase accumulation -> int64 [N][8]."""
    return _lns8("oracle_lns8_direct", t, dcode, xa)


def lns_tables(F):
    """(LOG8[0..128], KP[len], KM[len]) of the pure fractional-LNS reduction (BitState brief §5.2)."""
    lib().oracle_lns_table_len.argtypes = [C.c_int]
    lib().oracle_lns_table_len.restype = C.c_int64
    n = int(lib().oracle_lns_table_len(int(F)))
    if n < 0:
        raise ValueError("F must be 1..6")
    log8 = np.zeros(129, np.int64)
    kp = np.zeros(n, np.int64)
    km = np.zeros(n, np.int64)
    _check(lib().oracle_lns_tables(int(F), log8.ctypes.data_as(C.c_void_p), kp.ctypes.data_as(C.c_void_p),
                                   km.ctypes.data_as(C.c_void_p)), "oracle_lns_tables")
    return log8, kp, km


def lns8_purelns(t, dcode, xa, F):
    """Pure fractional-LNS reduction of the LNS8 product states (BitState brief
    §5.2, this library's reading; see oracle.c): (sign int64 [N], lam int64 [N]
    = log magnitude * 2^F in code units, S fp64 [N])."""
    t, pt = _c(t, np.int8)
    dcode, pd = _c(dcode, np.uint8)
    xa, px = _c(xa, np.uint8)
    N, K = t.shape
    if xa.shape != (K,) or dcode.shape != (N, K // 128):
        raise ValueError("shape mismatch")
    sign = np.zeros(N, np.int64)
    lam = np.zeros(N, np.int64)
    S = np.zeros(N, np.float64)
    _check(lib().oracle_lns8_purelns(N, K, pt, pd, px, int(F), sign.ctypes.data_as(C.c_void_p),
                                     lam.ctypes.data_as(C.c_void_p), S.ctypes.data_as(C.c_void_p)),
           "oracle_lns8_purelns")
    return sign, lam, S


def lns8_histogram(t, dcode, xa):
    return _lns8("oracle_lns8_histogram", t, dcode, xa)


def lns8_tile64(t, dcode, xa):
    return _lns8("oracle_lns8_tile64", t, dcode, xa)


def lns8_stateset(t, dcode, xa):
    return _lns8("oracle_lns8_stateset", t, dcode, xa)


def lns8_F():
    """F[p] = 2^((p-2)/8) as fp64 (libm exp2)."""
    F = np.zeros(8, dtype=np.float64)
    lib().oracle_lns8_F(F.ctypes.data_as(C.c_void_p))
    return F


def lns8_materialise(A, F=None):
    """S[r] = 2^-9 * sum_p A[r,p] F[p], fixed order, no FP contraction."""
    A, pa = _c(A, np.int64)
    F = lns8_F() if F is None else np.ascontiguousarray(F, dtype=np.float64)
    S = np.zeros(A.shape[0], dtype=np.float64)
    _check(lib().oracle_lns8_materialise(A.shape[0], pa, F.ctypes.data_as(C.c_void_p),
                                         S.ctypes.data_as(C.c_void_p)), "materialise")
    return S


def lns8_materialise_hi(A):
    """(S computed in long double, 2^-9 sum_p |A[p]| F[p]) both rounded to fp64."""
    A, pa = _c(A, np.int64)
    S = np.zeros(A.shape[0], dtype=np.float64)
    mag = np.zeros(A.shape[0], dtype=np.float64)
    _check(lib().oracle_lns8_materialise_hi(A.shape[0], pa, S.ctypes.data_as(C.c_void_p),
                                            mag.ctypes.data_as(C.c_void_p)), "materialise_hi")
    return S, mag


def lns8_decode_fp64(t, dcode, xa):
    """(sum of sign * 2^((k-74)/8) per row in fp64, sum of magnitudes)."""
    t, pt = _c(t, np.int8)
    dcode, pd = _c(dcode, np.uint8)
    xa, px = _c(xa, np.uint8)
    N, K = t.shape
    S = np.zeros(N, dtype=np.float64)
    mag = np.zeros(N, dtype=np.float64)
    _check(lib().oracle_lns8_decode_fp64(N, K, pt, pd, px, S.ctypes.data_as(C.c_void_p),
                                         mag.ctypes.data_as(C.c_void_p)), "decode_fp64")
    return S, mag


# ----------------------------------------------------------------------------
# lm_head over 8 base-3 planes
# ----------------------------------------------------------------------------

def lmhead_logits(planes, s, x):
    """logit[r] = s[r] * sum_i (sum_p planes[p,r,i] 3^(7-p)) x[i]  -> int64 [N]."""
    planes, pp = _c(planes, np.int8)
    s, ps = _c(s, np.int32)
    x, px = _c(x, np.int8)
    _, N, K = planes.shape
    out = np.zeros(N, dtype=np.int64)
    _check(lib().oracle_lmhead_logits(N, K, pp, ps, px, out.ctypes.data_as(C.c_void_p)), "logits")
    return out


def argmax(scores):
    scores, p = _c(scores, np.int64)
    return int(lib().oracle_argmax(scores.shape[0], p))


def topk(scores, k):
    """(ids int32[k], scores int64[k]) under (score desc, index asc)."""
    scores, p = _c(scores, np.int64)
    ids = np.zeros(k, dtype=np.int32)
    top = np.zeros(k, dtype=np.int64)
    _check(lib().oracle_topk(scores.shape[0], p, k, ids.ctypes.data_as(C.c_void_p),
                             top.ctypes.data_as(C.c_void_p)), "topk")
    return ids, top


def lmhead_two_stage(planes, s, x, k):
    """Two-stage exact top-k: (ids, scores, lo, hi, n_candidates)."""
    planes, pp = _c(planes, np.int8)
    s, ps = _c(s, np.int32)
    x, px = _c(x, np.int8)
    _, N, K = planes.shape
    ids = np.zeros(k, dtype=np.int32)
    top = np.zeros(k, dtype=np.int64)
    lo = np.zeros(N, dtype=np.int64)
    hi = np.zeros(N, dtype=np.int64)
    nc = np.zeros(1, dtype=np.int64)
    _check(lib().oracle_lmhead_two_stage(
        N, K, pp, ps, px, k, ids.ctypes.data_as(C.c_void_p), top.ctypes.data_as(C.c_void_p),
        lo.ctypes.data_as(C.c_void_p), hi.ctypes.data_as(C.c_void_p),
        nc.ctypes.data_as(C.c_void_p)), "two_stage")
    return ids, top, lo, hi, int(nc[0])


def planes_of_weight(w):
    """Balanced-ternary digits (plane 0 first) of an integer weight in [-3280, 3280]."""
    digits = np.zeros(8, dtype=np.int8)
    _check(lib().oracle_planes_of_weight(int(w), digits.ctypes.data_as(C.c_void_p)), "planes_of_weight")
    return digits
