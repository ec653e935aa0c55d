"""Seeded synthetic inputs for the ternary weight apply.

This module only draws random arrays with the shapes and value distributions of
the workloads below. It holds none of the method's arithmetic (no packing, no
sums, no products): the CUDA path and the CPU oracle both take its arrays as
their inputs, and neither shares any other code with the other.

Every array is drawn from its own named stream of ``numpy.random.default_rng``
(PCG64) keyed by ``[seed, stream id]``, so changing one array's shape never
changes another array.

Workloads (sizes and distributions):

* ``tiny``     N=256,    K=512,  M=1   t uniform {-1,0,+1}; d uniform [1, 2^15);
                                       x uniform [-127, 127].
* ``ffn_up``   N=6912,   K=2560, M=1   t with P(0)=P(+1)=P(-1)=1/3; d uniform
                                       [1, 2^15); x = clip(rint(N(0, 40^2)), +-127).
* ``ffn_up_q1`` as ``ffn_up`` with binary Q1_0 weights: -1 or +1 with
                                       probability 1/2 each.
* ``lns8``     N=4096,   K=4096        LNS8 activations: each lane is exact zero
                                       with probability 0.1, otherwise its code is
                                       clip(rint(N(74, 12^2)), 1, 127) with a fair
                                       random sign; t with P(0)=1/3; one scale code
                                       per 128-weight group, uniform in 60..88.
* ``lm_head``  N=128256, K=2560        8 ternary planes per weight. Exactly N/2
                                       rows (a seeded permutation) are exactly
                                       ternary: plane 0 uniform {-1,0,+1}, planes
                                       1-7 zero. The other rows have all 8 planes
                                       uniform. Row scale uniform [1, 2^12); x as
                                       in ffn_up; k = 200.
* ``batched``  M=64, N=13824, K=5120   t, d as in ffn_up; x uniform [-127, 127].
"""

from __future__ import annotations

import numpy as np

GROUP = 128

_STREAM_IDS = {
    "t": 1,
    "d": 2,
    "x": 3,
    "code": 4,
    "zero": 5,
    "sign": 6,
    "dcode": 7,
    "planes": 8,
    "ternary_rows": 9,
    "row_scale": 10,
    "signs": 11,
    "sparse_t": 12,
    "states": 13,
    "x64": 14,
    "code_full": 15,
}


def _rng(seed: int, stream: str) -> np.random.Generator:
    return np.random.default_rng([int(seed), _STREAM_IDS[stream]])


def trits(seed: int, shape, stream: str = "t") -> np.ndarray:
    """Ternary values with P(-1) = P(0) = P(+1) = 1/3, int8."""
    return _rng(seed, stream).integers(-1, 2, size=shape, dtype=np.int8)


def trits_sparse(seed: int, shape, zero_frac: float) -> np.ndarray:
    """Ternary values with P(0) = zero_frac and P(-1) = P(+1), int8."""
    r = _rng(seed, "sparse_t")
    t = np.where(r.random(shape) < 0.5, 1, -1).astype(np.int8)
    t[r.random(shape) < zero_frac] = 0
    return t


def signs(seed: int, shape) -> np.ndarray:
    """Binary Q1_0 weights: -1 or +1 with probability 1/2 each, int8."""
    return (2 * _rng(seed, "signs").integers(0, 2, size=shape, dtype=np.int8) - 1).astype(np.int8)


def group_scales(seed: int, n: int, k: int, lo: int = 1, hi: int = 1 << 15) -> np.ndarray:
    """One int32 scale per (row, 128-weight group), uniform over [lo, hi)."""
    return _rng(seed, "d").integers(lo, hi, size=(n, k // GROUP), dtype=np.int32)


def x_uniform(seed: int, shape) -> np.ndarray:
    """int8 activations uniform over [-127, 127]."""
    return _rng(seed, "x").integers(-127, 128, size=shape, dtype=np.int8)


def x_normal40(seed: int, shape) -> np.ndarray:
    """int8 activations clip(rint(N(0, 40^2)), -127, 127)."""
    v = _rng(seed, "x").normal(0.0, 40.0, size=shape)
    return np.clip(np.rint(v), -127, 127).astype(np.int8)


def lns8_activations(seed: int, k: int) -> np.ndarray:
    """LNS8 activation bytes s<<7 | code.

    Each lane is exact zero (code 0) with probability 0.1; otherwise its code
    is clip(rint(N(74, 12^2)), 1, 127). The sign bit is a fair coin for every
    lane, including the zero lanes (a signed zero is still zero).
    """
    code = np.clip(np.rint(_rng(seed, "code").normal(74.0, 12.0, size=k)), 1, 127).astype(np.int64)
    zero = _rng(seed, "zero").random(k) < 0.1
    code[zero] = 0
    sign = _rng(seed, "sign").integers(0, 2, size=k, dtype=np.int64)
    return ((sign << 7) | code).astype(np.uint8)


def lns8_activations_full_range(seed: int, k: int) -> np.ndarray:
    """LNS8 activation bytes with codes over the whole range: each lane is exact
    zero with probability 0.1, otherwise its code is uniform over 1..127 (so a
    fifth of the nonzero lanes sit within 14 codes of either end, where a
    product code can leave 1..127 for scale codes 60..88); fair sign."""
    code = _rng(seed, "code_full").integers(1, 128, size=k, dtype=np.int64)
    zero = _rng(seed, "zero").random(k) < 0.1
    code[zero] = 0
    sign = _rng(seed, "sign").integers(0, 2, size=k, dtype=np.int64)
    return ((sign << 7) | code).astype(np.uint8)


def x_fixed64(seed: int, shape, frac_bits: int = 16, sigma: float = 1.0) -> np.ndarray:
    """int64 fixed-point activations with frac_bits fractional bits:
    rint(N(0, sigma^2) * 2^frac_bits)."""
    return np.rint(_rng(seed, "x64").normal(0.0, sigma, size=shape) * float(1 << frac_bits)).astype(np.int64)


def x_int64_full(seed: int, shape) -> np.ndarray:
    """int64 activations uniform over the whole int64 range."""
    return _rng(seed, "x64").integers(np.iinfo(np.int64).min, np.iinfo(np.int64).max, size=shape,
                                      dtype=np.int64, endpoint=True)


def lns8_activations_states(seed: int, k: int, n_states: int) -> np.ndarray:
    """LNS8 activation bytes whose nonzero codes come from a set of n_states.

    The set is the n_states codes nearest to 74 (code 74 = 1.0; the lower code
    first on a tie), every nonzero lane draws one of them uniformly, and lanes
    are exact zero with probability 0.1 and carry a fair-coin sign, as in
    lns8_activations. n_states = 127 is every code 1..127.
    """
    pool = sorted(range(1, 128), key=lambda c: (abs(c - 74), c))[:n_states]
    r = _rng(seed, "states")
    code = np.asarray(pool, dtype=np.int64)[r.integers(0, n_states, size=k)]
    code[r.random(k) < 0.1] = 0
    sign = r.integers(0, 2, size=k, dtype=np.int64)
    return ((sign << 7) | code).astype(np.uint8)


def lns8_scale_codes(seed: int, n: int, k: int, lo: int = 60, hi: int = 88) -> np.ndarray:
    """One LNS8 scale code per (row, group), uniform over lo..hi inclusive."""
    return _rng(seed, "dcode").integers(lo, hi + 1, size=(n, k // GROUP), dtype=np.uint8)


def lm_head_planes(seed: int, n: int, k: int) -> np.ndarray:
    """[8][n][k] int8 ternary planes; exactly n//2 rows are exactly ternary."""
    planes = _rng(seed, "planes").integers(-1, 2, size=(8, n, k), dtype=np.int8)
    rows = _rng(seed, "ternary_rows").permutation(n)[: n // 2]
    planes[1:, rows, :] = 0
    return planes


def row_scales(seed: int, n: int, lo: int = 1, hi: int = 1 << 12) -> np.ndarray:
    """One int32 scale per row, uniform over [lo, hi)."""
    return _rng(seed, "row_scale").integers(lo, hi, size=n, dtype=np.int32)


# ---------------------------------------------------------------------------
# The named workloads. Each returns a dict of host numpy arrays plus sizes.
# Sizes can be overridden to draw smaller cases with the same distributions.
# ---------------------------------------------------------------------------

def tiny(seed: int = 0, N: int = 256, K: int = 512, M: int = 1) -> dict:
    return dict(kind="i8", N=N, K=K, M=M,
                t=trits(seed, (N, K)), d=group_scales(seed, N, K), x=x_uniform(seed, (M, K)))


def ffn_up(seed: int = 0, N: int = 6912, K: int = 2560, M: int = 1) -> dict:
    return dict(kind="i8", N=N, K=K, M=M,
                t=trits(seed, (N, K)), d=group_scales(seed, N, K), x=x_normal40(seed, (M, K)))


def ffn_up_q1(seed: int = 0, N: int = 6912, K: int = 2560, M: int = 1) -> dict:
    return dict(kind="q1", N=N, K=K, M=M,
                t=signs(seed, (N, K)), d=group_scales(seed, N, K), x=x_normal40(seed, (M, K)))


def lns8(seed: int = 0, N: int = 4096, K: int = 4096) -> dict:
    return dict(kind="lns8", N=N, K=K,
                t=trits(seed, (N, K)), dcode=lns8_scale_codes(seed, N, K), xa=lns8_activations(seed, K))


def lm_head(seed: int = 0, N: int = 128256, K: int = 2560, k: int = 200) -> dict:
    return dict(kind="planes8", N=N, K=K, k=k,
                planes=lm_head_planes(seed, N, K), s=row_scales(seed, N), x=x_normal40(seed, (K,)))


def batched(seed: int = 0, M: int = 64, N: int = 13824, K: int = 5120) -> dict:
    return dict(kind="i8", N=N, K=K, M=M,
                t=trits(seed, (N, K)), d=group_scales(seed, N, K), x=x_uniform(seed, (M, K)))


WORKLOADS = {
    "tiny": tiny,
    "ffn_up": ffn_up,
    "lns8": lns8,
    "lm_head": lm_head,
    "batched": batched,
}
