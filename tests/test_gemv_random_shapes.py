"""GPU parity of tg_gemv_i8 on seeded random shapes: row counts, lengths, token
counts, weight kinds, floor shifts and activation ranges drawn at random, so
that the kernel choice by token count and the launch plan by shape (whole or
half tiles, groups per warp, resident-CTA cap) are crossed in combinations no
other test names. Each case against the CPU oracle, element by element."""

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

CASES = 40


@pytest.fixture(scope="module", autouse=True)
def built():
    from gpu_helpers import ensure_built
    ensure_built()


def draw(case):
    """One case: (N, K, M, kind, frac, t, d, x) from its own seed."""
    r = np.random.default_rng(1000 + case)
    N = int(r.choice([1, 17, 33, 200, 511, 1000, 2049, 4100, 9800]))
    K = 128 * int(r.integers(1, 49))                 # 128 .. 6144
    M = int(r.choice([1, 1, 1, 2, 3, 4, 5, 6, 7, 8, 9, 12, 16, 17]))
    kind = "q1" if r.random() < 0.3 else "ternary"
    frac = int(r.choice([0, 0, 0, 1, 7, 20]))
    if kind == "q1":
        t = np.where(r.random((N, K)) < 0.5, 1, -1).astype(np.int8)
    else:
        t = r.integers(-1, 2, size=(N, K), dtype=np.int8)
    big = r.random() < 0.3                           # int32-range scales, else up to 2^15
    hi = np.iinfo(np.int32).max if big else 1 << 15
    d = r.integers(-hi, hi, size=(N, K // 128), dtype=np.int64).astype(np.int32)
    x = r.integers(-128, 128, size=(M, K), dtype=np.int64).astype(np.int8)
    return N, K, M, kind, frac, t, d, x


@pytest.mark.parametrize("case", range(CASES))
def test_random_shape(case):
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import gemv, pack_to_device
    N, K, M, kind, frac, t, d, x = draw(case)
    if kind == "q1":
        wd, L = pack_to_device(tg.TG_BINARY_Q1, t, d)
        L.frac = frac
        ref = oracle.gemv_q1((t > 0).astype(np.uint8), d, x, frac)
    else:
        wd, L = pack_to_device(tg.TG_TERNARY_I8, t, d)
        L.frac = frac
        ref = oracle.gemv_i8_frac(t, d, x, frac) if frac else oracle.gemv_i8(t, d, x)
    np.testing.assert_array_equal(gemv(wd, L, x), ref, err_msg=f"N={N} K={K} M={M} {kind} frac={frac}")
