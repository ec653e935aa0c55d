"""GPU parity of tg_gemv_lns8_phase against the CPU oracle.

A[r][p] must be bit-exact. S is compared within 1e-12 relative error, the
tolerance for the fp64 materialisation; the denominator is max(|S|, 2^-40 *
2^-9 sum_p |A[p]| F[p]) so that rows whose eight terms cancel to near zero
are judged against the size of the terms, not of the near-zero result.
"""

import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

S_RTOL = 1e-12


@pytest.fixture(scope="module", autouse=True)
def built():
    from gpu_helpers import ensure_built
    ensure_built()


def check(w, with_S=True):
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import lns8, pack_to_device
    wd, L = pack_to_device(tg.TG_TERNARY_LNS8, w["t"], w["dcode"])
    A, S = lns8(wd, L, w["xa"], with_S)
    A_ref = oracle.lns8_direct(w["t"], w["dcode"], w["xa"])
    np.testing.assert_array_equal(A, A_ref)
    if with_S:
        S_ref = oracle.lns8_materialise(A_ref)
        _, mag = oracle.lns8_materialise_hi(A_ref)
        denom = np.maximum(np.abs(S_ref), 2.0 ** -40 * mag)
        denom[denom == 0] = 1.0
        err = np.abs(S - S_ref) / denom
        assert np.all(err <= S_RTOL), float(err.max())
    return A, S


def test_lns8_workload_full_size():
    check(W.lns8())


def wide(seed, N, K):
    """Codes over 0..127 and scale codes over the whole byte range, so that both
    clamps (k <= 0 and k > 127) and signed zeros occur often."""
    w = W.lns8(seed=seed, N=N, K=K)
    rng = np.random.default_rng(seed)
    w["xa"] = rng.integers(0, 256, size=K, dtype=np.uint8)
    w["dcode"] = rng.integers(0, 256, size=w["dcode"].shape, dtype=np.uint8)
    return w


@pytest.mark.parametrize("N,K", [(1, 128), (33, 128), (95, 384), (1000, 4096), (40, 12800)])
def test_clamp_heavy_and_ragged(N, K):
    check(wide(N, N, K))


def test_extreme_codes():
    N, K = 64, 256
    t = np.ones((N, K), np.int8)
    t[1::2] = -1
    xa = np.full(K, 127, np.uint8)
    xa[::3] = 0x80 | 127
    dcode = np.full((N, 2), 255, np.uint8)
    dcode[::4] = 0
    dcode[1::4] = 74
    A, _ = check(dict(t=t, dcode=dcode, xa=xa))
    # scale code 255 saturates every product to code 127 = phase 7, band 15
    assert np.count_nonzero(A[2, :7]) == 0 and abs(A[2, 7]) > 0


def test_without_S():
    check(W.lns8(seed=3, N=77, K=512), with_S=False)
