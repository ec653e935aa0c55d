"""GPU parity of tg_gemv_lns8_phase (both exact routes) and tg_lmhead_argmax_topk
(both paths) on seeded random shapes and value ranges, against the CPU oracle:
A and the lm_head logits, ids, scores and argmax bit-exact, S within the fp64
materialisation tolerance (1e-12 relative, against max(|S|, 2^-40 * the size
of its terms), as in test_lns8_parity.py)."""

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.gpu

S_RTOL = 1e-12


@pytest.fixture(scope="module", autouse=True)
def built():
    from gpu_helpers import ensure_built
    ensure_built()


def lns8_case(case):
    r = np.random.default_rng(2000 + case)
    N = int(r.choice([1, 16, 33, 129, 640, 1500, 3001]))
    K = 128 * int(r.integers(1, 65))                 # 128 .. 8192
    t = r.integers(-1, 2, size=(N, K), dtype=np.int8)
    mode = int(r.integers(0, 3))
    if mode == 0:     # the configured distributions
        code = np.clip(np.rint(r.normal(74, 12, size=K)), 1, 127).astype(np.int64)
        dcode = r.integers(60, 89, size=(N, K // 128))
    elif mode == 1:   # codes over the whole range
        code = r.integers(1, 128, size=K)
        dcode = r.integers(60, 89, size=(N, K // 128))
    else:             # every byte value, scale codes over the whole byte
        code = r.integers(0, 128, size=K)
        dcode = r.integers(0, 256, size=(N, K // 128))
    code[r.random(K) < 0.1] = 0
    xa = ((r.integers(0, 2, size=K) << 7) | code).astype(np.uint8)
    return N, K, t, dcode.astype(np.uint8), xa


@pytest.mark.parametrize("route", ["direct", "stateset"])
@pytest.mark.parametrize("case", range(16))
def test_lns8_random_shape(case, route):
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import lns8, pack_to_device
    N, K, t, dcode, xa = lns8_case(case)
    wd, L = pack_to_device(tg.TG_TERNARY_LNS8, t, dcode)
    if route == "stateset":
        L.flags |= tg.TG_FLAG_LNS8_STATE_SET
    A, S = lns8(wd, L, xa)
    A_ref = oracle.lns8_direct(t, dcode, xa)
    np.testing.assert_array_equal(A, A_ref, err_msg=f"N={N} K={K}")
    S_ref = oracle.lns8_materialise(A_ref)
    _, mag = oracle.lns8_materialise_hi(A_ref)
    denom = np.maximum(np.abs(S_ref), 2.0 ** -40 * mag)
    denom[denom == 0] = 1.0
    assert np.all(np.abs(S - S_ref) / denom <= S_RTOL)


def lmhead_case(case):
    r = np.random.default_rng(3000 + case)
    N = int(r.choice([1, 7, 100, 1000, 4097, 20000]))
    K = 128 * int(r.integers(1, 41))                 # 128 .. 5120
    k = int(min(N, int(r.choice([1, 2, 10, 64, 200, 1024]))))
    planes = r.integers(-1, 2, size=(8, N, K), dtype=np.int8)
    ternary_rows = r.random(N) < float(r.choice([0.0, 0.5, 1.0]))
    planes[1:, ternary_rows, :] = 0
    # row scales up to 1, 2^12 or 2^20, held below the call's bound: max|logit| times
    # the key's index bits (enough for N) must stay below 4e18
    idx_bits = max(1, (N - 1).bit_length())
    s_cap = int(3.9e18 / (3280.0 * 128.0 * K * float(1 << idx_bits)))
    s_hi = min(int(r.choice([2, 1 << 12, 1 << 20])), max(2, s_cap))
    s = r.integers(1, s_hi, size=N).astype(np.int32)
    x = np.clip(np.rint(r.normal(0, float(r.choice([5.0, 40.0, 120.0])), size=K)), -127, 127).astype(np.int8)
    return N, K, k, planes, s, x


@pytest.mark.parametrize("case", range(16))
def test_lmhead_random_shape(case):
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import lmhead, pack_to_device
    N, K, k, planes, s, x = lmhead_case(case)
    wd, L = pack_to_device(tg.TG_PLANES8, planes, s)
    logits_ref = oracle.lmhead_logits(planes, s, x)
    ids_ref, top_ref = oracle.topk(logits_ref, k)
    am_ref = oracle.argmax(logits_ref)
    for full in (True, False):
        out = lmhead(wd, L, x, k, full)
        if full:
            np.testing.assert_array_equal(out["logits"], logits_ref)
        np.testing.assert_array_equal(out["ids"], ids_ref, err_msg=f"N={N} K={K} k={k} full={full}")
        np.testing.assert_array_equal(out["scores"], top_ref)
        assert out["argmax"] == am_ref
        assert k <= out["ncand"] <= N
