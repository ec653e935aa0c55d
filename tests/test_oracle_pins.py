"""Pins that tie the CPU oracle to what the pages and the mathematics fix.

No test here re-types the oracle's own formula. Each one checks the oracle
against something independent of it: a value the pages print (tests/golden/),
a closed form, an invariant, a special case that reduces to a library routine
(numpy integer matmul, numpy sorting), or brute force over tiny inputs. The
cases are chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, a transposed scale index, an off-by-one group boundary, a wrong
clamp) fails at least one of them.
"""

import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore")


def dequantised(t, d):
    """Dense integer weight matrix W[r,i] = d[r, i//128] * t[r,i]."""
    return t.astype(np.int64) * np.repeat(d.astype(np.int64), 128, axis=1)


# ---------------------------------------------------------------------------
# Ternary GEMV
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("N,K,M,seed", [(1, 128, 1, 0), (7, 384, 3, 1), (33, 640, 2, 2)])
def test_gemv_equals_dense_matmul(N, K, M, seed):
    # Distributing the group scale over its 128 lanes turns the grouped sum into
    # a plain matrix-vector product, which numpy computes by another route.
    w = W.tiny(seed=seed, N=N, K=K, M=M)
    y = oracle.gemv_i8(w["t"], w["d"], w["x"])
    ref = w["x"].astype(np.int64) @ dequantised(w["t"], w["d"]).T
    assert y.dtype == np.int64 and y.shape == (M, N)
    np.testing.assert_array_equal(y, ref)


def test_gemv_three_forms_agree():
    # direct signed sum == two-bitmask masked sum == state-set popcount form
    w = W.ffn_up(seed=3, N=9, K=256, M=2)
    a = oracle.gemv_i8(w["t"], w["d"], w["x"])
    np.testing.assert_array_equal(a, oracle.gemv_i8_masked(w["t"], w["d"], w["x"]))
    np.testing.assert_array_equal(a, oracle.gemv_i8_stateset(w["t"], w["d"], w["x"]))


def test_gemv_single_lane_closed_form():
    # x = v * e_i picks d[r, i // 128] * t[r, i] * v for every lane i.
    N, K = 3, 256
    w = W.tiny(seed=4, N=N, K=K)
    for v in (-128, -1, 1, 127):
        for i in range(K):
            x = np.zeros((1, K), dtype=np.int8)
            x[0, i] = v
            y = oracle.gemv_i8(w["t"], w["d"], x)[0]
            expect = [int(w["d"][r, i // 128]) * int(w["t"][r, i]) * v for r in range(N)]
            assert y.tolist() == expect


def test_gemv_all_trit_patterns_on_four_lanes():
    # Brute force: every one of the 3^4 trit patterns on lanes 0..3.
    K = 128
    x = np.zeros((1, K), dtype=np.int8)
    x[0, :4] = [5, -7, 11, -128]
    d = np.array([[3]], dtype=np.int32)
    for pat in itertools.product((-1, 0, 1), repeat=4):
        t = np.zeros((1, K), dtype=np.int8)
        t[0, :4] = pat
        expect = 3 * (5 * pat[0] - 7 * pat[1] + 11 * pat[2] - 128 * pat[3])
        assert oracle.gemv_i8(t, d, x)[0, 0] == expect


def test_gemv_special_cases():
    w = W.tiny(seed=5, N=6, K=384, M=2)
    t, d, x = w["t"], w["d"], w["x"]
    # all weights zero -> zero
    assert not oracle.gemv_i8(np.zeros_like(t), d, x).any()
    # all weights +1 -> sum_g d[r,g] * (sum of x over group g)
    ones = np.ones_like(t)
    gsum = x.astype(np.int64).reshape(2, 3, 128).sum(axis=2)          # [M][G]
    np.testing.assert_array_equal(oracle.gemv_i8(ones, d, x), gsum @ d.astype(np.int64).T)
    # negating x (no -128) negates y
    xs = np.clip(x, -127, 127)
    np.testing.assert_array_equal(oracle.gemv_i8(t, d, -xs), -oracle.gemv_i8(t, d, xs))
    # linear in the scales
    d2 = W.group_scales(9, 6, 384)
    np.testing.assert_array_equal(oracle.gemv_i8(t, d + d2, x),
                                  oracle.gemv_i8(t, d, x) + oracle.gemv_i8(t, d2, x))


def test_gemv_permutation_invariance():
    rng = np.random.default_rng(11)
    w = W.ffn_up(seed=6, N=5, K=512, M=2)
    t, d, x = w["t"], w["d"], w["x"]
    y = oracle.gemv_i8(t, d, x)
    # shuffle lanes within each group (same permutation on t columns and x)
    perm = np.concatenate([g * 128 + rng.permutation(128) for g in range(4)])
    np.testing.assert_array_equal(oracle.gemv_i8(t[:, perm], d, x[:, perm]), y)
    # permute whole groups together with their scales
    gp = rng.permutation(4)
    cols = np.concatenate([np.arange(g * 128, (g + 1) * 128) for g in gp])
    np.testing.assert_array_equal(oracle.gemv_i8(t[:, cols], d[:, gp], x[:, cols]), y)
    # a lane moved across a group boundary changes the result (group index matters)
    t2 = t.copy()
    t2[:, [127, 128]] = t2[:, [128, 127]]
    x2 = x.copy()
    x2[:, [127, 128]] = x2[:, [128, 127]]
    if not np.array_equal(d[:, 0], d[:, 1]):
        assert not np.array_equal(oracle.gemv_i8(t2, d, x2), y) or not (t[:, 127] * x[:, 127] - t[:, 128] * x[:, 128]).any()


def test_gemv_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oracle.gemv_i8(np.zeros((2, 100), np.int8), np.zeros((2, 0), np.int32), np.zeros((1, 100), np.int8))


# ---------------------------------------------------------------------------
# LNS8 eight-phase path
# ---------------------------------------------------------------------------

def one_lane(code, dcode, t=1, sign=0, K=128):
    """A single nonzero lane at position 0 of one group."""
    tt = np.zeros((1, K), dtype=np.int8)
    tt[0, 0] = t
    xa = np.zeros(K, dtype=np.uint8)
    xa[0] = (sign << 7) | code
    dc = np.full((1, K // 128), dcode, dtype=np.uint8)
    return tt, dc, xa


def test_lns8_page_values(golden_dir):
    # Values the BitState brief prints: code 0 = 0, code 74 = 1.0, code 122 = 64,
    # eight codes = exactly x2. With scale code 74 (= 1.0) the product code is
    # the activation code itself, so S is that code's value.
    cases = json.load(open(os.path.join(golden_dir, "lns8_page_values.json")))["cases"]
    for c in cases:
        if "code" in c and "value" in c:
            S = oracle.lns8_materialise(oracle.lns8_direct(*one_lane(c["code"], 74)))
            assert S[0] == c["value"], c
        if "ratio" in c:
            for a in range(1, 127 - c["code_step"] + 1):
                s0 = oracle.lns8_materialise(oracle.lns8_direct(*one_lane(a, 74)))[0]
                s1 = oracle.lns8_materialise(oracle.lns8_direct(*one_lane(a + c["code_step"], 74)))[0]
                assert s1 == c["ratio"] * s0


def test_lns8_single_lane_routes_to_phase_and_band(golden_dir):
    # A single product state k lands as +-2^(k>>3) in A[k&7] and nowhere else, and
    # k = (120 + phase) + 8 * (band - 15) recovers k from that position.
    for k in range(1, 128):
        for sign in (0, 1):
            A = oracle.lns8_direct(*one_lane(k, 74, sign=sign))[0]
            nz = np.flatnonzero(A)
            assert nz.tolist() == [k % 8]
            band = int(round(math.log2(abs(int(A[k % 8])))))
            assert abs(int(A[k % 8])) == 1 << band
            assert (120 + k % 8) + 8 * (band - 15) == k
            assert (A[k % 8] < 0) == bool(sign)


def test_lns8_value_is_two_to_the_code_offset():
    # S of one lane equals 2^((k-74)/8) to fp64 rounding, for every product code.
    for k in range(1, 128):
        S = oracle.lns8_materialise(oracle.lns8_direct(*one_lane(k, 74)))[0]
        assert abs(S - 2.0 ** ((k - 74) / 8)) <= 2.0 ** -52 * S


def test_lns8_sign_rule():
    # S1 = activation sign XOR weight sign.
    for t, sign, neg in ((1, 0, False), (1, 1, True), (-1, 0, True), (-1, 1, False)):
        A = oracle.lns8_direct(*one_lane(80, 74, t=t, sign=sign))[0]
        assert (A.sum() < 0) == neg


def test_lns8_clamp_edges():
    # k = a + d - 74: k <= 0 is exact zero, k > 127 saturates to 127.
    cases = [  # (a, d, expected k or None)
        (14, 60, None), (1, 60, None), (15, 60, 1), (1, 74, 1), (1, 88, 15),
        (113, 88, 127), (114, 88, 127), (127, 88, 127), (127, 74, 127), (100, 88, 114),
        (60, 60, 46),
    ]
    for a, d, k in cases:
        A = oracle.lns8_direct(*one_lane(a, d))[0]
        if k is None:
            assert not A.any(), (a, d)
        else:
            assert A.tolist() == [(1 << (k >> 3)) if p == (k & 7) else 0 for p in range(8)], (a, d)


def test_lns8_signed_zero_and_zero_weight():
    for xa_byte in (0x00, 0x80):
        tt, dc, xa = one_lane(1, 74)
        xa[0] = xa_byte
        assert not oracle.lns8_direct(tt, dc, xa).any()
    assert not oracle.lns8_direct(*one_lane(90, 74, t=0)).any()


def _lns8_case(seed, N, K, wide=False):
    w = W.lns8(seed=seed, N=N, K=K)
    if wide:
        # widen codes and scale codes to hit both clamps often
        rng = np.random.default_rng(seed + 100)
        code = rng.integers(0, 128, size=K)
        sign = rng.integers(0, 2, size=K)
        w["xa"] = ((sign << 7) | code).astype(np.uint8)
        w["dcode"] = rng.choice(np.array([0, 1, 30, 60, 74, 88, 120, 255], dtype=np.uint8),
                                size=w["dcode"].shape)
    return w


@pytest.mark.parametrize("seed,wide", [(0, False), (1, True), (2, True)])
def test_lns8_four_paths_exactly_equal(seed, wide):
    # direct == histogram-derived == Tile64x2 == state-set, exactly (Phase A).
    w = _lns8_case(seed, 6, 512, wide)
    a = oracle.lns8_direct(w["t"], w["dcode"], w["xa"])
    for f in (oracle.lns8_histogram, oracle.lns8_tile64, oracle.lns8_stateset):
        np.testing.assert_array_equal(f(w["t"], w["dcode"], w["xa"]), a)


def test_lns8_materialisation_matches_direct_decode():
    # S = 2^-9 sum_p A[p] F[p] equals the FP64 direct decode sum of
    # sign * 2^((k-74)/8) within fp64 rounding, and the long double value.
    w = _lns8_case(3, 16, 1024)
    A = oracle.lns8_direct(w["t"], w["dcode"], w["xa"])
    S = oracle.lns8_materialise(A)
    S_dec, mag = oracle.lns8_decode_fp64(w["t"], w["dcode"], w["xa"])
    S_hi, mag_hi = oracle.lns8_materialise_hi(A)
    K = 1024
    assert np.all(np.abs(S - S_dec) <= (K + 16) * 2.0 ** -52 * mag)
    assert np.all(np.abs(S - S_hi) <= 16 * 2.0 ** -52 * mag_hi)
    # per-phase cancellation can only shrink the magnitude sum
    assert np.all(mag_hi <= mag * (1 + 1e-12))


def test_lns8_materialise_basis():
    # A = 2^b e_p materialises to exactly 2^(b-9) F[p]; F[2] = 1; F[p]^8 = 2^(p-2).
    F = oracle.lns8_F()
    assert F[2] == 1.0
    for p in range(8):
        assert abs(F[p] ** 8 - 2.0 ** (p - 2)) <= 64 * 2.0 ** -52 * 2.0 ** (p - 2)
        for b in range(16):
            A = np.zeros((1, 8), dtype=np.int64)
            A[0, p] = 1 << b
            assert oracle.lns8_materialise(A, F)[0] == math.ldexp(F[p], b - 9)
    assert np.all(np.diff(F) > 0) and F[7] < 2 * F[0]


def test_lns8_shuffle_within_group_invariant():
    rng = np.random.default_rng(7)
    w = _lns8_case(4, 5, 384, wide=True)
    A = oracle.lns8_direct(w["t"], w["dcode"], w["xa"])
    perm = np.concatenate([g * 128 + rng.permutation(128) for g in range(3)])
    np.testing.assert_array_equal(oracle.lns8_direct(w["t"][:, perm], w["dcode"], w["xa"][perm]), A)


# ---------------------------------------------------------------------------
# lm_head over 8 base-3 planes
# ---------------------------------------------------------------------------

POW3 = np.array([3 ** (7 - p) for p in range(8)], dtype=np.int64)


def test_balanced_ternary_bijection():
    # Every integer in [-3280, 3280] has exactly one 8-digit balanced-ternary form.
    seen = set()
    for w in range(-3280, 3281):
        dg = oracle.planes_of_weight(w)
        assert set(dg.tolist()) <= {-1, 0, 1}
        assert int(dg.astype(np.int64) @ POW3) == w
        seen.add(tuple(dg.tolist()))
    assert len(seen) == 3 ** 8
    with pytest.raises(ValueError):
        oracle.planes_of_weight(3281)


def test_exactly_ternary_rows_are_lossless(golden_dir):
    # planes 1..7 zero -> W = 2187 * t, plane 0 carries the codes with no residual;
    # the planes of 2187*t are recovered as (t, 0, ..., 0).
    rng = np.random.default_rng(8)
    N, K = 12, 256
    t = rng.integers(-1, 2, size=(N, K), dtype=np.int8)
    planes = np.zeros((8, N, K), dtype=np.int8)
    planes[0] = t
    s = W.row_scales(1, N)
    x = W.x_normal40(1, (K,))
    logits = oracle.lmhead_logits(planes, s, x)
    np.testing.assert_array_equal(logits, s.astype(np.int64) * (2187 * (t.astype(np.int64) @ x.astype(np.int64))))
    for v in (-1, 0, 1):
        assert oracle.planes_of_weight(2187 * v).tolist() == [v] + [0] * 7


def _lm_case(seed, N, K):
    return W.lm_head(seed=seed, N=N, K=K)


@pytest.mark.parametrize("seed,N,K", [(0, 50, 128), (1, 301, 256)])
def test_lmhead_logits_equal_dense_matmul(seed, N, K):
    w = _lm_case(seed, N, K)
    Wint = np.tensordot(POW3, w["planes"].astype(np.int64), axes=(0, 0))   # [N][K]
    ref = w["s"].astype(np.int64) * (Wint @ w["x"].astype(np.int64))
    np.testing.assert_array_equal(oracle.lmhead_logits(w["planes"], w["s"], w["x"]), ref)


def test_topk_and_argmax_match_numpy_sort():
    rng = np.random.default_rng(9)
    for trial in range(20):
        n = int(rng.integers(1, 400))
        scores = rng.integers(-5, 6, size=n).astype(np.int64) * int(rng.integers(1, 1 << 40))
        k = int(rng.integers(1, n + 1))
        order = np.lexsort((np.arange(n), -scores))            # score desc, index asc
        ids, top = oracle.topk(scores, k)
        np.testing.assert_array_equal(ids, order[:k])
        np.testing.assert_array_equal(top, scores[order[:k]])
        assert oracle.argmax(scores) == int(np.argmax(scores)) == ids[0]


def test_ties_resolve_to_lowest_index():
    w = _lm_case(2, 40, 128)
    planes = w["planes"].copy()
    s = w["s"].copy()
    for dst, src in ((31, 3), (17, 3), (25, 8)):
        planes[:, dst] = planes[:, src]
        s[dst] = s[src]
    logits = oracle.lmhead_logits(planes, s, w["x"])
    ids, _ = oracle.topk(logits, 40)
    pos = {int(r): j for j, r in enumerate(ids)}
    assert pos[3] < pos[17] < pos[31] and pos[8] < pos[25]
    best = int(np.flatnonzero(logits == logits.max())[0])
    assert oracle.argmax(logits) == best


@pytest.mark.parametrize("seed,N,K,k", [(0, 500, 256, 20), (1, 2000, 128, 200), (2, 300, 384, 300), (3, 64, 128, 1)])
def test_two_stage_equals_full_topk(seed, N, K, k):
    w = _lm_case(seed, N, K)
    logits = oracle.lmhead_logits(w["planes"], w["s"], w["x"])
    order = np.lexsort((np.arange(N), -logits))
    ids, top, lo, hi, C = oracle.lmhead_two_stage(w["planes"], w["s"], w["x"], k)
    np.testing.assert_array_equal(ids, order[:k])
    np.testing.assert_array_equal(top, logits[order[:k]])
    # the bound brackets every exact logit, and the candidate set holds the top-k
    assert np.all(lo <= logits) and np.all(logits <= hi)
    assert k <= C <= N
    # lo/hi are the planes 0..3 dense product -+ s * 40 * sum|x| (page bound), and the
    # candidates are exactly the rows whose hi reaches the k-th largest lo
    x = w["x"].astype(np.int64)
    stage1 = np.tensordot(POW3[:4], w["planes"][:4].astype(np.int64), axes=(0, 0)) @ x
    B = w["s"].astype(np.int64) * 40 * np.abs(x).sum()
    np.testing.assert_array_equal(lo, w["s"].astype(np.int64) * stage1 - B)
    np.testing.assert_array_equal(hi, w["s"].astype(np.int64) * stage1 + B)
    tau = np.sort(lo)[::-1][k - 1]
    assert C == int((hi >= tau).sum())


def test_stage1_truncation_fraction(golden_dir):
    # The planes 4..7 residual of any weight is at most 40/2187 of plane 0's unit,
    # the page's "about 1.85%" (the infinite tail 3^-4 * 3/2 = 1/54 is 1.852%).
    case = [c for c in json.load(open(os.path.join(golden_dir, "lmhead_page_values.json")))["cases"]
            if "approx_fraction" in c][0]
    w = _lm_case(4, 200, 256)
    x = w["x"].astype(np.int64)
    rest = np.tensordot(POW3[4:], w["planes"][4:].astype(np.int64), axes=(0, 0)) @ x
    ratio = np.abs(rest) / (2187.0 * np.abs(x).sum())
    assert ratio.max() <= 40 / 2187
    # the page's figure is the infinite tail; the finite four-plane sum is below it
    assert abs(1 / 54 - case["approx_fraction"]) / case["approx_fraction"] < case["rel_tol"]
    assert 40 / 2187 < 1 / 54
    assert sum(3.0 ** -p for p in range(4, 8)) * 2187 == pytest.approx(40)


def test_lmhead_k_shuffle_invariant():
    rng = np.random.default_rng(10)
    w = _lm_case(5, 30, 256)
    perm = rng.permutation(256)
    np.testing.assert_array_equal(oracle.lmhead_logits(w["planes"][:, :, perm], w["s"], w["x"][perm]),
                                  oracle.lmhead_logits(w["planes"], w["s"], w["x"]))


def test_workload_distributions():
    # The generators draw what the workloads state (sizes reduced).
    w = W.lm_head(seed=0, N=1000, K=128)
    exact_rows = ~w["planes"][1:].any(axis=(0, 2))
    assert exact_rows.sum() == 500
    assert w["s"].min() >= 1 and w["s"].max() < 4096
    a = W.lns8(seed=0, N=4, K=4096)
    code = a["xa"] & 0x7F
    assert 0.07 < (code == 0).mean() < 0.13
    assert a["dcode"].min() >= 60 and a["dcode"].max() <= 88
    f = W.ffn_up(seed=0, N=300, K=2560)
    assert abs((f["t"] == 0).mean() - 1 / 3) < 0.01
    assert f["x"].min() >= -127 and f["x"].max() <= 127
    assert abs(f["x"].astype(float).std() - 40) < 3


def test_stage1_bound_is_tight():
    # A row whose planes 4..7 all equal sign(x_i) has residual exactly 40 * sum|x|,
    # so its exact logit equals the upper bound; with -sign(x) it equals the lower.
    N, K = 6, 256
    w = _lm_case(6, N, K)
    planes, s, x = w["planes"].copy(), w["s"], w["x"]
    sg = np.sign(x).astype(np.int8)
    planes[4:, 1, :] = sg
    planes[4:, 4, :] = -sg
    logits = oracle.lmhead_logits(planes, s, x)
    _, _, lo, hi, _ = oracle.lmhead_two_stage(planes, s, x, 2)
    assert logits[1] == hi[1] and logits[4] == lo[4]
    assert hi[1] - lo[1] == 2 * int(s[1]) * 40 * int(np.abs(x.astype(np.int64)).sum())


# ---------------------------------------------------------------------------
# Per-group floor (integer engine §4.1/§4.2 arshift(., frac)) and Q1_0 binary
# weights (integer engine §4.1)
# ---------------------------------------------------------------------------

def test_frac_zero_is_the_plain_apply():
    w = W.tiny(seed=3, N=40, K=384, M=3)
    np.testing.assert_array_equal(oracle.gemv_i8_frac(w["t"], w["d"], w["x"], 0),
                                  oracle.gemv_i8(w["t"], w["d"], w["x"]))


def test_frac_floors_toward_minus_infinity():
    # one group, one nonzero lane: the group's scaled sum is -5 or +5
    K = 128
    t = np.zeros((2, K), np.int8)
    t[0, 7] = -1
    t[1, 7] = 1
    d = np.ones((2, 1), np.int32)
    x = np.zeros((1, K), np.int8)
    x[0, 7] = 5
    y = oracle.gemv_i8_frac(t, d, x, 1)
    assert y[0, 0] == -3 and y[0, 1] == 2          # floor(-2.5) = -3, floor(2.5) = 2
    y = oracle.gemv_i8_frac(t, d, x, 3)
    assert y[0, 0] == -1 and y[0, 1] == 0          # floor(-5/8) = -1, floor(5/8) = 0


def test_frac_floor_is_per_group():
    # two groups whose scaled sums are each 1: floor(1/2) + floor(1/2) = 0, while
    # flooring after the sum would give floor(2/2) = 1
    K = 256
    t = np.zeros((1, K), np.int8)
    t[0, 0] = 1
    t[0, 128] = 1
    d = np.ones((1, 2), np.int32)
    x = np.zeros((1, K), np.int8)
    x[0, 0] = 1
    x[0, 128] = 1
    assert oracle.gemv_i8_frac(t, d, x, 1)[0, 0] == 0
    assert oracle.gemv_i8_frac(t, d, x, 0)[0, 0] == 2


def test_frac_matches_a_floor_division_of_each_group():
    w = W.tiny(seed=8, N=17, K=512, M=2)
    for frac in (1, 5, 13, 31):
        y = oracle.gemv_i8_frac(w["t"], w["d"], w["x"], frac)
        G = 4
        parts = np.stack([oracle.gemv_i8(w["t"][:, 128 * g:128 * (g + 1)], w["d"][:, g:g + 1],
                                         w["x"][:, 128 * g:128 * (g + 1)]) for g in range(G)])
        # python integers: // is floor division
        ref = np.array([[sum(int(parts[g, m, r]) // (1 << frac) for g in range(G)) for r in range(17)]
                        for m in range(2)], dtype=np.int64)
        np.testing.assert_array_equal(y, ref)


def test_q1_two_pos_minus_total_equals_signed_sum():
    # the page's identity 2 * pos_sum - block_total = sum sign * x, checked against
    # the ternary apply on the same +-1 weights
    rng = np.random.default_rng(9)
    N, K, M = 23, 640, 3
    bits = rng.integers(0, 2, size=(N, K)).astype(np.uint8)
    signs = (2 * bits.astype(np.int16) - 1).astype(np.int8)
    d = rng.integers(-(1 << 15), 1 << 15, size=(N, K // 128)).astype(np.int32)
    x = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    for frac in (0, 4):
        np.testing.assert_array_equal(oracle.gemv_q1(bits, d, x, frac), oracle.gemv_i8_frac(signs, d, x, frac))
    # and the plain matrix product for frac = 0
    ref = np.zeros((M, N), np.int64)
    for g in range(K // 128):
        sl = slice(128 * g, 128 * (g + 1))
        ref += (x[:, sl].astype(np.int64) @ signs[:, sl].T.astype(np.int64)) * d[:, g].astype(np.int64)
    np.testing.assert_array_equal(oracle.gemv_q1(bits, d, x, 0), ref)


def test_q1_special_cases():
    K = 256
    x = np.arange(-64, 192, dtype=np.int64).astype(np.int8).reshape(1, K)
    d = np.array([[3, -2]], np.int32)
    total = [int(x[0, :128].astype(np.int64).sum()), int(x[0, 128:].astype(np.int64).sum())]
    ones = np.ones((1, K), np.uint8)
    zeros = np.zeros((1, K), np.uint8)
    assert oracle.gemv_q1(ones, d, x)[0, 0] == 3 * total[0] - 2 * total[1]       # every sign +1
    assert oracle.gemv_q1(zeros, d, x)[0, 0] == -3 * total[0] + 2 * total[1]     # every sign -1
    with pytest.raises(ValueError):
        oracle.gemv_q1(np.full((1, K), 2, np.uint8), d, x)


# ---------------------------------------------------------------------------
# int64 fixed-point activations (integer engine §4.4), exact modulo 2^64 (its
# §5: the limb-decomposed apply "recombined in int64 (exact mod-2^64)").
# ---------------------------------------------------------------------------

def _signed_digits(x):
    """Signed base-256 digits s_0..s_7 in [-128, 127] with x = sum s_l 256^l
    (mod 2^64), from Python integers (a carry per digit, no wrapping)."""
    digits = np.zeros((8,) + x.shape, dtype=np.int8)
    u = [int(v) % (1 << 64) for v in x.ravel()]
    for l in range(8):
        for idx, v in enumerate(u):
            b = v & 0xFF
            s = b - 256 if b >= 128 else b
            digits[l].ravel()[idx] = s
            u[idx] = (v - s) >> 8
    return digits


def _wrap64(v):
    v %= 1 << 64
    return v - (1 << 64) if v >= 1 << 63 else v


def test_x64_on_the_int8_range_is_the_int8_apply():
    w = W.batched(seed=21, M=3, N=50, K=512)
    for frac in (0, 3, 40):
        np.testing.assert_array_equal(oracle.gemv_x64(w["t"], w["d"], w["x"].astype(np.int64), frac),
                                      oracle.gemv_i8_frac(w["t"], w["d"], w["x"], frac))


@pytest.mark.parametrize("frac", [0, 1, 17, 62])
def test_x64_matches_numpy_wrapping_int64(frac):
    """numpy int64 matmul, products and sums wrap modulo 2^64, and >> on int64
    is the arithmetic shift: the same definition through other primitives."""
    rng = np.random.default_rng(frac)
    N, K, M = 23, 384, 4
    t = rng.integers(-1, 2, size=(N, K), dtype=np.int8)
    d = rng.integers(np.iinfo(np.int32).min, np.iinfo(np.int32).max, size=(N, K // 128),
                     dtype=np.int64).astype(np.int32)
    x = rng.integers(np.iinfo(np.int64).min, np.iinfo(np.int64).max, size=(M, K), dtype=np.int64)
    x[0, :7] = np.iinfo(np.int64).min
    x[1, :7] = np.iinfo(np.int64).max
    G = K // 128
    with np.errstate(over="ignore"):
        P = np.einsum("rgi,mgi->mrg", t.reshape(N, G, 128).astype(np.int64), x.reshape(M, G, 128))
        ref = ((P * d.astype(np.int64)[None]) >> frac).sum(axis=2)
    np.testing.assert_array_equal(oracle.gemv_x64(t, d, x, frac), ref)


def test_x64_is_the_base256_limb_sum_of_int8_applies():
    """The page's decomposition: with x = sum_l 256^l s_l (signed digits), the
    apply of x equals sum_l 256^l (apply of s_l) modulo 2^64 (frac = 0)."""
    rng = np.random.default_rng(5)
    N, K, M = 9, 256, 2
    t = rng.integers(-1, 2, size=(N, K), dtype=np.int8)
    d = rng.integers(-(1 << 31), 1 << 31, size=(N, K // 128), dtype=np.int64).astype(np.int32)
    x = rng.integers(np.iinfo(np.int64).min, np.iinfo(np.int64).max, size=(M, K), dtype=np.int64)
    digits = _signed_digits(x)
    limb = [oracle.gemv_i8(t, d, digits[l]) for l in range(8)]
    expect = np.array([[_wrap64(sum(int(limb[l][m, r]) << (8 * l) for l in range(8))) for r in range(N)]
                       for m in range(M)], dtype=np.int64)
    np.testing.assert_array_equal(oracle.gemv_x64(t, d, x), expect)


def test_x64_wraparound_closed_forms():
    N, K = 3, 128
    t = np.zeros((N, K), np.int8)
    d = np.ones((N, 1), np.int32)
    x = np.zeros((1, K), np.int64)
    # row 0: 128 lanes of +2^57 -> P = 2^64 = 0 (mod 2^64)
    t[0] = 1
    x[0, :] = 1 << 57
    # row 1: one lane -1 on x = INT64_MIN -> P = 2^63 = INT64_MIN (mod 2^64)
    t[1, 5] = -1
    x2 = x.copy()
    x2[0, 5] = np.iinfo(np.int64).min
    y = oracle.gemv_x64(t, d, x)
    assert y[0, 0] == 0
    y2 = oracle.gemv_x64(t, d, x2)
    assert y2[0, 1] == np.iinfo(np.int64).min
    # the floor acts on the wrapped product: P = 2^62, d = 2 -> -2^63, >> 1 -> -2^62
    t3 = np.zeros((1, K), np.int8)
    t3[0, 0] = 1
    x3 = np.zeros((1, K), np.int64)
    x3[0, 0] = 1 << 62
    assert oracle.gemv_x64(t3, np.full((1, 1), 2, np.int32), x3, 1)[0, 0] == -(1 << 62)


# ---------------------------------------------------------------------------
# Pure fractional-LNS reduction (BitState brief §5.2): approximate, so no
# end-to-end exact pin; its parts are pinned where the mathematics fixes them.
# ---------------------------------------------------------------------------

def _hp_log8(v, F):
    """round-free 8 log2(v) 2^F in 50-digit decimal arithmetic."""
    from decimal import Decimal, getcontext
    getcontext().prec = 50
    return Decimal(8) * (Decimal(v).ln() / Decimal(2).ln()) * (Decimal(2) ** F)


@pytest.mark.parametrize("F", [1, 2, 3, 4, 5, 6])
def test_lns_tables_are_the_rounded_closed_forms(F):
    from decimal import Decimal, getcontext
    getcontext().prec = 50
    log8, kp, km = oracle.lns_tables(F)
    one = Decimal(1)
    assert log8[1] == 0 and kp[0] == 8 << F and kp[-1] == 0 and km[-1] == 0
    for j in range(8):
        assert log8[1 << j] == 8 * j << F            # powers of two are exact
    for n in (3, 5, 7, 100, 127, 128):
        assert abs(Decimal(int(log8[n])) - _hp_log8(n, F)) <= Decimal("0.5")
    scale = Decimal(8) * (Decimal(2) ** F)
    for i in list(range(1, 40)) + list(range(40, len(kp), max(1, len(kp) // 50))):
        q = (-(Decimal(i) / scale) * Decimal(2).ln()).exp()     # 2^(-i / (8 2^F))
        assert abs(Decimal(int(kp[i])) - _hp_log8(one + q, F)) <= Decimal("0.5")
        assert abs(Decimal(int(km[i])) - _hp_log8(one - q, F)) <= Decimal("0.5")
    assert np.all(np.diff(kp) <= 0) and np.all(np.diff(km[1:]) >= 0) and np.all(km[1:] <= 0)


def _one_group(N, lanes):
    """LNS8 weights with the given (row, lane, trit) nonzeros in one 128-lane group."""
    t = np.zeros((N, 128), np.int8)
    for r, i, v in lanes:
        t[r, i] = v
    return t


@pytest.mark.parametrize("F", [1, 4, 6])
def test_purelns_exact_cases(F):
    xa = np.zeros(128, np.uint8)
    xa[3] = 90                 # +2^(16/8)
    xa[7] = 90                 # the same state
    xa[9] = 0x80 | 60          # -2^(-14/8)
    dcode = np.full((5, 1), 74, np.uint8)    # e = 0: k = a
    t = _one_group(5, [(0, 3, 1),                  # one lane: (+, 90) exactly
                       (1, 3, 1), (1, 7, 1),       # two lanes of one state: +8 codes exactly
                       (2, 3, 1), (2, 7, -1),      # a state whose population cancels: zero
                       (3, 9, 1),                  # one negative lane
                       (4, 3, -1), (4, 7, -1)])    # two negative lanes of one state
    s, lam, S = oracle.lns8_purelns(t, dcode, xa, F)
    assert (s[0], lam[0]) == (1, 90 << F)
    assert (s[1], lam[1]) == (1, 98 << F)
    assert (s[2], lam[2]) == (0, 0) and S[2] == 0.0
    assert (s[3], lam[3]) == (-1, 60 << F)
    assert (s[4], lam[4]) == (-1, 98 << F)
    assert S[0] == 4.0 and S[1] == 8.0          # 2^((90 - 74) / 8), doubled


def test_purelns_opposite_equal_buckets_cancel_across_groups():
    """The same magnitude with opposite signs in two groups meets in the group
    tree and cancels to exact zero."""
    xa = np.zeros(256, np.uint8)
    xa[5] = 100
    xa[128 + 5] = 100
    t = np.zeros((1, 256), np.int8)
    t[0, 5] = 1
    t[0, 128 + 5] = -1
    s, lam, S = oracle.lns8_purelns(t, np.full((1, 2), 74, np.uint8), xa, 3)
    assert s[0] == 0 and S[0] == 0.0


@pytest.mark.parametrize("F", [1, 2, 3, 4, 5, 6])
def test_purelns_error_bound_without_cancellation(F):
    """All terms positive: each table rounding moves L by at most 1/2 unit of
    2^-F codes and positive sums do not amplify it, so along any path to the
    root (one count fold, 4 band levels, log2(G) group levels, 3 phase levels)
    |log error| <= (depth + 1) / 2 * 2^-F codes."""
    N, K = 64, 1024
    w = W.lns8(seed=F, N=N, K=K)
    t = np.abs(w["t"])
    xa = w["xa"] & 0x7F
    s, lam, S = oracle.lns8_purelns(t, w["dcode"], xa, F)
    exact = oracle.lns8_materialise(oracle.lns8_direct(t, w["dcode"], xa))
    depth = 4 + int(np.log2(K // 128)) + 3
    bound = 2.0 ** ((depth + 1) * 0.5 * 2.0 ** -F / 8) - 1
    rel = np.abs(S / exact - 1)
    assert np.all(s == 1) and np.all(rel <= bound * (1 + 1e-12)), (float(rel.max()), bound)
