"""GPU parity of tg_gemv_lns8_phase against the CPU oracle, for both routes:
the direct per-lane route and the state-population route
(TG_FLAG_LNS8_STATE_SET).

A[r][p] must be bit-exact. S is compared within 1e-12 relative error, the
tolerance for the fp64 materialisation; the denominator is max(|S|, 2^-40 *
2^-9 sum_p |A[p]| F[p]) so that rows whose eight terms cancel to near zero
are measured against the size of the terms, not of the near-zero result.
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


ROUTES = ["direct", "stateset"]


def check(w, with_S=True, route="direct"):
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import lns8, pack_to_device
    wd, L = pack_to_device(tg.TG_TERNARY_LNS8, w["t"], w["dcode"])
    if route == "stateset":
        L.flags |= tg.TG_FLAG_LNS8_STATE_SET
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


@pytest.mark.parametrize("route", ROUTES)
def test_lns8_workload_full_size(route):
    check(W.lns8(), route=route)


@pytest.mark.parametrize("route", ROUTES)
def test_lns8_full_range_codes_full_size(route):
    """The bench's full-range row: codes uniform over 1..127, so most (row, group)
    pairs of N = K = 4096 have lanes that clamp at scale codes 60..88."""
    w = W.lns8()
    w["xa"] = W.lns8_activations_full_range(0, 4096)
    check(w, route=route)


def wide(seed, N, K):
    """Codes over 0..127 and scale codes over the whole byte range, so that both
    clamps (k <= 0 and k > 127) and signed zeros occur often."""
    w = W.lns8(seed=seed, N=N, K=K)
    rng = np.random.default_rng(seed)
    w["xa"] = rng.integers(0, 256, size=K, dtype=np.uint8)
    w["dcode"] = rng.integers(0, 256, size=w["dcode"].shape, dtype=np.uint8)
    return w


@pytest.mark.parametrize("route", ROUTES)
@pytest.mark.parametrize("N,K", [(1, 128), (33, 128), (95, 384), (1000, 4096), (40, 12800)])
def test_clamp_heavy_and_ragged(N, K, route):
    check(wide(N, N, K), route=route)


@pytest.mark.parametrize("route", ROUTES)
def test_extreme_codes(route):
    N, K = 64, 256
    t = np.ones((N, K), np.int8)
    t[1::2] = -1
    xa = np.full(K, 127, np.uint8)
    xa[::3] = 0x80 | 127
    dcode = np.full((N, 2), 255, np.uint8)
    dcode[::4] = 0
    dcode[1::4] = 74
    A, _ = check(dict(t=t, dcode=dcode, xa=xa), route=route)
    # scale code 255 saturates every product to code 127 = phase 7, band 15
    assert np.count_nonzero(A[2, :7]) == 0 and abs(A[2, 7]) > 0


@pytest.mark.parametrize("route", ROUTES)
def test_without_S(route):
    check(W.lns8(seed=3, N=77, K=512), with_S=False, route=route)


@pytest.mark.parametrize("route", ROUTES)
@pytest.mark.parametrize("n_states", [1, 2, 8, 32, 127])
def test_state_cardinality(n_states, route):
    """Activations drawn from a set of n_states codes: every state has many
    lanes when the set is small, one lane each when it is large."""
    w = W.lns8(seed=n_states, N=300, K=2048)
    w["xa"] = W.lns8_activations_states(n_states, 2048, n_states)
    check(w, route=route)


@pytest.mark.parametrize("route", ROUTES)
@pytest.mark.parametrize("zero_frac", [0.0, 0.9, 1.0])
def test_weight_zero_density(zero_frac, route):
    w = W.lns8(seed=5, N=130, K=1024)
    w["t"] = W.trits_sparse(5, (130, 1024), zero_frac)
    check(w, route=route)


@pytest.mark.parametrize("route", ROUTES)
def test_all_activations_zero(route):
    """Every activation code 0 (with both signs): no state is active, A = 0."""
    w = W.lns8(seed=9, N=70, K=256)
    w["xa"] = np.where(np.arange(256) % 2 == 0, 0x80, 0x00).astype(np.uint8)
    A, S = check(w, route=route)
    assert not A.any() and not S.any()


@pytest.mark.parametrize("route", ROUTES)
def test_one_state_saturates_or_vanishes(route):
    """One active code per group and scale codes at both ends, so that in each
    (row, group) the single state is either dropped (k <= 0), saturated
    (k > 127) or routed, on both sides of a 64-row tile boundary."""
    N, K = 130, 512
    rng = np.random.default_rng(11)
    t = rng.integers(-1, 2, size=(N, K), dtype=np.int8)
    xa = np.repeat(np.array([1, 127, 74, 0x80 | 60], np.uint8), 128)
    dcode = rng.choice(np.array([0, 1, 73, 74, 75, 128, 200, 255], np.uint8), size=(N, K // 128))
    check(dict(t=t, dcode=dcode, xa=xa), route=route)


@pytest.mark.parametrize("route", ROUTES)
def test_caller_phase_constants(route):
    """S with the caller's F (a device fp64 [8]): the built-in values passed in
    give S bit for bit equal to F = NULL; another table (signs, zeros, a scaled
    basis) gives 2^-9 sum_p A[p] F[p] in the order p = 0..7 with that table,
    which the oracle's materialisation computes with the same F."""
    import torch
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import dev, pack_to_device
    w = W.lns8(seed=21, N=700, K=1024)
    wd, L = pack_to_device(tg.TG_TERNARY_LNS8, w["t"], w["dcode"])
    if route == "stateset":
        L.flags |= tg.TG_FLAG_LNS8_STATE_SET
    xa = dev(w["xa"])
    A = torch.empty((L.N, 8), dtype=torch.int64, device="cuda")
    S0 = torch.empty((L.N,), dtype=torch.float64, device="cuda")
    tg.tg_gemv_lns8_phase(L, wd, xa, A, S0)
    A_ref = oracle.lns8_direct(w["t"], w["dcode"], w["xa"])
    for F in (oracle.lns8_F(), np.array([0.5, -1.0, 0.0, 3.0, 1e-3, -2.5, 7.0, 1.0 / 3.0])):
        S = torch.full((L.N,), float("nan"), dtype=torch.float64, device="cuda")
        tg.tg_gemv_lns8_phase(L, wd, xa, A, S, F=dev(np.asarray(F, np.float64)))
        torch.cuda.synchronize()
        np.testing.assert_array_equal(A.cpu().numpy(), A_ref)
        S_ref = oracle.lns8_materialise(A_ref, np.asarray(F, np.float64))
        np.testing.assert_array_equal(S.cpu().numpy(), S_ref)
    np.testing.assert_array_equal(S0.cpu().numpy(), oracle.lns8_materialise(A_ref))


def test_routes_agree_bitwise_on_the_workload():
    """The two routes return the same A and the same S bits on the workload."""
    w = W.lns8(seed=4, N=1024, K=4096)
    A0, S0 = check(w, route="direct")
    A1, S1 = check(w, route="stateset")
    np.testing.assert_array_equal(A0, A1)
    np.testing.assert_array_equal(S0.view(np.int64), S1.view(np.int64))



# ---------------------------------------------------------------------------
# Pure fractional-LNS route (TG_FLAG_LNS8_PURE_LNS): approximate by design, so
# the comparison is with the oracle's statement of the same reduction: sign
# and log magnitude bit-exact, S within the rounding of the final fp64 exp2.
# ---------------------------------------------------------------------------

def check_pure(w, F, with_S=True):
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import lns8, pack_to_device
    wd, L = pack_to_device(tg.TG_TERNARY_LNS8, w["t"], w["dcode"])
    L.flags |= tg.TG_FLAG_LNS8_PURE_LNS
    L.frac = F
    A, S = lns8(wd, L, w["xa"], with_S)
    s_ref, lam_ref, S_ref = oracle.lns8_purelns(w["t"], w["dcode"], w["xa"], F)
    np.testing.assert_array_equal(A[:, 0], s_ref)
    np.testing.assert_array_equal(A[:, 1], lam_ref)
    assert not A[:, 2:].any()
    if with_S:
        np.testing.assert_allclose(S, S_ref, rtol=1e-14, atol=0)
    return A, S


@pytest.mark.parametrize("F", [1, 2, 3, 4, 5, 6])
def test_purelns_workload_full_size(F):
    check_pure(W.lns8(), F)


@pytest.mark.parametrize("N,K", [(1, 128), (33, 384), (95, 4096), (40, 12800), (17, 32768)])
def test_purelns_shapes_and_clamps(N, K):
    """Ragged N; one group; more groups than lanes (a lane's run of groups,
    K = 12800 and 32768); codes and scale codes over the whole byte range."""
    check_pure(wide(N, N, K), 4)


@pytest.mark.parametrize("F", [2, 6])
@pytest.mark.parametrize("n_states", [1, 3, 127])
def test_purelns_state_cardinality(n_states, F):
    w = W.lns8(seed=n_states, N=130, K=2048)
    w["xa"] = W.lns8_activations_states(n_states, 2048, n_states)
    check_pure(w, F)


@pytest.mark.parametrize("F", [1, 4])
def test_purelns_full_bins(F):
    """Groups whose 128 lanes all fall into one product-code bin with one sign
    (population counts +128 and -128, the two ends of the count range), rows
    one lane short of that (127), and rows where every lane clamps into the
    top code."""
    N, K = 24, 512
    t = np.ones((N, K), np.int8)
    t[1::4] = -1                         # every lane negative
    t[2::4, ::128] = 0                   # one lane of each group zero
    xa = np.full(K, 74, np.uint8)        # one code, positive ...
    xa[256:] |= 0x80                     # ... and negative in groups 2 and 3
    dcode = np.full((N, K // 128), 74, np.uint8)
    dcode[3::4] = 200                    # 74 + 200 - 74 > 127: clamped
    check_pure(dict(t=t, dcode=dcode, xa=xa), F)


def test_purelns_zero_rows_and_without_S():
    w = W.lns8(seed=6, N=70, K=512)
    w["t"][::3] = 0
    A, _ = check_pure(w, 3, with_S=False)
    assert not A[::3].any()
    w["xa"] = np.where(np.arange(512) % 2 == 0, 0x80, 0x00).astype(np.uint8)
    A, S = check_pure(w, 5)
    assert not A.any() and not S.any()
