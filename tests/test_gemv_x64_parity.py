"""GPU parity of tg_gemv_i8 with int64 fixed-point activations
(TG_FLAG_X_INT64; integer engine §4.4, exact modulo 2^64 as its §5 states)
against the CPU oracle: bit-exact int64 outputs, including wraparound."""

import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from gpu_helpers import ensure_built
    ensure_built()


def run_x64(kind, t_or_bits, d, x, frac=0):
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import gemv, pack_to_device
    wd, L = pack_to_device(kind, t_or_bits, d)
    L.flags |= tg.TG_FLAG_X_INT64
    L.frac = frac
    return gemv(wd, L, np.ascontiguousarray(np.atleast_2d(x), dtype=np.int64))


def check(t, d, x, frac=0):
    import bit_decode_gemv_gb300 as tg
    y = run_x64(tg.TG_TERNARY_I8, t, d, x, frac)
    np.testing.assert_array_equal(y, oracle.gemv_x64(t, d, x, frac))


def check_q1(t, d, x, frac=0):
    """Q1_0 weights (t in {-1, +1}); the oracle's definition takes them as trits."""
    import bit_decode_gemv_gb300 as tg
    y = run_x64(tg.TG_BINARY_Q1, t, d, x, frac)
    np.testing.assert_array_equal(y, oracle.gemv_x64(t, d, x, frac))


@pytest.mark.parametrize("M", [1, 2, 7, 64])
@pytest.mark.parametrize("N,K", [(97, 128), (40, 640), (33, 2560)])
def test_full_range_int64_wraps_like_the_oracle(N, K, M):
    w = W.batched(seed=N + K + M, M=M, N=N, K=K)
    check(w["t"], w["d"], W.x_int64_full(N * K + M, (M, K)))


@pytest.mark.parametrize("M", [1, 3])
@pytest.mark.parametrize("frac", [0, 5, 40])
@pytest.mark.parametrize("bits", [7, 15, 23, 31, 39, 47])
def test_fixed_point_magnitudes(bits, frac, M):
    """|x| < 2^bits: one plane for int8-range values, more as they grow (at one
    token: one pass of four planes up to 2^31, two beyond)."""
    w = W.batched(seed=bits, M=M, N=70, K=768)
    x = W.x_fixed64(bits, (M, 768), frac_bits=bits - 3)
    x = np.clip(x, -(1 << bits), (1 << bits) - 1)
    check(w["t"], w["d"], x, frac)


@pytest.mark.parametrize("K", [6144, 12800])
def test_one_token_two_and_four_groups_per_warp(K):
    """One token of int64 activations with two groups per warp (K up to 8192)
    and four (beyond), full range and Q.16, with the floor."""
    w = W.batched(seed=K, M=1, N=300, K=K)
    check(w["t"], w["d"], W.x_int64_full(K, (1, K)))
    check(w["t"], w["d"], W.x_fixed64(K, (1, K)), 11)


def test_one_token_groups_of_different_sizes():
    """One token whose groups need no plane (all zero), one pass and two passes,
    side by side, ternary and Q1_0, on more rows than two tiles per SM."""
    K = 1280
    w = W.batched(seed=91, M=1, N=10000, K=K)
    x = W.x_int64_full(91, (1, K))
    x[0, 0:128] = 0                                         # group 0: zeros
    x[0, 128:256] = np.clip(x[0, 128:256], -100, 100)      # group 1: one digit
    x[0, 256:384] >>= 40                                    # group 2: three digits
    check(w["t"], w["d"], x)
    check(w["t"], w["d"], x, 7)
    bits = (w["t"] > 0)
    t_pm = np.where(bits, 1, -1).astype(np.int8)
    check_q1(t_pm, w["d"], x, 3)


def test_ffn_up_shape_q16_activations():
    w = W.ffn_up()
    x = W.x_fixed64(1, (1, w["K"]), frac_bits=16)
    check(w["t"], w["d"], x)


def test_planes_change_from_chunk_to_chunk():
    """Tokens staged in several chunks (K = 5120 holds few tokens of eight
    planes), each chunk needing a different number of digit planes."""
    M, N, K = 20, 40, 5120
    w = W.batched(seed=3, M=M, N=N, K=K)
    x = W.x_fixed64(3, (M, K), frac_bits=4)          # small: a couple of planes
    x[4:8] = W.x_int64_full(4, (4, K))                # full range in one chunk
    x[12] = np.arange(K) - K // 2                     # int8 overflow by a little
    check(w["t"], w["d"], x)
    check(w["t"], w["d"], x, 9)


@pytest.mark.parametrize("M", [1, 5, 33])
def test_q1_weights(M):
    w = W.ffn_up_q1(seed=M, N=77, K=1024, M=M)
    check_q1(w["t"], w["d"], W.x_int64_full(M, (M, 1024)))
    check_q1(w["t"], w["d"], W.x_fixed64(M, (M, 1024), frac_bits=20), 13)


def test_extreme_values():
    N, K = 64, 256
    rng = np.random.default_rng(2)
    t = rng.integers(-1, 2, size=(N, K), dtype=np.int8)
    t[0] = 1
    t[1] = -1
    d = rng.integers(np.iinfo(np.int32).min, np.iinfo(np.int32).max, size=(N, K // 128),
                     dtype=np.int64).astype(np.int32)
    d[::4] = np.iinfo(np.int32).min
    d[1::4] = np.iinfo(np.int32).max
    x = np.zeros((4, K), np.int64)
    x[0] = np.iinfo(np.int64).min
    x[1] = np.iinfo(np.int64).max
    x[2, ::2] = np.iinfo(np.int64).min
    x[2, 1::2] = np.iinfo(np.int64).max
    x[3] = -1
    for frac in (0, 1, 62):
        check(t, d, x, frac)


def test_int8_range_values_equal_the_int8_call():
    """The same activations as int8 and as int64 give the same outputs."""
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import gemv, pack_to_device
    w = W.batched(seed=8, M=6, N=200, K=1280)
    y64 = run_x64(tg.TG_TERNARY_I8, w["t"], w["d"], w["x"].astype(np.int64))
    wd, L = pack_to_device(tg.TG_TERNARY_I8, w["t"], w["d"])
    np.testing.assert_array_equal(y64, gemv(wd, L, w["x"]))


@pytest.mark.parametrize("M", [1, 2])
def test_const_weights_back_to_back_int64(M):
    """Programmatic dependent launch on the int64 path: a torch kernel rewrites
    x between calls that all write the same y."""
    import torch
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import dev, pack_to_device
    N, K = 300, 1024
    cases = [W.batched(seed=300 + i, M=M, N=N, K=K) for i in range(3)]
    packed = []
    for w in cases:
        wd, L = pack_to_device(tg.TG_TERNARY_I8, w["t"], w["d"])
        L.flags |= tg.TG_FLAG_CONST_WEIGHTS | tg.TG_FLAG_X_INT64
        packed.append((wd, L))
    xs = [dev(W.x_fixed64(400 + i, (M, K), frac_bits=12)) for i in range(3)]
    x = torch.empty((M, K), dtype=torch.int64, device="cuda")
    y = torch.empty((M, N), dtype=torch.int64, device="cuda")
    outs = [torch.empty((M, N), dtype=torch.int64, device="cuda") for _ in range(3)]
    for i, (wd, L) in enumerate(packed):
        torch.add(xs[i], 0, out=x)
        tg.tg_gemv_i8(L, wd, x, M, y)
        outs[i].copy_(y)
    torch.cuda.synchronize()
    for i, w in enumerate(cases):
        np.testing.assert_array_equal(outs[i].cpu().numpy(), oracle.gemv_x64(w["t"], w["d"], xs[i].cpu().numpy()))


def test_largest_k():
    """K = 17792, the largest K whose eight digit planes of several tokens fit
    the staging area, and K = 23680, the largest for one token."""
    w = W.batched(seed=17, M=2, N=40, K=17792)
    check(w["t"], w["d"], W.x_int64_full(17, (2, 17792)))
    w = W.batched(seed=18, M=1, N=40, K=23680)
    check(w["t"], w["d"], W.x_int64_full(18, (1, 23680)))
