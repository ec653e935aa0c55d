"""GPU parity of tg_gemv_i8 against the CPU oracle: bit-exact int64 outputs.

Sizes the oracle finishes in seconds span several tiles and a ragged tail;
the full-size workloads (ffn_up for batch 1, the batched M=64 case) run in the
launch configuration the bench times and are compared on every output (the
batched case's oracle runs as row slices on the host's cores).
"""

import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from gpu_helpers import ensure_built
    ensure_built()


def check(w, rows=None):
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import gemv, pack_to_device
    wd, L = pack_to_device(tg.TG_TERNARY_I8, w["t"], w["d"])
    y = gemv(wd, L, w["x"])
    if rows is None:
        ref = oracle.gemv_i8(w["t"], w["d"], w["x"])
        np.testing.assert_array_equal(y, ref)
    else:
        ref = oracle.gemv_i8(w["t"][rows], w["d"][rows], w["x"])
        np.testing.assert_array_equal(y[:, rows], ref)
    return y


def test_tiny_workload():
    check(W.tiny())


def test_ffn_up_workload_full_size():
    check(W.ffn_up())


@pytest.mark.parametrize("N,K", [(1, 128), (31, 128), (33, 256), (100, 384), (257, 2560),
                                 (6913, 2560), (64, 6912), (40, 16384)])
def test_ragged_shapes(N, K):
    check(W.ffn_up(seed=N + K, N=N, K=K))


def test_extreme_values():
    N, K = 70, 1024
    t = -np.ones((N, K), np.int8)
    d = np.full((N, K // 128), np.iinfo(np.int32).min, np.int32)
    d[::2] = np.iinfo(np.int32).max
    x = np.full((1, K), -128, np.int8)
    y = check(dict(t=t, d=d, x=x))
    assert y[0, 0] == (K // 128) * 128 * 128 * np.iinfo(np.int32).max
    # mixed signs, zero rows, a single nonzero lane
    w = W.tiny(seed=1, N=N, K=K)
    w["t"][5] = 0
    w["x"][:] = 0
    w["x"][0, 777] = -128
    check(w)


@pytest.mark.parametrize("M", [2, 7, 16, 17, 33, 64])
def test_small_batch(M):
    check(W.batched(seed=M, M=M, N=97, K=640))


def test_batched_workload_full_size_every_row():
    """The batched workload (M = 64, N = 13824, K = 5120) in the launch the bench
    times, every one of its 884,736 outputs against the oracle (computed as row
    slices on the host's cores)."""
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import gemv, oracle_by_row_slices, pack_to_device
    w = W.batched()
    wd, L = pack_to_device(tg.TG_TERNARY_I8, w["t"], w["d"])
    y = gemv(wd, L, w["x"])
    np.testing.assert_array_equal(y, oracle_by_row_slices(oracle.gemv_i8, w["t"], w["d"], w["x"]))


def test_deterministic_and_shard_invariant():
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import gemv, pack_to_device
    w = W.ffn_up(seed=5, N=1000, K=2560)
    wd, L = pack_to_device(tg.TG_TERNARY_I8, w["t"], w["d"])
    y1 = gemv(wd, L, w["x"])
    y2 = gemv(wd, L, w["x"])
    np.testing.assert_array_equal(y1, y2)
    # rows split into two independently packed shards give the same outputs
    parts = []
    for sl in (slice(0, 413), slice(413, 1000)):
        wd_s, L_s = pack_to_device(tg.TG_TERNARY_I8, w["t"][sl], w["d"][sl])
        parts.append(gemv(wd_s, L_s, w["x"]))
    np.testing.assert_array_equal(np.concatenate(parts, axis=1), y1)


def test_output_untouched_on_argument_error():
    import torch
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import dev, pack_to_device
    w = W.tiny(seed=2, N=64, K=256)
    wd, L = pack_to_device(tg.TG_TERNARY_I8, w["t"], w["d"])
    y = torch.full((1, 64), 12345, dtype=torch.int64, device="cuda")
    with pytest.raises(tg.TgError):
        tg.tg_gemv_i8(L, wd, dev(w["x"]), 0, y)
    torch.cuda.synchronize()
    assert (y == 12345).all()


@pytest.mark.parametrize("N,K", [(6912, 2560), (1000, 6912)])
@pytest.mark.parametrize("M", [1, 3, 8, 12])
def test_const_weights_back_to_back(N, K, M):
    # With TG_FLAG_CONST_WEIGHTS a call with up to 16 tokens may start streaming
    # its weights while the previous kernel runs; x and y must still be ordered
    # after it. Several calls in a row on one stream: each on other weights, all
    # writing the same y, with x rewritten by a torch kernel between some of them.
    import torch
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import dev, pack_to_device
    cases = [W.ffn_up(seed=100 + i, N=N, K=K) for i in range(4)]
    packed = []
    for w in cases:
        wd, L = pack_to_device(tg.TG_TERNARY_I8, w["t"], w["d"])
        L.flags |= tg.TG_FLAG_CONST_WEIGHTS
        packed.append((wd, L))
    xs = [dev(W.x_normal40(200 + i, (M, K))) for i in range(4)]
    x = torch.empty((M, K), dtype=torch.int8, device="cuda")
    y = torch.empty((M, N), dtype=torch.int64, device="cuda")
    outs = [torch.empty((M, N), dtype=torch.int64, device="cuda") for _ in range(8)]
    for rep in range(2):
        for i, (wd, L) in enumerate(packed):
            torch.add(xs[(i + rep) % 4], 0, out=x)          # a kernel writes x
            tg.tg_gemv_i8(L, wd, x, M, y)
            tg.tg_gemv_i8(L, wd, x, M, y)                    # same y again, back to back
            outs[rep * 4 + i].copy_(y)
    torch.cuda.synchronize()
    for rep in range(2):
        for i, w in enumerate(cases):
            xi = xs[(i + rep) % 4].cpu().numpy()
            np.testing.assert_array_equal(outs[rep * 4 + i].cpu().numpy(), oracle.gemv_i8(w["t"], w["d"], xi))


@pytest.mark.parametrize("M", [2, 4, 5, 12, 31, 64])
def test_extreme_values_batched(M):
    """Largest group sums |P| = 2^14 and int32-extreme scales with several tokens."""
    N, K = 300, 1024
    rng = np.random.default_rng(5 + M)
    t = rng.integers(-1, 2, size=(N, K)).astype(np.int8)
    t[:50] = -1
    t[50:100] = 1
    d = rng.integers(np.iinfo(np.int32).min, np.iinfo(np.int32).max, size=(N, K // 128),
                     dtype=np.int64).astype(np.int32)
    d[::3] = np.iinfo(np.int32).max
    d[1::3] = np.iinfo(np.int32).min
    x = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    x[0] = -128
    x[-1] = 127
    check(dict(t=t, d=d, x=x))


@pytest.mark.parametrize("M", [2, 64])
def test_narrow_fold_at_its_bound(M):
    """Scales at |d| = 32767 (the largest the 32-bit block fold of the batched
    kernel accepts) with every group sum at |P| = 2^14: four groups of P * d sum
    to 4 * 2^14 * 32767, just inside int32, with both signs."""
    N, K = 160, 1024
    t = -np.ones((N, K), np.int8)
    t[N // 2:] = 1
    d = np.full((N, K // 128), 32767, np.int32)
    d[::3] = -32767
    d[1::7, 2] = 1
    x = np.full((M, K), -128, np.int8)
    x[M // 2:, ::2] = 127
    check(dict(t=t, d=d, x=x))


# ---------------------------------------------------------------------------
# Binary Q1_0 weights and the per-group floor (integer engine §4.1, §4.2)
# ---------------------------------------------------------------------------

def check_q1(w, frac=0, rows=None):
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import gemv, pack_to_device
    wd, L = pack_to_device(tg.TG_BINARY_Q1, w["t"], w["d"])
    L.frac = frac
    y = gemv(wd, L, w["x"])
    bits = (w["t"] > 0).astype(np.uint8)
    if rows is None:
        np.testing.assert_array_equal(y, oracle.gemv_q1(bits, w["d"], w["x"], frac))
    else:
        np.testing.assert_array_equal(y[:, rows], oracle.gemv_q1(bits[rows], w["d"][rows], w["x"], frac))


def check_frac(w, frac):
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import gemv, pack_to_device
    wd, L = pack_to_device(tg.TG_TERNARY_I8, w["t"], w["d"])
    L.frac = frac
    np.testing.assert_array_equal(gemv(wd, L, w["x"]), oracle.gemv_i8_frac(w["t"], w["d"], w["x"], frac))


def test_q1_ffn_up_full_size():
    check_q1(W.ffn_up_q1())


@pytest.mark.parametrize("N,K,M", [(1, 128, 1), (33, 256, 1), (257, 2560, 1), (40, 16384, 1),
                                   (97, 640, 2), (97, 640, 17), (300, 1024, 64)])
def test_q1_shapes(N, K, M):
    check_q1(W.ffn_up_q1(seed=N + K + M, N=N, K=K, M=M))


def test_q1_batched_full_size_every_row():
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import gemv, oracle_by_row_slices, pack_to_device
    w = W.ffn_up_q1(seed=5, N=13824, K=5120, M=64)
    w["x"] = W.x_uniform(5, (64, 5120))
    wd, L = pack_to_device(tg.TG_BINARY_Q1, w["t"], w["d"])
    bits = (w["t"] > 0).astype(np.uint8)
    np.testing.assert_array_equal(gemv(wd, L, w["x"]), oracle_by_row_slices(oracle.gemv_q1, bits, w["d"], w["x"]))


@pytest.mark.parametrize("M", [1, 2, 5, 12, 64])
@pytest.mark.parametrize("frac", [1, 7, 20])
def test_frac_ternary(M, frac):
    w = W.batched(seed=M + frac, M=M, N=300, K=1024)
    check_frac(w, frac)


@pytest.mark.parametrize("M", [1, 3, 8, 64])
@pytest.mark.parametrize("frac", [3, 15])
def test_frac_q1(M, frac):
    check_q1(W.ffn_up_q1(seed=7 * M + frac, N=200, K=768, M=M), frac)


@pytest.mark.parametrize("M", [1, 2, 5, 12, 64])
def test_extreme_values_q1_and_floor(M):
    """int32-extreme scales (the 64-bit fold), with and without the floor."""
    N, K = 160, 512
    rng = np.random.default_rng(11 + M)
    t = (2 * rng.integers(0, 2, size=(N, K)) - 1).astype(np.int8)
    t[:40] = -1
    d = rng.integers(np.iinfo(np.int32).min, np.iinfo(np.int32).max, size=(N, K // 128),
                     dtype=np.int64).astype(np.int32)
    d[::3] = np.iinfo(np.int32).max
    d[1::3] = np.iinfo(np.int32).min
    x = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    x[0] = -128
    for frac in (0, 1, 33, 62):
        check_q1(dict(t=t, d=d, x=x), frac)
    check_frac(dict(t=np.where(t > 0, 1, np.where(rng.random((N, K)) < 0.3, 0, -1)).astype(np.int8), d=d, x=x), 9)


# Token counts on both sides of every kernel boundary of tg_gemv_i8 (the
# few-token kernels up to 8 tokens on these row counts -- sums in registers up
# to 4, in shared memory above; two groups per warp up to K = 8192 and four
# above -- the warp-MMA kernel up to 16 when K <= 4096 and the activations'
# fragments fit, the tensor-memory kernel above), at K below and above those
# limits, ternary and Q1_0, with and without the floor.
@pytest.mark.parametrize("K", [640, 4608, 12800, 16384])
@pytest.mark.parametrize("M", [2, 3, 4, 5, 6, 7, 8, 9, 16, 17])
def test_every_token_count_path(M, K):
    N = 97 if K <= 4608 else 40
    check(W.batched(seed=M * K, M=M, N=N, K=K))
    check_frac(W.batched(seed=M * K + 1, M=M, N=N, K=K), 5)
    check_q1(W.ffn_up_q1(seed=M * K + 2, N=N, K=K, M=M))
    check_q1(W.ffn_up_q1(seed=M * K + 3, N=N, K=K, M=M), 11)


# One token on more 32-row tiles than twice the SM count (32000 rows: 1000
# tiles), the launch that reserves shared memory at the thread-limited CTA
# count, and on at most twice the SM count (the two-CTA cap), ternary and Q1_0.
@pytest.mark.parametrize("N", [32000, 4000])
def test_one_token_launch_plans(N):
    check(W.batched(seed=N, M=1, N=N, K=2560))
    check_q1(W.ffn_up_q1(seed=N + 1, N=N, K=2560, M=1), 2)


# The smallest shapes through every one-to-eight-token launch: one group (the
# half-tile kernel's second half-warp has no group), three groups (an odd
# pair), one row, a ragged last tile; ternary and Q1_0, with the floor.
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("N,K", [(1, 128), (31, 384), (33, 128), (65, 256)])
def test_smallest_shapes_every_token_count(M, N, K):
    check(W.batched(seed=N * K + M, M=M, N=N, K=K))
    check_frac(W.batched(seed=N * K + M + 1, M=M, N=N, K=K), 3)
    check_q1(W.ffn_up_q1(seed=N * K + M + 2, N=N, K=K, M=M), 2)


# One token with K > 4096 takes the half-tile kernel: one pair of groups per
# warp up to K = 8192, two up to K = 16384 (and four beyond, in
# test_few_tokens_wide_rows), ternary and Q1_0, with and without the floor.
@pytest.mark.parametrize("K", [5120, 8192, 12800])
def test_one_token_half_tiles(K):
    check(W.batched(seed=K, M=1, N=1000, K=K))
    check_frac(W.batched(seed=K + 1, M=1, N=333, K=K), 9)
    check_q1(W.ffn_up_q1(seed=K + 2, N=1000, K=K, M=1))
    check_q1(W.ffn_up_q1(seed=K + 3, N=333, K=K, M=1), 4)


# Seven and eight tokens on more tiles than SMs with K > 4096 (and more than
# twice as many with K <= 4096) go to the warp-MMA kernel; five and six stay on
# the few-token kernels.
@pytest.mark.parametrize("M", [5, 7, 8])
@pytest.mark.parametrize("N,K", [(5000, 4608), (10000, 1024)])
def test_seven_eight_tokens_on_many_tiles(M, N, K):
    check(W.batched(seed=M + N, M=M, N=N, K=K))
    check_q1(W.ffn_up_q1(seed=M + N + 1, N=N, K=K, M=M), 1)


# Two to four int8 tokens whose activations overflow the few-token kernel's
# shared memory (M * K bytes above about 200 KB) go to the dp4a kernel, which
# stages them in chunks; one token at the same K stays on the few-token kernel.
@pytest.mark.parametrize("M", [1, 2, 4])
def test_few_tokens_wide_rows(M):
    K = 65536
    check(W.batched(seed=M + 900, M=M, N=40, K=K))
    check_q1(W.ffn_up_q1(seed=M + 901, N=40, K=K, M=M), 3)


# The tensor-memory kernel gives a CTA one to four 32-row tiles, the fewest that
# still fit one wave on the device's SMs. On a 152-SM part these row counts take
# two, three and four tiles per CTA, each with a last CTA that owns fewer tiles;
# K = 1024 cycles the input ring (eight groups, six stages).
@pytest.mark.parametrize("N", [6939, 12807, 15043])
@pytest.mark.parametrize("M", [17, 64])
def test_tiles_per_cta(N, M):
    check(W.batched(seed=N + M, M=M, N=N, K=1024))
    if M == 64:
        check_frac(W.batched(seed=N + 1, M=M, N=N, K=1024), 6)
        check_q1(W.ffn_up_q1(seed=N + 2, N=N, K=1024, M=M))
