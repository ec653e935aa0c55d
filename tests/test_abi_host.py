"""Host-side checks of libtg.so that need no GPU.

The library must load and export every entry point include/tg.h declares; the
packer (pure host code) must write exactly the layout tg.h documents, checked
here by decoding it with an independent reader; and every argument error must
be reported before anything is enqueued. No test here launches a kernel.
"""

import ctypes as C
import os
import re

import numpy as np
import pytest

import bit_decode_gemv_gb300 as tg
from bit_decode_gemv_gb300 import build as tgbuild
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    tgbuild.build()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "tg.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tg_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol():
    names = declared_symbols()
    assert len(names) >= 9
    lib = C.CDLL(tg.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(tg.EXPORTS) == names


def test_status_strings():
    for code in range(-7, 1):
        s = tg.tg_status_string(code)
        assert s and s != "unknown status"
    assert tg.tg_status_string(-99) == "unknown status"


def test_layout_sizes():
    L = tg.tg_layout_init(tg.TG_TERNARY_I8, 6912, 2560)
    assert (L.tiles, L.G) == (216, 20)
    assert L.mask_bytes == 216 * 20 * 1024 and L.scale_bytes == 216 * 20 * 32 * 4
    assert L.scale_off % 256 == 0 and L.total_bytes % 256 == 0
    assert tg.tg_packed_bytes(tg.TG_TERNARY_I8, 6912, 2560) == L.total_bytes
    P = tg.tg_layout_init(tg.TG_PLANES8, 128256, 2560)
    assert P.mask_bytes == P.aux_bytes == 128256 * 2560
    assert P.scale_bytes == 128256 * 4 and P.aux2_bytes == 128256
    for off in (P.aux_off, P.scale_off, P.aux2_off):
        assert off % 256 == 0
    assert tg.tg_packed_bytes(tg.TG_TERNARY_I8, 10, 100) == 0
    for kind, N, K in ((tg.TG_TERNARY_I8, 0, 128), (tg.TG_TERNARY_I8, 4, 64), (tg.TG_PLANES8, 4, 200)):
        with pytest.raises(tg.TgError) as e:
            tg.tg_layout_init(kind, N, K)
        assert e.value.status == tg.TG_ERR_SHAPE
    with pytest.raises(tg.TgError) as e:
        tg.tg_layout_init(7, 4, 128)
    assert e.value.status == tg.TG_ERR_ARG


def decode_masked(blob, L, scale_dtype):
    """Independent reader of the tiled mask layout -> (t [N][K], scales [N][G])."""
    N, K, G, T = L.N, L.K, L.G, L.tiles
    m = blob[L.mask_off:L.mask_off + L.mask_bytes].reshape(T, G, 2, 32, 16)
    words = m.view("<u4").reshape(T, G, 2, 32, 4)                  # [T][G][h][row][u]
    t = np.zeros((T * 32, K), dtype=np.int8)
    for j in range(4):
        for b in range(4):
            sh = 8 * b + 2 * j
            nz = (words >> sh) & 1
            ng = (words >> (sh + 1)) & 1
            assert not (ng & ~nz).any(), "W_negative outside W_nonzero"
            val = nz.astype(np.int8) - 2 * ng.astype(np.int8)       # [T][G][h][row][u]
            # lane within group = 64h + 16u + 4j + b
            for h in range(2):
                for u in range(4):
                    lanes = np.arange(G) * 128 + 64 * h + 16 * u + 4 * j + b
                    t[:, lanes] = val[:, :, h, :, u].transpose(0, 2, 1).reshape(T * 32, G)
    s = blob[L.scale_off:L.scale_off + L.scale_bytes].view(scale_dtype).reshape(T, G, 32)
    scales = s.transpose(0, 2, 1).reshape(T * 32, G)
    return t, scales


@pytest.mark.parametrize("N,K", [(1, 128), (33, 256), (70, 640)])
def test_pack_i8_layout(N, K):
    w = W.tiny(seed=N, N=N, K=K)
    blob, L = tg.tg_pack_weights(tg.TG_TERNARY_I8, w["t"], w["d"])
    assert L.kind == tg.TG_TERNARY_I8 and L.max_abs_scale == int(np.abs(w["d"].astype(np.int64)).max())
    t, s = decode_masked(blob, L, "<i4")
    np.testing.assert_array_equal(t[:N], w["t"])
    np.testing.assert_array_equal(s[:N], w["d"])
    assert not t[N:].any() and not s[N:].any()          # padding rows are zero


def decode_q1(blob, L):
    """Independent reader of the Q1 layout -> (signs [N][K] in {-1,+1}, scales [N][G])."""
    N, K, G, T = L.N, L.K, L.G, L.tiles
    words = blob[L.mask_off:L.mask_off + L.mask_bytes].view("<u4").reshape(T, G, 32, 4)   # [T][G][row][u]
    sg = np.zeros((T * 32, K), dtype=np.int8)
    for j in range(8):
        for b in range(4):
            bit = ((words >> (8 * b + j)) & 1).astype(np.int8)        # [T][G][row][u]
            for u in range(4):
                lanes = np.arange(G) * 128 + 32 * u + 4 * j + b
                sg[:, lanes] = (2 * bit[:, :, :, u] - 1).transpose(0, 2, 1).reshape(T * 32, G)
    s = blob[L.scale_off:L.scale_off + L.scale_bytes].view("<i4").reshape(T, G, 32)
    return sg, s.transpose(0, 2, 1).reshape(T * 32, G)


@pytest.mark.parametrize("N,K", [(1, 128), (33, 256), (70, 640)])
def test_pack_q1_layout(N, K):
    rng = np.random.default_rng(N + K)
    signs = (2 * rng.integers(0, 2, size=(N, K)) - 1).astype(np.int8)
    d = rng.integers(-(1 << 20), 1 << 20, size=(N, K // 128)).astype(np.int32)
    blob, L = tg.tg_pack_weights(tg.TG_BINARY_Q1, signs, d)
    assert L.kind == tg.TG_BINARY_Q1 and L.frac == 0
    assert L.mask_bytes == L.tiles * L.G * 32 * 16          # one bit per weight
    assert L.max_abs_scale == int(np.abs(d.astype(np.int64)).max())
    sg, s = decode_q1(blob, L)
    np.testing.assert_array_equal(sg[:N], signs)
    np.testing.assert_array_equal(s[:N], d)
    assert not s[N:].any()
    with pytest.raises(tg.TgError) as e:                      # a zero is not a binary weight
        bad = signs.copy()
        bad[0, 0] = 0
        tg.tg_pack_weights(tg.TG_BINARY_Q1, bad, d)
    assert e.value.status == tg.TG_ERR_VALUE


def decode_lns8(blob, L):
    """Independent reader of the LNS8 fragment layout -> (t [16*tiles][K], codes)."""
    G, T, K = L.G, L.tiles, L.K
    words = blob[L.mask_off:L.mask_off + L.mask_bytes].view("<u4").reshape(T, G, 32, 4)
    t = np.zeros((T * 16, K), dtype=np.int8)
    for lane in range(32):
        q, j = lane >> 2, lane & 3
        for c in range(8):
            w = words[:, :, lane, c >> 1].astype(np.int64)            # [T][G]
            for r in range(4):
                row = q + (8 if r & 1 else 0)
                col = 16 * c + 2 * j + (8 if r & 2 else 0)
                rp = 4 * (c & 1) + r
                for h in range(2):
                    nz = (w >> (16 * h + 7 - rp)) & 1
                    ng = (w >> (16 * h + 15 - rp)) & 1
                    assert not (ng & ~nz).any()
                    val = (nz - 2 * ng).astype(np.int8)                  # [T][G]
                    for g in range(G):
                        t[np.arange(T) * 16 + row, g * 128 + col + h] = val[:, g]
    codes = blob[L.scale_off:L.scale_off + L.scale_bytes].reshape(T, G, 16).transpose(0, 2, 1).reshape(T * 16, G)
    return t, codes


def test_pack_lns8_layout():
    w = W.lns8(seed=1, N=45, K=384)
    blob, L = tg.tg_pack_weights(tg.TG_TERNARY_LNS8, w["t"], w["dcode"])
    assert L.tiles == 3 and L.mask_bytes == 3 * 3 * 512
    t, s = decode_lns8(blob, L)
    np.testing.assert_array_equal(t[:45], w["t"])
    np.testing.assert_array_equal(s[:45], w["dcode"])
    assert not t[45:].any() and not s[45:].any()


def test_pack_planes_layout():
    w = W.lm_head(seed=2, N=37, K=256)
    blob, L = tg.tg_pack_weights(tg.TG_PLANES8, w["planes"], w["s"])
    N, K = 37, 256
    # rows of 2K bytes: the row's planes 0-3 digits, then its planes 4-7 digits
    assert L.mask_off == 0 and L.aux_off == K and L.mask_bytes == L.aux_bytes == N * K
    assert L.scale_off >= 2 * N * K and L.scale_off % 256 == 0
    rows = blob[:2 * N * K].view(np.int8).reshape(N, 2 * K).astype(np.int64)
    hi, lo = rows[:, :K], rows[:, K:]
    pw = np.array([3 ** (7 - p) for p in range(8)], dtype=np.int64)
    Wint = np.tensordot(pw, w["planes"].astype(np.int64), axes=(0, 0))
    np.testing.assert_array_equal(81 * hi + lo, Wint)
    assert np.abs(hi).max() <= 40 and np.abs(lo).max() <= 40
    np.testing.assert_array_equal(blob[L.scale_off:L.scale_off + 4 * N].view("<i4"), w["s"])
    m = blob[L.aux2_off:L.aux2_off + N]
    np.testing.assert_array_equal(m, np.abs(lo).max(axis=1))
    exact = ~w["planes"][1:].any(axis=(0, 2))
    assert (m[exact] == 0).all()


def test_pack_rejects_bad_values():
    t = np.zeros((4, 128), np.int8)
    t[2, 5] = 2
    with pytest.raises(tg.TgError) as e:
        tg.tg_pack_weights(tg.TG_TERNARY_I8, t, np.ones((4, 1), np.int32))
    assert e.value.status == tg.TG_ERR_VALUE
    planes = np.zeros((8, 3, 128), np.int8)
    with pytest.raises(tg.TgError) as e:
        tg.tg_pack_weights(tg.TG_PLANES8, planes, np.array([1, 0, 1], np.int32))
    assert e.value.status == tg.TG_ERR_VALUE
    planes[7, 1, 3] = -2
    with pytest.raises(tg.TgError) as e:
        tg.tg_pack_weights(tg.TG_PLANES8, planes, np.array([1, 1, 1], np.int32))
    assert e.value.status == tg.TG_ERR_VALUE


def test_pack_deterministic_across_calls():
    w = W.ffn_up(seed=3, N=300, K=512)
    a, _ = tg.tg_pack_weights(tg.TG_TERNARY_I8, w["t"], w["d"])
    b, _ = tg.tg_pack_weights(tg.TG_TERNARY_I8, w["t"], w["d"])
    np.testing.assert_array_equal(a, b)


# Argument errors are all detected on the host, before any CUDA call; fake but
# well-aligned addresses are enough to reach each check.
A256 = 1 << 20


def status_of(fn, *args):
    with pytest.raises(tg.TgError) as e:
        fn(*args)
    return e.value.status


def test_gemv_argument_errors():
    w = W.tiny(seed=0, N=8, K=256)
    _, L = tg.tg_pack_weights(tg.TG_TERNARY_I8, w["t"], w["d"])
    f = tg.tg_gemv_i8
    assert status_of(f, L, None, A256, 1, A256, 0) == tg.TG_ERR_ARG
    assert status_of(f, L, A256 + 16, A256, 1, A256, 0) == tg.TG_ERR_ARG      # w not 256-aligned
    assert status_of(f, L, A256, A256 + 1, 1, A256, 0) == tg.TG_ERR_ARG       # x not 16-aligned
    assert status_of(f, L, A256, A256, 1, A256 + 4, 0) == tg.TG_ERR_ARG       # y not 8-aligned
    assert status_of(f, L, A256, A256, 0, A256, 0) == tg.TG_ERR_SHAPE
    assert status_of(f, L, A256, A256, 65, A256, 0) == tg.TG_ERR_SHAPE
    bad = tg.tg_layout.from_buffer_copy(L)
    bad.kind = tg.TG_PLANES8
    assert status_of(f, bad, A256, A256, 1, A256, 0) == tg.TG_ERR_ARG
    big = tg.tg_layout.from_buffer_copy(L)
    big.G, big.K, big.max_abs_scale = 1 << 20, 128 << 20, (1 << 31) - 1
    assert status_of(f, big, A256, A256, 1, A256, 0) == tg.TG_ERR_BOUND
    for frac in (-1, 63):                                                     # floor shift out of range
        fr = tg.tg_layout.from_buffer_copy(L)
        fr.frac = frac
        assert status_of(f, fr, A256, A256, 1, A256, 0) == tg.TG_ERR_ARG
    neg = tg.tg_layout.from_buffer_copy(L)
    neg.wait_limit = -1                                                       # a wait bound below zero
    assert status_of(f, neg, A256, A256, 17, A256, 0) == tg.TG_ERR_ARG


def test_lns8_argument_errors():
    w = W.lns8(seed=0, N=8, K=256)
    _, L = tg.tg_pack_weights(tg.TG_TERNARY_LNS8, w["t"], w["dcode"])
    f = tg.tg_gemv_lns8_phase
    assert status_of(f, L, A256, A256, None, None, 0) == tg.TG_ERR_ARG
    assert status_of(f, L, A256, A256 + 8, A256, None, 0) == tg.TG_ERR_ARG
    assert status_of(f, L, A256, A256, A256, A256 + 3, 0) == tg.TG_ERR_ARG
    big = tg.tg_layout.from_buffer_copy(L)
    big.K, big.G = 65536, 512
    assert status_of(f, big, A256, A256, A256, None, 0) == tg.TG_ERR_BOUND
    fr = tg.tg_layout.from_buffer_copy(L)
    fr.frac = 3                                                                # no floor for LNS8
    assert status_of(f, fr, A256, A256, A256, None, 0) == tg.TG_ERR_ARG
    # the pure-LNS route takes frac = 1..6 as its internal precision, and not
    # together with the state-set route
    for frac in (0, 7, -1):
        pl = tg.tg_layout.from_buffer_copy(L)
        pl.flags = tg.TG_FLAG_LNS8_PURE_LNS
        pl.frac = frac
        assert status_of(f, pl, A256, A256, A256, None, 0) == tg.TG_ERR_ARG
    both = tg.tg_layout.from_buffer_copy(L)
    both.flags = tg.TG_FLAG_LNS8_PURE_LNS | tg.TG_FLAG_LNS8_STATE_SET
    both.frac = 3
    assert status_of(f, both, A256, A256, A256, None, 0) == tg.TG_ERR_ARG
    # the caller's phase constants F: 8-byte aligned, and not with the pure route
    assert status_of(f, L, A256, A256, A256, None, 0, A256 + 4) == tg.TG_ERR_ARG
    pl = tg.tg_layout.from_buffer_copy(L)
    pl.flags = tg.TG_FLAG_LNS8_PURE_LNS
    pl.frac = 4
    assert status_of(f, pl, A256, A256, A256, None, 0, A256) == tg.TG_ERR_ARG


def test_lmhead_argument_errors():
    w = W.lm_head(seed=0, N=64, K=256)
    _, L = tg.tg_pack_weights(tg.TG_PLANES8, w["planes"], w["s"])
    wsb = tg.tg_lmhead_workspace_bytes(L, 10)
    assert wsb >= 64 * 16
    f = tg.tg_lmhead_argmax_topk
    ok = dict(w=A256, x=A256, k=10, logits=None, argmax=A256, ids=A256, scores=A256, ncand=None,
              ws=A256, ws_bytes=wsb)

    def call(**kw):
        a = dict(ok, **kw)
        return status_of(f, L, a["w"], a["x"], a["k"], a["logits"], a["argmax"], a["ids"],
                         a["scores"], a["ncand"], a["ws"], a["ws_bytes"], 0)

    assert call(argmax=None) == tg.TG_ERR_ARG
    assert call(scores=A256 + 4) == tg.TG_ERR_ARG
    assert call(k=0) == tg.TG_ERR_SHAPE
    assert call(k=65) == tg.TG_ERR_SHAPE
    assert call(ws=None) == tg.TG_ERR_WORKSPACE
    assert call(ws_bytes=wsb - 1) == tg.TG_ERR_WORKSPACE
    assert call(ws=A256 + 64) == tg.TG_ERR_WORKSPACE
    big = tg.tg_layout.from_buffer_copy(L)
    big.max_abs_scale = 1 << 31
    assert status_of(f, big, A256, A256, 10, None, A256, A256, A256, None, A256, wsb, 0) == tg.TG_ERR_BOUND
    assert tg.tg_lmhead_workspace_bytes(tg.tg_layout_init(tg.TG_TERNARY_I8, 8, 128), 4) == 0


def test_noalloc_checks_arguments_before_the_scratch_size():
    """tg_lmhead_argmax_topk_noalloc reports the same argument and shape errors as
    the workspace-taking call, in the same order, whatever the problem size: a
    problem too large for the fixed scratch is only refused (TG_ERR_WORKSPACE)
    once its other arguments are valid. Every case returns before any CUDA call."""
    f = tg.tg_lmhead_argmax_topk_noalloc
    L = tg.tg_layout_init(tg.TG_PLANES8, 300000, 128)     # workspace far above the scratch
    L.max_abs_scale = 1
    assert tg.tg_lmhead_workspace_bytes(L, 10) > tg.TG_NOALLOC_SCRATCH_BYTES

    def call(layout=L, w=A256, x=A256, k=10, logits=None, argmax=A256, ids=A256, scores=A256, ncand=None):
        return status_of(f, layout, w, x, k, logits, argmax, ids, scores, ncand, 0)

    assert call() == tg.TG_ERR_WORKSPACE
    assert call(argmax=None) == tg.TG_ERR_ARG
    assert call(w=None) == tg.TG_ERR_ARG
    assert call(x=A256 + 8) == tg.TG_ERR_ARG
    assert call(scores=A256 + 4) == tg.TG_ERR_ARG
    assert call(k=0) == tg.TG_ERR_SHAPE
    assert call(k=tg.TG_MAX_K + 1) == tg.TG_ERR_SHAPE
    small = tg.tg_layout_init(tg.TG_PLANES8, 8, 128)
    small.max_abs_scale = 1
    assert call(layout=small, k=9) == tg.TG_ERR_SHAPE               # k > N
    wrong = tg.tg_layout_init(tg.TG_TERNARY_I8, 300000, 128)
    assert call(layout=wrong) == tg.TG_ERR_ARG
    # the scratch's exact limit: N = 259008 rows fit, one more row does not
    edge = tg.tg_layout_init(tg.TG_PLANES8, 259008, 128)
    assert tg.tg_lmhead_workspace_bytes(edge, 10) == tg.TG_NOALLOC_SCRATCH_BYTES
    edge.N = 259009
    assert tg.tg_lmhead_workspace_bytes(edge, 10) > tg.TG_NOALLOC_SCRATCH_BYTES
    edge.max_abs_scale = 1
    assert call(layout=edge) == tg.TG_ERR_WORKSPACE


def test_layout_flags_are_distinct_bits():
    import bit_decode_gemv_gb300 as tg
    flags = [tg.TG_FLAG_CONST_WEIGHTS, tg.TG_FLAG_LNS8_STATE_SET, tg.TG_FLAG_X_INT64, tg.TG_FLAG_LNS8_PURE_LNS]
    assert all(f & (f - 1) == 0 for f in flags)
    assert len(set(flags)) == len(flags) and sum(flags) == (flags[0] | flags[1] | flags[2] | flags[3])


@pytest.mark.parametrize("M,K", [(2, 17920), (1, 23808)])
def test_int64_activations_k_limit(M, K):
    """Eight digit planes must fit the staging area: K = 17920 with several
    tokens and K = 23808 with one are TG_ERR_SHAPE before any device query or
    launch (17792 and 23680 run in the GPU tests' range)."""
    import bit_decode_gemv_gb300 as tg
    _, L = tg.tg_pack_weights(tg.TG_TERNARY_I8, np.zeros((1, K), np.int8), np.ones((1, K // 128), np.int32))
    L.flags |= tg.TG_FLAG_X_INT64
    assert status_of(tg.tg_gemv_i8, L, A256, A256, M, A256, 0) == tg.TG_ERR_SHAPE


def test_compiled_and_ctypes_call_paths_agree():
    """tg_gemv_i8 has two marshalling paths (the compiled module when it was built,
    ctypes otherwise): both must pass the same arguments to the library, so every
    argument error comes back with the same status."""
    import ctypes as C
    f = tg._fast()
    if f is None:
        pytest.skip("the compiled call path was not built")
    w = W.tiny(seed=3, N=64, K=256)
    blob, L = tg.tg_pack_weights(tg.TG_TERNARY_I8, w["t"], w["d"])
    lib = tg.lib()
    cases = [(0, 0, 0, 1, 0, 0), (C.addressof(L), 0, 0, 1, 0, 0), (C.addressof(L), 256, 16, 0, 8, 0),
             (C.addressof(L), 256, 16, tg.TG_MAX_M + 1, 8, 0), (C.addressof(L), 257, 16, 1, 8, 0),
             (C.addressof(L), 256, 15, 1, 8, 0)]
    for args in cases:
        lp = C.cast(args[0], C.POINTER(tg.tg_layout)) if args[0] else None
        assert f.gemv_i8(*args) == lib.tg_gemv_i8(lp, *args[1:]), args
