"""Guard bytes around every output buffer: each call writes its outputs into
the middle of a larger buffer whose guard regions hold a sentinel, on ragged
shapes (N not a multiple of any tile, the last tile partly padding); the
guards must come back untouched and the outputs must equal the oracle."""

import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 4096          # elements on each side
SENTINEL = -0x2545F4914F6CDD1D


@pytest.fixture(scope="module", autouse=True)
def built():
    from gpu_helpers import ensure_built
    ensure_built()


def guarded(n, dtype):
    import torch
    buf = torch.full((n + 2 * GUARD,), SENTINEL if dtype == torch.int64 else -7, dtype=dtype, device="cuda")
    return buf, buf[GUARD:GUARD + n]


def assert_guards(buf, n):
    import torch
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    fill = SENTINEL if buf.dtype == torch.int64 else -7
    assert np.all(b[:GUARD] == fill) and np.all(b[GUARD + n:] == fill), "a guard byte changed"


@pytest.mark.parametrize("kind", ["ternary", "q1", "x64"])
@pytest.mark.parametrize("M", [1, 3, 8, 64])
def test_gemv_outputs_stay_in_bounds(kind, M):
    import torch
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import dev, pack_to_device
    N, K = 97, 640
    if kind == "q1":
        w = W.ffn_up_q1(seed=M, N=N, K=K, M=M)
        wd, L = pack_to_device(tg.TG_BINARY_Q1, w["t"], w["d"])
    else:
        w = W.batched(seed=M, M=M, N=N, K=K)
        wd, L = pack_to_device(tg.TG_TERNARY_I8, w["t"], w["d"])
    x = w["x"]
    if kind == "x64":
        L.flags |= tg.TG_FLAG_X_INT64
        x = W.x_int64_full(M, (M, K))
    buf, y = guarded(M * N, torch.int64)
    tg.tg_gemv_i8(L, wd, dev(x), M, y)
    assert_guards(buf, M * N)
    ref = oracle.gemv_x64(w["t"], w["d"], x) if kind == "x64" else oracle.gemv_i8(w["t"], w["d"], x)
    np.testing.assert_array_equal(y.cpu().numpy().reshape(M, N), ref)


@pytest.mark.parametrize("route", ["direct", "stateset", "pure"])
def test_lns8_outputs_stay_in_bounds(route):
    import torch
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import dev, pack_to_device
    w = W.lns8(seed=7, N=133, K=640)
    wd, L = pack_to_device(tg.TG_TERNARY_LNS8, w["t"], w["dcode"])
    if route == "stateset":
        L.flags |= tg.TG_FLAG_LNS8_STATE_SET
    if route == "pure":
        L.flags |= tg.TG_FLAG_LNS8_PURE_LNS
        L.frac = 3
    bufA, A = guarded(L.N * 8, torch.int64)
    bufS, S = guarded(L.N, torch.float64)
    tg.tg_gemv_lns8_phase(L, wd, dev(w["xa"]), A, S)
    assert_guards(bufA, L.N * 8)
    assert_guards(bufS, L.N)
    if route == "pure":
        s, lam, _ = oracle.lns8_purelns(w["t"], w["dcode"], w["xa"], 3)
        got = A.cpu().numpy().reshape(L.N, 8)
        np.testing.assert_array_equal(got[:, 0], s)
        np.testing.assert_array_equal(got[:, 1], lam)
    else:
        np.testing.assert_array_equal(A.cpu().numpy().reshape(L.N, 8),
                                      oracle.lns8_direct(w["t"], w["dcode"], w["xa"]))


@pytest.mark.parametrize("full", [False, True])
def test_lmhead_outputs_stay_in_bounds(full):
    import torch
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import dev, pack_to_device
    w = W.lm_head(seed=3, N=3001, K=384)
    k = 37
    wd, L = pack_to_device(tg.TG_PLANES8, w["planes"], w["s"])
    bl, logits = guarded(L.N, torch.int64) if full else (None, None)
    ba, am = guarded(1, torch.int32)
    bi, ids = guarded(k, torch.int32)
    bs, sc = guarded(k, torch.int64)
    bn, nc = guarded(1, torch.int32)
    wsb = tg.tg_lmhead_workspace_bytes(L, k)
    ws = torch.empty((wsb,), dtype=torch.uint8, device="cuda")
    tg.tg_lmhead_argmax_topk(L, wd, dev(w["x"]), k, logits, am, ids, sc, nc, ws, wsb)
    for b, n in ((ba, 1), (bi, k), (bs, k), (bn, 1)) + (((bl, L.N),) if full else ()):
        assert_guards(b, n)
    ref = oracle.lmhead_logits(w["planes"], w["s"], w["x"])
    ids_ref, sc_ref = oracle.topk(ref, k)
    np.testing.assert_array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_array_equal(sc.cpu().numpy(), sc_ref)
    if full:
        np.testing.assert_array_equal(logits.cpu().numpy(), ref)
