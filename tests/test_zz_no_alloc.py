"""The lm_head call for callers that cannot allocate device memory.

tg_lmhead_argmax_topk_noalloc exists for callers that cannot give the library a
workspace of their own (a plugin whose host framework owns all device memory, a
server whose memory is reserved by a cache pool, a loop that may not block in
cudaMalloc). It runs the same kernels on a fixed scratch array inside the
library. These tests call it through the C ABI and check that it returns exactly
what the workspace-taking call returns, on two calls in a row (the second call
finds the first call's data still in the shared scratch), and that a problem too
large for the scratch is refused before anything runs.

The file is named so that pytest collects it after every other test.
"""

import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from gpu_helpers import ensure_built
    ensure_built()


def run(tg, torch, L, wd, x, k, full, noalloc):
    xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    logits = torch.full((L.N,), -7, dtype=torch.int64, device="cuda") if full else None
    am = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    ids = torch.full((k,), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((k,), -7, dtype=torch.int64, device="cuda")
    nc = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    if noalloc:
        tg.tg_lmhead_argmax_topk_noalloc(L, wd, xd, k, logits, am, ids, sc, nc)
    else:
        wsb = tg.tg_lmhead_workspace_bytes(L, k)
        ws = torch.empty((wsb,), dtype=torch.uint8, device="cuda")
        tg.tg_lmhead_argmax_topk(L, wd, xd, k, logits, am, ids, sc, nc, ws, wsb)
    torch.cuda.synchronize()
    return dict(logits=None if logits is None else logits.cpu().numpy(), argmax=int(am.item()),
                ids=ids.cpu().numpy(), scores=sc.cpu().numpy(), ncand=int(nc.item()))


def test_noalloc_matches_workspace_call_twice_in_a_row():
    import torch
    import bit_decode_gemv_gb300 as tg
    w = W.lm_head(seed=11, N=60000, K=2560)
    blob, L = tg.tg_pack_weights(tg.TG_PLANES8, w["planes"], w["s"])
    assert tg.tg_lmhead_workspace_bytes(L, 200) <= tg.TG_NOALLOC_SCRATCH_BYTES
    wd = torch.from_numpy(blob).cuda()
    x_first = w["x"]
    x_second = W.x_normal40(12, (2560,))
    for x in (x_first, x_second):              # two calls in a row on the shared scratch
        for full in (False, True):
            got = run(tg, torch, L, wd, x, 200, full, noalloc=True)
            ref = run(tg, torch, L, wd, x, 200, full, noalloc=False)
            np.testing.assert_array_equal(got["ids"], ref["ids"])
            np.testing.assert_array_equal(got["scores"], ref["scores"])
            assert got["argmax"] == ref["argmax"] == int(ref["ids"][0])
            assert got["ncand"] == ref["ncand"]
            if full:
                np.testing.assert_array_equal(got["logits"], ref["logits"])


@pytest.mark.parametrize("rows", ["random", "all_equal"])
def test_noalloc_at_the_scratch_limit(rows):
    """The largest problem the fixed scratch holds: N = 259,008 rows, whose
    workspace is exactly TG_NOALLOC_SCRATCH_BYTES, so the per-row stage-1 sums and
    the candidate list reach the array's last byte. With every row equal, every
    row is a candidate and the candidate list is filled to its end. Both paths,
    two calls in a row, each compared with the workspace-taking call."""
    import torch
    import bit_decode_gemv_gb300 as tg
    N, K, k = 259008, 128, 16
    w = W.lm_head(seed=13, N=8 if rows == "all_equal" else N, K=K)
    if rows == "all_equal":
        w["planes"] = np.ascontiguousarray(np.broadcast_to(w["planes"][:, :1, :], (8, N, K)))
        w["s"] = np.full(N, int(w["s"][0]), np.int32)
    blob, L = tg.tg_pack_weights(tg.TG_PLANES8, w["planes"], w["s"])
    del w["planes"]
    assert tg.tg_lmhead_workspace_bytes(L, k) == tg.TG_NOALLOC_SCRATCH_BYTES
    wd = torch.from_numpy(blob).cuda()
    for x in (W.x_normal40(14, (K,)), W.x_normal40(15, (K,))):
        for full in (False, True):
            got = run(tg, torch, L, wd, x, k, full, noalloc=True)
            ref = run(tg, torch, L, wd, x, k, full, noalloc=False)
            np.testing.assert_array_equal(got["ids"], ref["ids"])
            np.testing.assert_array_equal(got["scores"], ref["scores"])
            assert got["argmax"] == ref["argmax"] == int(ref["ids"][0])
            assert got["ncand"] == ref["ncand"]
            if full:
                np.testing.assert_array_equal(got["logits"], ref["logits"])
            if rows == "all_equal":
                # equal scores: the lowest indices, in order (integer_engine.md §3.3)
                np.testing.assert_array_equal(got["ids"], np.arange(k))
                if not full:
                    assert got["ncand"] == N


def test_noalloc_refuses_problems_larger_than_the_scratch():
    import bit_decode_gemv_gb300 as tg
    L = tg.tg_layout_init(tg.TG_PLANES8, 300000, 128)
    L.max_abs_scale = 1
    assert tg.tg_lmhead_workspace_bytes(L, 10) > tg.TG_NOALLOC_SCRATCH_BYTES
    a = 1 << 20                                 # never dereferenced: refused first
    with pytest.raises(tg.TgError) as e:
        tg.tg_lmhead_argmax_topk_noalloc(L, a, a, 10, None, a, a, a, None)
    assert e.value.status == tg.TG_ERR_WORKSPACE
