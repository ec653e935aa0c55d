"""GPU parity of tg_lmhead_argmax_topk against the CPU oracle.

Every output is an integer and must match bit-exactly: the logits (full path),
the argmax, and the top-k ids and scores in (score desc, index asc) order, for
both the full 8-plane path and the two-stage path.
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


def check(planes, s, x, k, logits_ref=None):
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import lmhead, pack_to_device
    wd, L = pack_to_device(tg.TG_PLANES8, planes, s)
    if logits_ref is None:
        logits_ref = oracle.lmhead_logits(planes, s, x)
    ids_ref, top_ref = oracle.topk(logits_ref, k)
    am_ref = oracle.argmax(logits_ref)
    out = {}
    for full in (True, False):
        r = lmhead(wd, L, x, k, full)
        if full:
            np.testing.assert_array_equal(r["logits"], logits_ref)
        np.testing.assert_array_equal(r["ids"], ids_ref)
        np.testing.assert_array_equal(r["scores"], top_ref)
        assert r["argmax"] == am_ref
        assert k <= r["ncand"] <= L.N
        out["full" if full else "two_stage"] = r
    return out


def test_lm_head_workload_full_size():
    w = W.lm_head()
    out = check(w["planes"], w["s"], w["x"], w["k"])
    # the two-stage path reads planes 4-7 of only a fraction of the vocabulary
    assert out["two_stage"]["ncand"] < w["planes"].shape[1] // 4


@pytest.mark.parametrize("N,K,k", [(1000, 256, 20), (5000, 384, 1024), (64, 128, 1), (300, 128, 300),
                                   (2049, 8192, 7), (3333, 2560, 200)])
def test_shapes(N, K, k):
    w = W.lm_head(seed=N, N=N, K=K)
    check(w["planes"], w["s"], w["x"], k)


def test_ties_resolve_to_lowest_index():
    w = W.lm_head(seed=4, N=700, K=256)
    planes, s = w["planes"].copy(), w["s"].copy()
    best = int(np.argmax(oracle.lmhead_logits(planes, s, w["x"])))
    for dst in (3, 200, 699):
        planes[:, dst] = planes[:, best]
        s[dst] = s[best]
    out = check(planes, s, w["x"], 10)
    ids = out["full"]["ids"].tolist()
    lead = sorted({3, 200, 699, best})
    assert ids[:len(lead)] == lead and out["full"]["argmax"] == lead[0]


def test_all_rows_equal():
    w = W.lm_head(seed=5, N=300, K=128)
    planes = np.repeat(w["planes"][:, :1], 300, axis=1)
    s = np.full(300, 7, np.int32)
    out = check(planes, s, w["x"], 50)
    assert out["full"]["ids"].tolist() == list(range(50))


def test_only_exact_ternary_rows():
    w = W.lm_head(seed=6, N=4000, K=256)
    planes = w["planes"].copy()
    planes[1:] = 0
    check(planes, w["s"], w["x"], 64)


def test_row_shards_merge_to_global_topk():
    """Vocabulary split into three independently packed row shards: each shard's
    two-stage top-k on the GPU, merged on the host, equals the global top-k."""
    import bit_decode_gemv_gb300 as tg
    from bit_decode_gemv_gb300.shard import merge_topk, shard_rows
    from gpu_helpers import lmhead, pack_to_device
    w = W.lm_head(seed=21, N=6000, K=512)
    k = 64
    logits_ref = oracle.lmhead_logits(w["planes"], w["s"], w["x"])
    ids, scores = [], []
    for r in range(3):
        a, b = shard_rows(w["planes"].shape[1], 3, r)
        wd, L = pack_to_device(tg.TG_PLANES8, np.ascontiguousarray(w["planes"][:, a:b]), w["s"][a:b])
        out = lmhead(wd, L, w["x"], k, False)
        ids.append(out["ids"].astype(np.int64) + a)
        scores.append(out["scores"])
    got_ids, got_scores = merge_topk(ids, scores, k)
    ref_ids, ref_scores = oracle.topk(logits_ref, k)
    np.testing.assert_array_equal(got_ids, ref_ids)
    np.testing.assert_array_equal(got_scores, ref_scores)
    assert got_ids[0] == oracle.argmax(logits_ref)


def test_back_to_back_calls_read_x_written_just_before():
    """Calls on one stream with no host synchronisation between them: before each
    call a device copy rewrites x, and every call reuses one workspace. The call's
    first kernel is a programmatic dependent of whatever precedes it, so it must
    wait for that copy; each result must be the one for the x just written."""
    import torch
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import dev, pack_to_device
    w = W.lm_head(seed=11, N=20000, K=2560)
    wd, L = pack_to_device(tg.TG_PLANES8, w["planes"], w["s"])
    k = 50
    xs = [W.lm_head(seed=20 + i, N=64, K=2560)["x"] for i in range(4)]
    src = [dev(x) for x in xs]
    xd = torch.empty_like(src[0])
    wsb = tg.tg_lmhead_workspace_bytes(L, k)
    ws = torch.full((wsb,), 0xAB, dtype=torch.uint8, device="cuda")
    calls = []
    for i in range(len(xs)):
        for full in (False, True):
            o = dict(logits=torch.full((L.N,), -7, dtype=torch.int64, device="cuda") if full else None,
                     argmax=torch.full((1,), -7, dtype=torch.int32, device="cuda"),
                     ids=torch.full((k,), -7, dtype=torch.int32, device="cuda"),
                     scores=torch.full((k,), -7, dtype=torch.int64, device="cuda"),
                     ncand=torch.full((1,), -7, dtype=torch.int32, device="cuda"))
            xd.copy_(src[i])
            tg.tg_lmhead_argmax_topk(L, wd, xd, k, o["logits"], o["argmax"], o["ids"], o["scores"], o["ncand"],
                                     ws, wsb)
            calls.append((i, full, o))
    torch.cuda.synchronize()
    for i, full, o in calls:
        logits_ref = oracle.lmhead_logits(w["planes"], w["s"], xs[i])
        ids_ref, top_ref = oracle.topk(logits_ref, k)
        if full:
            np.testing.assert_array_equal(o["logits"].cpu().numpy(), logits_ref)
        np.testing.assert_array_equal(o["ids"].cpu().numpy(), ids_ref)
        np.testing.assert_array_equal(o["scores"].cpu().numpy(), top_ref)
        assert int(o["argmax"].item()) == oracle.argmax(logits_ref)
