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
