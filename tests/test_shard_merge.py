"""Row sharding: shard boundaries and the exact merge of per-shard top-k lists.

CPU only. The per-shard lists come from the oracle's full-logit top-k over each
shard's rows; the merged result must equal the oracle's top-k over all rows.
The gather runs as two gloo ranks on 127.0.0.1.
"""

import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import oracle
import workloads as W
from bit_decode_gemv_gb300.shard import gather_merge_topk, merge_topk, shard_rows


def test_shard_rows_cover_exactly():
    for N in (0, 1, 7, 128, 1001):
        for world in (1, 2, 3, 8):
            blocks = [shard_rows(N, world, r) for r in range(world)]
            assert blocks[0][0] == 0 and blocks[-1][1] == N
            for (a, b), (c, d) in zip(blocks, blocks[1:]):
                assert b == c and a <= b
            sizes = [b - a for a, b in blocks]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard_rows(10, 2, 2)


def _shard_lists(logits, world, k):
    ids, scores = [], []
    for r in range(world):
        a, b = shard_rows(len(logits), world, r)
        kk = min(k, b - a)
        if kk == 0:
            ids.append(np.zeros(0, np.int64))
            scores.append(np.zeros(0, np.int64))
            continue
        i, s = oracle.topk(logits[a:b], kk)
        ids.append(np.asarray(i, np.int64) + a)
        scores.append(s)
    return ids, scores


@pytest.mark.parametrize("world", [1, 2, 3, 5])
def test_merge_equals_global_topk(world):
    w = W.lm_head(seed=11, N=900, K=256)
    logits = oracle.lmhead_logits(w["planes"], w["s"], w["x"])
    for k in (1, 7, 200):
        ids, scores = _shard_lists(logits, world, k)
        got_ids, got_scores = merge_topk(ids, scores, k)
        ref_ids, ref_scores = oracle.topk(logits, k)
        np.testing.assert_array_equal(got_ids, ref_ids)
        np.testing.assert_array_equal(got_scores, ref_scores)
        assert got_ids[0] == oracle.argmax(logits)


def test_merge_ties_across_shard_boundary():
    # equal scores everywhere: the global order is by index alone, across shards
    logits = np.full(50, 123, np.int64)
    logits[40] = 124
    ids, scores = _shard_lists(logits, 4, 5)
    got_ids, _ = merge_topk(ids, scores, 5)
    np.testing.assert_array_equal(got_ids, [40, 0, 1, 2, 3])


def test_merge_rejects_bad_lists():
    with pytest.raises(ValueError):
        merge_topk([np.array([1, 2])], [np.array([5, 5])], 3)
    with pytest.raises(ValueError):
        merge_topk([np.array([1]), np.array([1])], [np.array([5]), np.array([5])], 1)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, logits, k, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        a, b = shard_rows(len(logits), world, rank)
        ids, scores = oracle.topk(logits[a:b], min(k, b - a))
        got_ids, got_scores = gather_merge_topk(ids, scores, a, k)
        out[rank] = (got_ids.tolist(), got_scores.tolist())
    finally:
        dist.destroy_process_group()


def test_gloo_two_ranks():
    w = W.lm_head(seed=12, N=777, K=128)
    logits = oracle.lmhead_logits(w["planes"], w["s"], w["x"])
    k = 50
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, logits, k, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        ref_ids, ref_scores = oracle.topk(logits, k)
        for r in range(2):
            np.testing.assert_array_equal(out[r][0], ref_ids)
            np.testing.assert_array_equal(out[r][1], ref_scores)
