"""Row sharding of the weight apply across ranks (one GPU per rank).

Every output row depends only on its own weight row, its scale and the shared
activation vector, so the rows of any of the three weight kinds can be split
into contiguous blocks, packed and applied independently, and the outputs
concatenated: nothing is exchanged on the data path.

The one exchange is the vocabulary-sharded lm_head selection. A row of the
global top-k is, within its own shard, among that shard's top-k under the same
total order (score descending, then row index ascending), because every row
that precedes it in the shard also precedes it globally. So the global top-k is
the top-k of the union of the per-shard lists, and the global argmax is the
first entry of it. Ranks exchange their k keys (one gather of world x k pairs)
and merge them on the host.

Host logic only: the per-shard top-k comes from tg_lmhead_argmax_topk on each
rank's GPU; this module never computes a score.
"""

from __future__ import annotations

import numpy as np


def shard_rows(N: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous row block [start, stop) of rank `rank` out of `world`.

    The first N % world ranks get one row more; blocks are in rank order and
    cover 0..N-1 exactly once. A rank may get an empty block when world > N.
    """
    if world < 1 or not 0 <= rank < world or N < 0:
        raise ValueError(f"bad shard request N={N} world={world} rank={rank}")
    base, extra = divmod(N, world)
    start = rank * base + min(rank, extra)
    stop = start + base + (1 if rank < extra else 0)
    return start, stop


def merge_topk(shard_ids, shard_scores, k: int):
    """Exact global top-k from per-shard top-k lists.

    shard_ids[j] holds GLOBAL row indices (shard offset already added) and
    shard_scores[j] their int64 scores, each list at least min(k, rows of
    shard j) long and holding that shard's top entries. Returns (ids, scores)
    of the first k rows under (score descending, index ascending), as int32 and
    int64 arrays; argmax is ids[0].
    """
    if k < 1:
        raise ValueError("k must be >= 1")
    ids = np.concatenate([np.asarray(a, dtype=np.int64).ravel() for a in shard_ids])
    scores = np.concatenate([np.asarray(a, dtype=np.int64).ravel() for a in shard_scores])
    if ids.shape != scores.shape:
        raise ValueError("ids and scores differ in length")
    if len(np.unique(ids)) != len(ids):
        raise ValueError("a row appears in more than one shard list")
    if len(ids) < k:
        raise ValueError(f"only {len(ids)} candidates for k={k}")
    # lexsort: last key is primary -> score descending, then index ascending
    order = np.lexsort((ids, -scores))[:k]
    return ids[order].astype(np.int32), scores[order]


def gather_merge_topk(local_ids, local_scores, row_offset: int, k: int, group=None):
    """Gather every rank's local top-k and merge them into the global top-k.

    local_ids are row indices within this rank's shard (as returned by the
    library), row_offset the shard's first global row. Uses one
    torch.distributed all_gather over the default (or given) process group;
    every rank returns the same (ids, scores).
    """
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    ids = np.asarray(local_ids, dtype=np.int64).ravel() + int(row_offset)
    scores = np.asarray(local_scores, dtype=np.int64).ravel()
    n = len(ids)
    sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
    dist.all_gather(sizes, torch.tensor([n], dtype=torch.int64), group=group)
    cap = int(max(int(s.item()) for s in sizes))
    pack = torch.zeros((2, cap), dtype=torch.int64)
    pack[0, :n] = torch.from_numpy(ids)
    pack[1, :n] = torch.from_numpy(scores)
    got = [torch.zeros((2, cap), dtype=torch.int64) for _ in range(world)]
    dist.all_gather(got, pack, group=group)
    all_ids = [g[0, : int(s.item())].numpy() for g, s in zip(got, sizes)]
    all_scores = [g[1, : int(s.item())].numpy() for g, s in zip(got, sizes)]
    return merge_topk(all_ids, all_scores, k)
