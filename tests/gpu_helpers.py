"""Device-side helpers for the GPU tests: upload inputs, call the C ABI through
the binding, bring results back. Argument marshalling only."""

import numpy as np
import torch

import bit_decode_gemv_gb300 as tg
from bit_decode_gemv_gb300 import build as tgbuild

_built = False


def ensure_built():
    global _built
    if not _built:
        tgbuild.build()
        _built = True


def dev(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def pack_to_device(kind, trits, scales):
    blob, L = tg.tg_pack_weights(kind, trits, scales)
    return dev(blob), L


def gemv(wd, L, x, stream=None) -> np.ndarray:
    x = np.atleast_2d(x)
    M = x.shape[0]
    xd = dev(x)
    y = torch.full((M, L.N), -7, dtype=torch.int64, device="cuda")
    tg.tg_gemv_i8(L, wd, xd, M, y, stream)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def lns8(wd, L, xa, with_S=True):
    xd = dev(xa)
    A = torch.full((L.N, 8), -7, dtype=torch.int64, device="cuda")
    S = torch.full((L.N,), float("nan"), dtype=torch.float64, device="cuda") if with_S else None
    tg.tg_gemv_lns8_phase(L, wd, xd, A, S)
    torch.cuda.synchronize()
    return A.cpu().numpy(), (S.cpu().numpy() if with_S else None)


def lmhead(wd, L, x, k, full):
    xd = dev(x)
    logits = torch.full((L.N,), -7, dtype=torch.int64, device="cuda") if full else None
    argmax = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    ids = torch.full((k,), -7, dtype=torch.int32, device="cuda")
    scores = torch.full((k,), -7, dtype=torch.int64, device="cuda")
    ncand = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    wsb = tg.tg_lmhead_workspace_bytes(L, k)
    ws = torch.full((wsb,), 0xAB, dtype=torch.uint8, device="cuda")
    tg.tg_lmhead_argmax_topk(L, wd, xd, k, logits, argmax, ids, scores, ncand, ws, wsb)
    torch.cuda.synchronize()
    return dict(logits=None if logits is None else logits.cpu().numpy(), argmax=int(argmax.item()),
                ids=ids.cpu().numpy(), scores=scores.cpu().numpy(), ncand=int(ncand.item()))


def oracle_by_row_slices(fn, t, d, *rest, threads=None):
    """An oracle GEMV over all rows, computed as contiguous row slices on
    concurrent threads (the oracle's C call releases the GIL) and concatenated
    along the output's row axis. Every row is still the oracle's own result; the
    split only spreads the work over the host's cores."""
    import concurrent.futures as cf
    import os
    N = t.shape[0]
    n = max(1, min(threads or os.cpu_count() or 1, N))
    cuts = [N * i // n for i in range(n + 1)]
    with cf.ThreadPoolExecutor(max_workers=n) as ex:
        parts = list(ex.map(lambda ab: fn(t[ab[0]:ab[1]], d[ab[0]:ab[1]], *rest), zip(cuts[:-1], cuts[1:])))
    return np.concatenate(parts, axis=-1)

