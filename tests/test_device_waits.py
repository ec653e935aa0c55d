"""The give-up path of the library's bounded device-side waits.

The tensor-memory batched GEMM hands work between warps through mbarriers;
every wait on one is bounded (layout field wait_limit, in SM clock cycles; 0 =
the default of 2^32). A wait that runs out sets the library's device error word,
the other warps stop at their next wait, the CTA lets the copies and MMAs it
started finish, frees its tensor memory and exits: the call's outputs are then
undefined, tg_device_error reports TG_ERR_DEVICE once, and the GPU stays usable.
This file makes the waits run out on purpose -- a limit of one cycle, so that
the first wait for a copy from memory gives up -- and checks exactly that:
nothing traps, nothing hangs, the error is reported once and cleared, and the
next call with the default limit is bit-exact against the oracle
(integer_engine.md §3.4: fail loud, never return a silently wrong result).
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


@pytest.mark.parametrize("N,K,M", [(32, 256, 17), (300, 1024, 64)])
def test_batched_wait_gives_up_reports_and_recovers(N, K, M):
    import torch
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import dev, gemv, pack_to_device
    w = W.batched(seed=N + M, M=M, N=N, K=K)
    wd, L = pack_to_device(tg.TG_TERNARY_I8, w["t"], w["d"])
    assert tg.tg_device_error() == tg.TG_OK           # nothing pending before
    short = tg.tg_layout.from_buffer_copy(L)
    short.wait_limit = 1
    y = torch.full((M, N), -7, dtype=torch.int64, device="cuda")
    tg.tg_gemv_i8(short, wd, dev(w["x"]), M, y)       # enqueues normally
    torch.cuda.synchronize()                          # and the kernel ends
    assert tg.tg_device_error() == tg.TG_ERR_DEVICE   # the give-up is reported
    assert tg.tg_device_error() == tg.TG_OK           # once: reading clears it
    np.testing.assert_array_equal(gemv(wd, L, w["x"]), oracle.gemv_i8(w["t"], w["d"], w["x"]))
    assert tg.tg_device_error() == tg.TG_OK           # the normal call reports nothing


def test_generous_limit_changes_nothing():
    """A limit far above what a wait needs gives the same exact result and no error."""
    import bit_decode_gemv_gb300 as tg
    from gpu_helpers import gemv, pack_to_device
    w = W.batched(seed=5, M=33, N=200, K=768)
    wd, L = pack_to_device(tg.TG_TERNARY_I8, w["t"], w["d"])
    L.wait_limit = 1 << 34
    np.testing.assert_array_equal(gemv(wd, L, w["x"]), oracle.gemv_i8(w["t"], w["d"], w["x"]))
    assert tg.tg_device_error() == tg.TG_OK
