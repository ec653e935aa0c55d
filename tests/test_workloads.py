"""The seeded input generators (workloads.py): every generator runs, is
deterministic for a seed, and draws values in the ranges the input recipe
states. CPU only."""

import numpy as np

import workloads as W


def test_every_named_stream_draws():
    for name in W._STREAM_IDS:
        a = W._rng(3, name).integers(0, 1 << 30, size=4)
        b = W._rng(3, name).integers(0, 1 << 30, size=4)
        np.testing.assert_array_equal(a, b)
    ids = list(W._STREAM_IDS.values())
    assert len(set(ids)) == len(ids)


def test_lns8_activation_generators():
    for gen in (W.lns8_activations, W.lns8_activations_full_range):
        xa = gen(1, 4096)
        assert xa.dtype == np.uint8 and xa.shape == (4096,)
        np.testing.assert_array_equal(xa, gen(1, 4096))
        code = xa & 0x7F
        zero = np.mean(code == 0)
        assert 0.07 < zero < 0.13
        assert code.max() <= 127
    full = W.lns8_activations_full_range(2, 1 << 16) & 0x7F
    nz = full[full != 0]
    # uniform over 1..127: every code appears, and the ends are as common as the middle
    assert set(np.unique(nz)) == set(range(1, 128))
    assert 0.15 < np.mean((nz <= 14) | (nz >= 114)) < 0.30


def test_named_workloads_small():
    w = W.tiny(seed=0, N=8, K=128)
    assert w["t"].shape == (8, 128) and w["d"].shape == (8, 1) and w["x"].shape == (1, 128)
    assert set(np.unique(w["t"])) <= {-1, 0, 1}
    assert w["d"].min() >= 1 and w["d"].max() < (1 << 15)
    w = W.lns8(seed=0, N=16, K=256)
    assert w["dcode"].min() >= 60 and w["dcode"].max() <= 88
    w = W.lm_head(seed=0, N=10, K=128)
    assert w["planes"].shape == (8, 10, 128) and w["s"].min() >= 1
