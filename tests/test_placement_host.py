"""The library's host-side expert placement (moe_place_experts) against the oracle's, and its
argument checks; no GPU work."""
import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import combine_grouped_gemm_gb300 as m
    return m


def test_library_placement_equals_the_oracles(moe):
    rng = np.random.default_rng(1)
    for trial in range(300):
        E = int(rng.integers(1, 48))
        R = int(rng.integers(1, 9))
        S = int(rng.integers((E + R - 1) // R, (E + R - 1) // R + 5))
        if trial % 3 == 0:
            load = np.round(rng.random(E) * 3, 1)            # many ties
        else:
            load = rng.integers(0, 60, E).astype(np.float64)
        mc = 4 if trial % 5 == 0 else 64                      # sometimes too few copies allowed
        try:
            got = moe.place_experts(load, R, S, max_copies=mc)
        except moe.MoEError as e:
            assert e.code == 1
            got = None
        try:
            ref = oracle.place_experts(load, R, S, max_copies=mc)
        except ValueError:
            ref = None
        assert (got is None) == (ref is None), (trial, E, R, S)
        if got is not None:
            for a, b in zip(got, ref):
                assert np.array_equal(a, b), (trial, E, R, S)


def test_placement_of_the_decode_layer_with_32_redundant_experts(moe):
    """256 experts on 8 ranks of 36 slots (32 spare copies): every slot filled, the heaviest
    experts copied, and the planned rank loads within a few percent of each other."""
    rng = np.random.default_rng(7)
    E, R, S = 256, 8, 36
    # popularity falling as rank^-0.6 over a random permutation: the hottest expert about 10x
    # the mean load, as in the skewed prefill workload
    load = np.empty(E)
    load[rng.permutation(E)] = 1000.0 * np.arange(1, E + 1) ** -0.6
    assert 8 < load.max() / load.mean() < 13
    se, nc, cs = moe.place_experts(load, R, S, max_copies=16)
    assert nc.sum() == R * S and (nc >= 1).all()
    assert np.array_equal(np.bincount(se, minlength=E), nc)
    top = np.argsort(-load, kind="stable")[:8]
    assert (nc[top] >= 2).all()
    rank = np.zeros(R)
    for p, e in enumerate(se):
        rank[p // S] += load[e] / nc[e]
    assert rank.max() / rank.mean() <= 1.05


def test_placement_arguments_are_checked(moe):
    import ctypes
    L = moe._lib
    load = np.ones(8)
    out = np.zeros(64, dtype=np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)   # noqa: E731
    assert L.moe_place_experts(8, 2, 3, p(load), 4, p(out), p(out), p(out)) == 1   # 6 < 8 slots
    assert L.moe_place_experts(8, 2, 4, None, 4, p(out), p(out), p(out)) == 1
    bad = load.copy()
    bad[3] = np.nan
    assert L.moe_place_experts(8, 2, 4, p(bad), 4, p(out), p(out), p(out)) == 1
    bad[3] = -1.0
    assert L.moe_place_experts(8, 2, 4, p(bad), 4, p(out), p(out), p(out)) == 1
    assert L.moe_place_experts(8, 2, 4, p(load), 0, p(out), p(out), p(out)) == 1
    assert L.moe_place_experts(8, 2, 4, p(load), 4, p(out), p(out), p(out)) == 0


def test_placed_sizes(moe):
    import synth
    c = synth.CONFIGS["dsv3_skew_prefill"]
    s = moe.query_sizes_placed(c, 36)
    cap = (c.T // c.R) * min(c.k, 36)
    assert s["cap"] == cap and s["recv_rows"] == c.R * c.R * cap
    assert s["ws_bytes"] >= moe.query_sizes(c)["ws_bytes"]
    with pytest.raises(moe.MoEError):
        moe.query_sizes_placed(c, 31)          # 8 x 31 < 256 experts
