"""moe_route_noalloc: the router entry point for callers that cannot hand the library a
workspace (a plugin without access to its host framework's allocator, a fully pre-planned
memory budget, or a hot path that must not call the driver allocator). Its scratch is a fixed
device array inside the library. It must give the same routing as moe_route, call after call,
and refuse batches whose scratch would not fit.

This file is collected last on purpose, and passes both alone and after the other tests."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import combine_grouped_gemm_gb300 as m
    return m


def _route_both(moe, cfg, inp):
    """Routing of inp by moe_route (with a workspace) and by moe_route_noalloc, both through
    the C ABI."""
    dev = inp["x"].device
    ws = torch.zeros(moe.query_sizes(cfg)["ws_bytes"], dtype=torch.uint8, device=dev)
    ref_i = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=dev)
    ref_w = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev)
    moe.route(cfg, inp["x"], inp["w_gate"], inp["bias"], ref_i, ref_w, ws)
    got_i = torch.full((cfg.T, cfg.k), -1, dtype=torch.int32, device=dev)
    got_w = torch.full((cfg.T, cfg.k), -1.0, dtype=torch.float32, device=dev)
    c = moe.make_cfg(cfg)
    rc = moe._lib.moe_route_noalloc(ctypes.byref(c), inp["x"].data_ptr(),
                                    inp["w_gate"].data_ptr(), inp["bias"].data_ptr(),
                                    got_i.data_ptr(), got_w.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)
    assert rc == 0, moe._lib.moe_strerror(rc)
    torch.cuda.synchronize()
    return ref_i.cpu().numpy(), ref_w.cpu().numpy(), got_i.cpu().numpy(), got_w.cpu().numpy()


def _oracle_route(cfg, inp):
    x = inp["x"].cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return oracle.route(x, inp["w_gate"].cpu().numpy(), inp["bias"].cpu().numpy(), cfg.k,
                        cfg.n_group, cfg.topk_group, cfg.route_scale)


def test_noalloc_router_matches_the_workspace_router_on_consecutive_calls(moe):
    big = synth.CONFIGS["dsv3_decode"]                   # T=64 x E=256: 1 MiB of scratch
    small = synth.CONFIGS["tiny"]                        # a smaller call after a larger one
    for cfg in (big, small, big.with_seed(1234)):
        inp = synth.make_router_inputs(cfg, "cuda")
        ref_i, ref_w, got_i, got_w = _route_both(moe, cfg, inp)
        assert np.array_equal(got_i, ref_i)
        # the same kernels in the same order: the weights agree exactly, within the 1e-5 bound
        assert np.abs(got_w - ref_w).max() <= 1e-5
        assert np.array_equal(got_w, ref_w)
        # and both are the oracle's, bit for bit
        o_i, o_w = _oracle_route(cfg, inp)
        assert np.array_equal(got_i, o_i)
        assert np.array_equal(got_w, o_w)


def test_noalloc_router_at_1024_tokens_through_the_binding(moe):
    """1024 tokens take the warp-per-token selection kernel (and its shared-memory opt-in); at
    128 experts the partial table fills the fixed array exactly (16 x 1024 x 128 floats)."""
    cfg = synth.MoEConfig("noalloc_t1024", T=1024, d=1024, E=128, k=8, n_group=8, topk_group=4,
                          d_ff=128, d_ff_shared=0, R=8, route_scale=2.5, seed=21)
    inp = synth.make_router_inputs(cfg, "cuda")
    o_i, o_w = _oracle_route(cfg, inp)
    for _ in range(2):                                   # two calls in a row share the array
        got_i = torch.full((cfg.T, cfg.k), -1, dtype=torch.int32, device="cuda")
        got_w = torch.full((cfg.T, cfg.k), -1.0, dtype=torch.float32, device="cuda")
        moe.route_noalloc(cfg, inp["x"], inp["w_gate"], inp["bias"], got_i, got_w)
        torch.cuda.synchronize()
        assert np.array_equal(got_i.cpu().numpy(), o_i)
        assert np.array_equal(got_w.cpu().numpy(), o_w)
    ref_i, ref_w, g_i, g_w = _route_both(moe, cfg, inp)
    assert np.array_equal(g_i, ref_i) and np.array_equal(g_w, ref_w)


def test_noalloc_router_rejects_batches_beyond_its_scratch(moe):
    cfg = synth.CONFIGS["dsv3_sweep"].with_T(1024)       # 16 * 1024 * 256 floats > 2^21
    c = moe.make_cfg(cfg)
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = dummy.data_ptr()
    rc = moe._lib.moe_route_noalloc(ctypes.byref(c), p, p, p, p, p, None)
    assert rc == 2   # MOE_ERR_UNSUPPORTED, nothing enqueued
    ok = synth.CONFIGS["dsv3_sweep"].with_T(512)         # exactly at the limit
    inp = synth.make_router_inputs(ok, "cuda")
    ref_i, _, got_i, _ = _route_both(moe, ok, inp)
    assert np.array_equal(got_i, ref_i)
