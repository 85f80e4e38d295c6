"""The C-ABI library loads, exports every symbol include/moe.h declares, and its host-side
checks behave; nothing here launches GPU work."""
import ctypes
import os
import re

import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def moe():
    import __graft_entry__
    __graft_entry__.build()
    import combine_grouped_gemm_gb300 as m
    return m


def declared_functions():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(moe_\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(moe):
    names = declared_functions()
    assert len(names) >= 12
    lib = ctypes.CDLL(moe.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(moe.EXPORTED)


def test_abi_version_and_strerror(moe):
    assert moe.abi_version() == 3
    for code in range(5):
        assert moe._lib.moe_strerror(code)
    assert b"unknown" in moe._lib.moe_strerror(99)


def test_workload_configs_validate(moe):
    for c in synth.CONFIGS.values():
        assert moe.validate(c) == 0, c.name


@pytest.mark.parametrize("change,code", [
    (dict(T=17), 1),                      # T % R
    (dict(E=15), 1),                      # E % R
    (dict(k=9), 1),                       # k > topk_group * E / n_group (16 / 1 ... with n_group 2)
    (dict(topk_group=3), 1),              # topk_group > n_group
    (dict(d=200), 2),                     # d % 128
    (dict(d_ff=100), 2),                  # d_ff % 128
    (dict(E=2048, R=2), 2),               # E > 1024
    (dict(k=33, E=64, n_group=1), 2),     # k > 32
    (dict(d_ff_shared=256), 2),           # shared width != routed width
    (dict(act="fp8"), 2),                 # mixed activation / weight formats
    (dict(act="fp8", w="fp8", scales="pow2", d=384), 2),   # power-of-two recipe: d % 256
])
def test_invalid_configs_are_rejected(moe, change, code):
    import dataclasses
    base = dataclasses.replace(synth.CONFIGS["tiny"], n_group=2, topk_group=1)
    c = dataclasses.replace(base, **change)
    assert moe.validate(c) == code


def test_pow2_recipe_maps_to_its_own_format(moe):
    """An e4m3 configuration with power-of-two scales is its own element format; out-of-range
    format codes are rejected."""
    import dataclasses
    c = synth.CONFIGS["dsv3_fp8_pow2_prefill"]
    mc = moe.make_cfg(c)
    assert mc.act_dtype == mc.w_dtype == moe.MOE_FP8_E4M3_POW2
    assert moe.make_cfg(synth.CONFIGS["dsv3_fp8_prefill"]).act_dtype == moe.MOE_FP8_E4M3
    s2, s8 = moe.query_sizes(c), moe.query_sizes(synth.CONFIGS["dsv3_fp8_prefill"])
    assert {k: v for k, v in s2.items() if k != "ws_bytes"} == \
        {k: v for k, v in s8.items() if k != "ws_bytes"}
    # the workspace adds the 64-byte scale rows of the GEMM inputs: 2 x T*k + 2 x T of them
    assert s2["ws_bytes"] - s8["ws_bytes"] >= 64 * (2 * c.T * c.k + 2 * c.T)
    L = moe._lib
    for bad in (-1, 3):
        b = moe.make_cfg(dataclasses.replace(synth.CONFIGS["tiny"], n_group=2, topk_group=1))
        b.act_dtype = b.w_dtype = bad
        assert L.moe_validate(ctypes.byref(b)) == 1


def test_workspace_mirror_matches_the_library(moe):
    """The tests' copy of the workspace layout (used to read intermediates) ends where the
    library's does, for every format."""
    import dataclasses
    from gpu_util import ws_offsets
    for c in list(synth.CONFIGS.values()) + [
            dataclasses.replace(synth.CONFIGS["dsv3_fp8_pow2_e32"], T=200, R=8, E=32)]:
        assert ws_offsets(c)["total"] == moe.query_sizes(c)["ws_bytes"], c.name


def test_sizes_follow_the_layout(moe):
    c = synth.CONFIGS["dsv3_decode"]
    s = moe.query_sizes(c)
    assert s["cap"] == c.cap == 64
    assert s["recv_rows"] == c.R * c.R * c.cap
    assert s["recv_bytes"] == s["recv_rows"] * c.d * 2 == s["ebuf_bytes"]
    assert s["recv_scale_bytes"] == 0
    f = synth.CONFIGS["dsv3_fp8_prefill"]
    s8 = moe.query_sizes(f)
    assert s8["recv_bytes"] == s8["recv_rows"] * f.d
    assert s8["recv_scale_bytes"] == s8["recv_rows"] * (f.d // 128) * 4
    assert s8["ebuf_bytes"] == 2 * s8["recv_bytes"]


def test_null_and_misaligned_pointers_are_rejected_before_any_launch(moe):
    c = moe.make_cfg(synth.CONFIGS["tiny"])
    L = moe._lib
    ok = 1 << 20  # an aligned fake address: never dereferenced, checks fail first
    assert L.moe_route(ctypes.byref(c), None, ok, ok, ok, ok, ok, None) == 1
    assert L.moe_route(ctypes.byref(c), ok + 2, ok, ok, ok, ok, ok, None) == 3
    assert L.moe_combine(ctypes.byref(c), ok, ok, ok, ok + 8, ok, None, None) == 3
    assert L.moe_combine(ctypes.byref(c), ok, ok, ok, None, ok, ok + 2, None) == 3  # status
    assert L.moe_dispatch(ctypes.byref(c), ok, ok, ok, None, ok, None, None, None, None) == 1
    assert L.moe_dispatch(ctypes.byref(c), ok, ok, ok, None, ok, ok, None, ok + 1, None) == 3
    assert L.moe_dispatch_index(ctypes.byref(c), ok, ok, ok, None, None, None) == 1
    assert L.moe_expert_ffn_gather(ctypes.byref(c), ok, ok, None, ctypes.byref(moe.Weights()),
                                   ok, None, ok, None) == 1
    # moe_layer_ex: an unknown option bit, or a side stream asked for without stream and events
    o = moe.LayerOpts(flags=64)
    assert L.moe_layer_ex(ctypes.byref(c), ctypes.byref(o), *([ok] * 14), None, None) == 1
    w = moe.Weights()
    assert L.moe_expert_ffn(ctypes.byref(c), ok, None, ok, None, ctypes.byref(w), ok, None, ok,
                            None) == 1
    bad = moe.make_cfg(synth.CONFIGS["tiny"])
    bad.T = 15
    assert L.moe_layer(ctypes.byref(bad), *([ok] * 14), None, None) == 1
    assert L.moe_read_status(None, None, None) == 1
    # the wait diagnostic: no workspace, a misaligned one, or a limit outside 1 us .. 10 s
    assert L.moe_selftest_wait(None, 10 ** 6, None) == 1
    assert L.moe_selftest_wait(ok + 4, 10 ** 6, None) == 1
    assert L.moe_selftest_wait(ok, 999, None) == 1
    assert L.moe_selftest_wait(ok, 10 ** 10 + 1, None) == 1


def test_noalloc_router_checks_before_any_launch(moe):
    # every refusal of moe_route_noalloc comes before it touches the device
    L = moe._lib
    ok = 1 << 20
    c = moe.make_cfg(synth.CONFIGS["tiny"])
    assert L.moe_route_noalloc(None, ok, ok, ok, ok, ok, None) == 1
    assert L.moe_route_noalloc(ctypes.byref(c), None, ok, ok, ok, ok, None) == 1
    assert L.moe_route_noalloc(ctypes.byref(c), ok, ok, ok, ok + 4, ok, None) == 3
    bad = moe.make_cfg(synth.CONFIGS["tiny"])
    bad.T = 15                                              # T % R != 0
    assert L.moe_route_noalloc(ctypes.byref(bad), ok, ok, ok, ok, ok, None) == 1
    # 16 partials per token and expert: 512 tokens at 256 experts fill the fixed 8 MiB scratch,
    # 520 do not fit
    fits = moe.make_cfg(synth.CONFIGS["dsv3_sweep"].with_T(512))
    big = moe.make_cfg(synth.CONFIGS["dsv3_sweep"].with_T(520))
    assert 16 * fits.T * fits.E == 2 ** 21
    assert L.moe_route_noalloc(ctypes.byref(big), ok, ok, ok, ok, ok, None) == 2
