"""Parity of the CUDA path (called through the C ABI) with the CPU oracle.

Indices, counts, permutations and e4m3 codes must match bit for bit; gate weights within 1e-5;
expert outputs and layer outputs within 2e-2 of max-abs error relative to the output RMS (bf16).
Small workloads are compared element by element in full; the DeepSeek-V3-sized workloads on
sampled tokens / rows the oracle computes one by one, plus invariants that hold at any size.
"""
import dataclasses
import functools

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import (bf16_to_f64, expert_getter, format_err, host_bits, rel_max_err,
                      shared_host, weight_dict)
from layer_check import check_layer, experts_by_rows, hot_expert_pairs

pytestmark = pytest.mark.gpu

TOL_BF16 = 2e-2


@functools.lru_cache(maxsize=1)
def moe():
    import combine_grouped_gemm_gb300 as m
    return m


# A small layer whose shapes span several tiles and ragged tails: 5 gate/up weight tiles,
# 3 down tiles, a shared expert with more rows than one token tile, 3 logical ranks.
SMALL = synth.MoEConfig("small", T=96, d=384, E=12, k=3, n_group=4, topk_group=2, d_ff=640,
                        d_ff_shared=640, R=3, route_scale=2.5, seed=77)
# 64 experts per logical rank: the schedule takes its block-wide scan path (the other shapes
# have at most 32 experts per rank, one warp).
ER64 = synth.MoEConfig("er64", T=64, d=256, E=128, k=4, n_group=4, topk_group=2, d_ff=128,
                       d_ff_shared=128, R=2, route_scale=1.0, seed=11)
# 64 logical ranks of 3 experts: the counts table (64 x 192 x 4 = 48 KB) is too large to stage
# in the schedule kernel's shared memory, and a rank's experts do not divide a warp.
E192_R64 = synth.MoEConfig("e192_r64", T=128, d=256, E=192, k=4, n_group=4, topk_group=2,
                           d_ff=128, d_ff_shared=128, R=64, route_scale=1.0, seed=19)
# One expert receives every token (bias +10): several token tiles of one expert.
HOT = synth.MoEConfig("hot", T=256, d=256, E=16, k=2, n_group=1, topk_group=1, d_ff=256,
                      d_ff_shared=256, R=2, route_scale=1.0, seed=5)
# A full 128-row token tile per expert on average (T*k >= 128*E): the bf16 GEMMs run on the
# schedule's 256-row token tiles. Experts of 1, 2 and 3 ragged 128-row tiles; and the hot
# expert with 1024 rows (and the shared expert's 1024).
PAIRED = synth.MoEConfig("paired", T=512, d=256, E=8, k=2, n_group=2, topk_group=2, d_ff=256,
                         d_ff_shared=256, R=2, route_scale=1.0, seed=29)
HOT_PAIRED = dataclasses.replace(HOT, name="hot_paired", T=1024)
# ... with T = 700: the shared expert's last 256-row tile has 188 rows, its second 128-row box
# runs past the last token (zero-filled)
PAIRED_RAGGED = dataclasses.replace(PAIRED, name="paired_ragged", T=700, seed=31)

_cache = {}       # router inputs per workload
_wcache = {}      # expert weights per (seed, shapes, format): sweep points share one set
BIG_KEEP = 4      # DeepSeek-V3-sized weight sets kept at once (<= 23 GB each)


def inputs(cfg):
    """Device inputs for cfg. Weight sets are shared by workloads that differ only in T; at most
    BIG_KEEP large ones stay alive."""
    wkey = (cfg.seed, cfg.E, cfg.d, cfg.d_ff, cfg.d_ff_shared, cfg.w, cfg.scales)
    if wkey not in _wcache:
        big = cfg.d * cfg.d_ff * cfg.E > 10 ** 8
        if big:
            bigs = [k for k in _wcache if _wcache[k][1]]
            for k in bigs[:max(0, len(bigs) - BIG_KEEP + 1)]:
                del _wcache[k]
            torch.cuda.empty_cache()
        _wcache[wkey] = (synth.make_expert_weights(cfg, "cuda"), big)
    key = (cfg.name, cfg.seed, cfg.T, cfg.bias)
    if key not in _cache:
        inp = synth.make_router_inputs(cfg, "cuda")
        if cfg.name == "hot":
            inp["bias"][3] = 10.0
        _cache[key] = inp
    return _cache[key], _wcache[wkey][0]


def run_stages(cfg, inp, W, src_tok=True):
    m = moe()
    b = m.Buffers(cfg)
    m.clear_status(b["ws"])
    m.route(cfg, inp["x"], inp["w_gate"], inp["bias"], b["topk_idx"], b["topk_w"], b["ws"])
    st = None
    if src_tok:
        st = torch.empty(b.sizes["recv_rows"], dtype=torch.int32, device="cuda")
    m.dispatch(cfg, inp["x"], b["topk_idx"], b["recv"], b["recv_scales"], b["counts"],
               b["row_of"], st)
    out = dict(b)
    out["src_tok"] = st
    return out


def oracle_route(cfg, inp, tokens=None):
    x = host_bits(inp["x"])
    if tokens is not None:
        x = x[tokens]
    return oracle.route(x, inp["w_gate"].cpu().numpy(), inp["bias"].cpu().numpy(), cfg.k,
                        cfg.n_group, cfg.topk_group, cfg.route_scale)


# ------------------------------------------------------------------------------------------
# Router
# ------------------------------------------------------------------------------------------
# T spans the partial-dot kernels (the resident slice with 32 / 64 / 128-token tiles up to 128
# tokens, ragged at 40 and 104; staged 64x64 tiles below 512, the cp.async ring's 128x128 tiles
# from there) and the selection kernels (a CTA per token below 1024 tokens, a warp per token
# from there, 2 / 4 warps per CTA at 1024 and 1152 / 1536 tokens; 8 lanes per token for 256
# experts in 8 groups from 2048 tokens: the direct tests below)
ROUTE_FULL = [synth.CONFIGS["tiny"], SMALL, HOT, synth.CONFIGS["dsv3_decode"],
              synth.CONFIGS["dsv3_sweep"].with_T(8), synth.CONFIGS["dsv3_sweep"].with_T(40),
              synth.CONFIGS["dsv3_sweep"].with_T(104), synth.CONFIGS["dsv3_sweep"].with_T(256),
              synth.CONFIGS["dsv3_sweep"].with_T(1024), synth.CONFIGS["dsv3_sweep"].with_T(1536),
              dataclasses.replace(HOT, name="hot_T1152", T=1152)]


@pytest.mark.parametrize("cfg", ROUTE_FULL, ids=lambda c: c.name)
def test_route_bit_exact(cfg):
    inp, W = inputs(cfg)
    r = run_stages(cfg, inp, W)
    idx, w = oracle_route(cfg, inp)
    assert np.array_equal(r["topk_idx"].cpu().numpy(), idx)
    assert np.abs(r["topk_w"].cpu().numpy() - w).max() <= 1e-5
    assert np.array_equal(r["topk_w"].cpu().numpy(), w)   # same op sequence: exact


@pytest.mark.parametrize("name", ["dsv3_skew_prefill", "dsv3_fp8_prefill"])
def test_route_bit_exact_sampled_large(name):
    cfg = synth.CONFIGS[name]
    inp = synth.make_router_inputs(cfg, "cuda")
    m = moe()
    ws = torch.zeros(m.query_sizes(cfg)["ws_bytes"], dtype=torch.uint8, device="cuda")
    idx_d = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device="cuda")
    w_d = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device="cuda")
    m.route(cfg, inp["x"], inp["w_gate"], inp["bias"], idx_d, w_d, ws)
    rng = np.random.default_rng(cfg.seed)
    tokens = np.unique(np.concatenate([[0, cfg.T - 1], rng.choice(cfg.T, 254, replace=False)]))
    idx, w = oracle_route(cfg, inp, tokens)
    assert np.array_equal(idx_d.cpu().numpy()[tokens], idx)
    assert np.abs(w_d.cpu().numpy()[tokens] - w).max() <= 1e-5
    if cfg.bias == "zipf":   # the skew recipe: hottest expert about 10x the mean load
        c = np.bincount(idx_d.cpu().numpy().reshape(-1), minlength=cfg.E)
        assert 8.0 <= c.max() / c.mean() <= 12.0


# From 512 tokens the partial dot products go through the cp.async ring kernel (128x128 tiles,
# 16-column k-steps): token and expert counts that leave the last tiles part-filled, a chunk of
# two k-steps (fewer than the ring's stages), expert counts that are not a multiple of 4 (the
# scalar store path), and the full model width at ragged token counts, the second one past
# 2048 tokens (8-lane-per-token selection, its last CTA part-filled). Every token is checked.
RING_RAGGED = [
    dataclasses.replace(SMALL, name="ring_small", T=702, d=512),
    synth.MoEConfig("ring_e18", T=531, d=768, E=18, k=3, n_group=3, topk_group=2, d_ff=128,
                    d_ff_shared=0, R=3, route_scale=1.5, seed=123),
    synth.CONFIGS["dsv3_sweep"].with_T(600),
    synth.CONFIGS["dsv3_sweep"].with_T(2056),
]


@pytest.mark.parametrize("cfg", RING_RAGGED, ids=lambda c: c.name)
def test_route_bit_exact_ring_ragged(cfg):
    inp = synth.make_router_inputs(cfg, "cuda")
    m = moe()
    ws = torch.zeros(m.query_sizes(cfg)["ws_bytes"], dtype=torch.uint8, device="cuda")
    idx_d = torch.full((cfg.T, cfg.k), -1, dtype=torch.int32, device="cuda")
    w_d = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device="cuda")
    m.route(cfg, inp["x"], inp["w_gate"], inp["bias"], idx_d, w_d, ws)
    idx, w = oracle_route(cfg, inp)
    assert np.array_equal(idx_d.cpu().numpy(), idx)
    assert np.array_equal(w_d.cpu().numpy(), w)   # same op sequence: exact


@pytest.mark.parametrize("T", [64, 1024, 2048])
def test_route_ties_go_to_the_lower_index(T):
    # experts 2i and 2i+1 get the same gate row and bias, so every key comes in equal pairs
    # (and a group's two largest keys can be a pair): the three selection kernels (a CTA per
    # token, a warp per token, 8 lanes per token) must pick the lower index first, as the
    # oracle does
    cfg = synth.CONFIGS["dsv3_sweep"].with_T(T)
    inp = synth.make_router_inputs(cfg, "cuda")
    wg = inp["w_gate"].clone()
    wg[1::2] = wg[0::2]
    b = inp["bias"].clone()
    b[1::2] = b[0::2]
    inp = dict(x=inp["x"], w_gate=wg, bias=b)
    m = moe()
    ws = torch.zeros(m.query_sizes(cfg)["ws_bytes"], dtype=torch.uint8, device="cuda")
    idx_d = torch.full((cfg.T, cfg.k), -1, dtype=torch.int32, device="cuda")
    w_d = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device="cuda")
    m.route(cfg, inp["x"], inp["w_gate"], inp["bias"], idx_d, w_d, ws)
    idx, w = oracle_route(cfg, inp)
    got = idx_d.cpu().numpy()
    assert np.array_equal(got, idx)
    assert np.array_equal(w_d.cpu().numpy(), w)
    # both members of a pair chosen: the even one comes first
    for row in got:
        pos = {e: i for i, e in enumerate(row)}
        for e, i in pos.items():
            if e % 2 == 1 and e - 1 in pos:
                assert pos[e - 1] < i


# ------------------------------------------------------------------------------------------
# Dispatch
# ------------------------------------------------------------------------------------------
@pytest.mark.parametrize("cfg", ROUTE_FULL, ids=lambda c: c.name)
def test_dispatch_bit_exact(cfg):
    inp, W = inputs(cfg)
    r = run_stages(cfg, inp, W)
    idx = r["topk_idx"].cpu().numpy()
    counts, _, row_of, src_tok = oracle.dispatch_index(oracle_route(cfg, inp)[0], cfg.E, cfg.R)
    assert np.array_equal(r["counts"].cpu().numpy(), counts)
    assert np.array_equal(r["row_of"].cpu().numpy(), row_of)
    assert np.array_equal(r["src_tok"].cpu().numpy(), src_tok)
    recv = host_bits(r["recv"])
    ref, _ = oracle.dispatch_payload(host_bits(inp["x"]), row_of, src_tok.size)
    filled = src_tok >= 0
    assert np.array_equal(recv[filled], ref[filled])
    assert counts.sum() == cfg.T * cfg.k and idx.shape == (cfg.T, cfg.k)


def test_dispatch_given_topk_matches_oracle():
    """Dispatch alone on seeded random choices (not produced by the router)."""
    cfg = SMALL
    rng = np.random.default_rng(3)
    ti = np.stack([rng.permutation(cfg.E)[:cfg.k] for _ in range(cfg.T)]).astype(np.int32)
    inp, _ = inputs(cfg)
    m = moe()
    b = m.Buffers(cfg)
    st = torch.empty(b.sizes["recv_rows"], dtype=torch.int32, device="cuda")
    m.dispatch(cfg, inp["x"], torch.from_numpy(ti).cuda(), b["recv"], None, b["counts"],
               b["row_of"], st)
    counts, _, row_of, src_tok = oracle.dispatch_index(ti, cfg.E, cfg.R)
    assert np.array_equal(b["counts"].cpu().numpy(), counts)
    assert np.array_equal(b["row_of"].cpu().numpy(), row_of)
    assert np.array_equal(st.cpu().numpy(), src_tok)


FP8_SMALL = dataclasses.replace(SMALL, name="small_fp8", act="fp8", w="fp8", d=512, d_ff=256,
                                d_ff_shared=256)
# the same with power-of-two block scales (block-scaled MMA)
P2_SMALL = dataclasses.replace(FP8_SMALL, name="small_fp8p2", scales="pow2")


def test_dispatch_e4m3_codes_and_scales_bit_exact():
    cfg = FP8_SMALL
    inp = synth.make_router_inputs(cfg, "cuda")
    m = moe()
    b = m.Buffers(cfg)
    m.route(cfg, inp["x"], inp["w_gate"], inp["bias"], b["topk_idx"], b["topk_w"], b["ws"])
    m.dispatch(cfg, inp["x"], b["topk_idx"], b["recv"], b["recv_scales"], b["counts"],
               b["row_of"], None)
    idx, _ = oracle_route(cfg, inp)
    assert np.array_equal(b["topk_idx"].cpu().numpy(), idx)
    _, _, row_of, src_tok = oracle.dispatch_index(idx, cfg.E, cfg.R)
    q, sc = oracle.dispatch_payload(host_bits(inp["x"]), row_of, src_tok.size, fp8=True)
    filled = src_tok >= 0
    assert np.array_equal(b["recv"].cpu().numpy()[filled], q[filled])
    # the library's scales are block-major [d/128][rows]
    assert np.array_equal(b["recv_scales"].cpu().numpy().T[filled], sc[filled])


@pytest.mark.parametrize("name", ["dsv3_skew_prefill", "dsv3_fp8_prefill"])
def test_dispatch_invariants_large(name):
    """At full size: the permutation is the unique stable rank-major layout of the routing,
    and sampled receive rows hold their token's row (bf16) or its e4m3 codes."""
    cfg = synth.CONFIGS[name]
    inp = synth.make_router_inputs(cfg, "cuda")
    m = moe()
    b = m.Buffers(cfg)
    st = torch.empty(b.sizes["recv_rows"], dtype=torch.int32, device="cuda")
    m.route(cfg, inp["x"], inp["w_gate"], inp["bias"], b["topk_idx"], b["topk_w"], b["ws"])
    m.dispatch(cfg, inp["x"], b["topk_idx"], b["recv"], b["recv_scales"], b["counts"],
               b["row_of"], st)
    ti = b["topk_idx"].cpu().numpy().astype(np.int64)
    ro = b["row_of"].cpu().numpy().astype(np.int64)
    counts = b["counts"].cpu().numpy()
    src = st.cpu().numpy()
    T, k, E, R = cfg.T, cfg.k, cfg.E, cfg.R
    Ts, Er, cap = cfg.T_s, cfg.E_r, cfg.cap
    assert counts.sum() == T * k
    assert len(np.unique(ro)) == T * k                      # injective
    tok = np.repeat(np.arange(T), k)
    assert np.array_equal(src[ro.reshape(-1)], tok)          # src_tok inverts row_of
    assert (src >= 0).sum() == T * k
    s_of = tok // Ts
    e_of = ti.reshape(-1)
    r_of = e_of // Er
    seg = ro.reshape(-1) // cap
    assert np.array_equal(seg, r_of * R + s_of)              # right (destination, source) segment
    # inside a segment: expert-major (ascending), token ascending, packed from 0
    exp_cnt = np.zeros((R, E), np.int64)
    np.add.at(exp_cnt, (s_of, e_of), 1)
    assert np.array_equal(exp_cnt, counts)
    ex = np.cumsum(counts.reshape(R, R, Er), axis=2) - counts.reshape(R, R, Er)
    first = ex.reshape(R, E)[s_of, e_of]
    order = np.lexsort((tok, e_of, seg))
    pos = np.empty(T * k, np.int64)
    run = np.zeros((R, E), np.int64)
    for j in order:                                          # ranks by token inside (s, e)
        pos[j] = run[s_of[j], e_of[j]]
        run[s_of[j], e_of[j]] += 1
    assert np.array_equal(ro.reshape(-1) % cap, first + pos)
    rng = np.random.default_rng(1)
    rows = rng.choice(T * k, 64, replace=False)
    x = host_bits(inp["x"])
    if cfg.act == "fp8":
        toks = tok[rows]
        q, sc = oracle.quant_rows_e4m3(oracle.bf16_to_f32(x[toks]))
        assert np.array_equal(b["recv"][ro.reshape(-1)[rows]].cpu().numpy(), q)
        assert np.array_equal(b["recv_scales"][:, ro.reshape(-1)[rows]].cpu().numpy().T, sc)
    else:
        assert np.array_equal(host_bits(b["recv"][ro.reshape(-1)[rows]]), x[tok[rows]])


# ------------------------------------------------------------------------------------------
# Combine
# ------------------------------------------------------------------------------------------
@pytest.mark.parametrize("cfg", [synth.CONFIGS["tiny"], SMALL, synth.CONFIGS["dsv3_decode"]],
                         ids=lambda c: c.name)
def test_combine_identity_experts_give_scaled_x(cfg):
    inp, W = inputs(cfg)
    r = run_stages(cfg, inp, W)
    m = moe()
    y = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    m.combine(cfg, r["recv"], r["row_of"], r["topk_w"], None, y)
    x = bf16_to_f64(host_bits(inp["x"]))
    yf = bf16_to_f64(host_bits(y))
    assert np.all(np.abs(yf - cfg.route_scale * x) <= 2 ** -7 * np.abs(cfg.route_scale * x) + 1e-30)
    ref = oracle.combine(host_bits(r["recv"]), r["row_of"].cpu().numpy(), r["topk_w"].cpu().numpy())
    assert np.abs(host_bits(y).astype(np.int32) - ref.astype(np.int32)).max() <= 1


def test_combine_with_shared_matches_oracle():
    cfg = SMALL
    inp, W = inputs(cfg)
    r = run_stages(cfg, inp, W)
    g = torch.Generator().manual_seed(4)
    ebuf = (torch.randn(r["ebuf"].shape, generator=g) * 0.5).to(torch.bfloat16).cuda()
    sh = torch.randn((cfg.T, cfg.d), generator=g).to(torch.bfloat16).cuda()
    y = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    moe().combine(cfg, ebuf, r["row_of"], r["topk_w"], sh, y)
    ref = oracle.combine(host_bits(ebuf), r["row_of"].cpu().numpy(), r["topk_w"].cpu().numpy(),
                         host_bits(sh))
    assert np.abs(host_bits(y).astype(np.int32) - ref.astype(np.int32)).max() <= 1


# ------------------------------------------------------------------------------------------
# Expert FFN and the whole layer
# ------------------------------------------------------------------------------------------
def _ffn(cfg, inp, W, r):
    m = moe()
    m.expert_ffn(cfg, r["recv"], r["recv_scales"], r["counts"], inp["x"], weight_dict(W),
                 r["ebuf"], r["shared_out"], r["ws"])
    return r


@pytest.mark.parametrize("cfg", [synth.CONFIGS["tiny"], SMALL, HOT], ids=lambda c: c.name)
def test_expert_ffn_every_row(cfg):
    inp, W = inputs(cfg)
    r = _ffn(cfg, inp, W, run_stages(cfg, inp, W))
    assert moe().read_status(r["ws"]) == 0
    src = r["src_tok"].cpu().numpy()
    ti = r["topk_idx"].cpu().numpy()
    ro = r["row_of"].cpu().numpy()
    x = host_bits(inp["x"])
    eb = host_bits(r["ebuf"])
    get = expert_getter(W, False)
    worst = 0.0
    for e in range(cfg.E):
        Wt = get(e)
        for t, i in zip(*np.nonzero(ti == e)):
            ref, _ = oracle.swiglu_row_bf16(x[t], Wt["w13"], Wt["w2"])
            worst = max(worst, rel_max_err(bf16_to_f64(eb[ro[t, i]]), bf16_to_f64(ref)))
            assert src[ro[t, i]] == t
    assert worst <= TOL_BF16, worst
    if cfg.d_ff_shared:
        S = shared_host(W, False)
        sh = host_bits(r["shared_out"])
        for t in range(cfg.T):
            ref, _ = oracle.swiglu_row_bf16(x[t], S["ws13"], S["ws2"])
            assert rel_max_err(bf16_to_f64(sh[t]), bf16_to_f64(ref)) <= TOL_BF16


def _layer_tokens_check(cfg, tokens, inp, W, y):
    ref = oracle.layer_tokens(cfg, host_bits(inp["x"]), inp["w_gate"].cpu().numpy(),
                              inp["bias"].cpu().numpy(), expert_getter(W, cfg.w == "fp8"),
                              shared_host(W, cfg.w == "fp8"), tokens)
    got = bf16_to_f64(host_bits(y)[tokens])
    return format_err(got, ref["y_exact"])


@pytest.mark.parametrize("cfg", [synth.CONFIGS["tiny"], SMALL, HOT, ER64, E192_R64, PAIRED,
                                 HOT_PAIRED, PAIRED_RAGGED], ids=lambda c: c.name)
def test_layer_all_tokens(cfg):
    inp, W = inputs(cfg)
    lay = moe().MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))
    y = lay(inp["x"])
    assert moe().read_status(lay.bufs["ws"]) == 0
    assert _layer_tokens_check(cfg, np.arange(cfg.T), inp, W, y) <= TOL_BF16


def test_bounded_wait_gives_up_reports_and_leaves_the_context_usable():
    """Failure handling on the device: a wait on a barrier that nothing completes gives up
    after its limit, records MOE_DEV_TIMEOUT in the workspace status word and raises the CTA's
    abort flag, on which a second wait (limit 3x) returns at once; afterwards a layer still
    runs and matches the oracle."""
    m = moe()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    m.clear_status(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    limit_ms = 50.0
    e0.record()
    m.selftest_wait(ws, int(limit_ms * 1e6))
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    assert m.read_status(ws) == m.MOE_DEV_TIMEOUT
    assert limit_ms <= ms < 2.5 * limit_ms, ms   # the second wait left on the abort flag
    m.clear_status(ws)
    assert m.read_status(ws) == 0
    cfg = synth.CONFIGS["tiny"]
    inp, W = inputs(cfg)
    lay = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))
    y = lay(inp["x"])
    assert m.read_status(lay.bufs["ws"]) == 0
    assert _layer_tokens_check(cfg, np.arange(cfg.T), inp, W, y) <= TOL_BF16


def _run_layer(cfg):
    inp, W = inputs(cfg)
    lay = moe().MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))
    y = lay(inp["x"])
    assert moe().read_status(lay.bufs["ws"]) == 0
    return inp, W, lay, y


@pytest.mark.slow
def test_layer_dsv3_decode_every_token():
    """The DeepSeek-V3 decode layer (T=64): every token's output and every expert-output row
    (all 512 routed rows, 64 shared rows) against the oracle."""
    cfg = synth.CONFIGS["dsv3_decode"]
    inp, W, lay, y = _run_layer(cfg)
    res = check_layer(cfg, inp, W, lay.bufs, y, np.arange(cfg.T), tol=TOL_BF16)
    print(cfg.name, res)
    assert res["rows"] == cfg.T * cfg.k and res["tokens"] == cfg.T


@pytest.mark.slow
@pytest.mark.parametrize("T", synth.SWEEP_T)
def test_layer_dsv3_sweep_point(T):
    """Each point of the decode sweep (1..128 tokens per logical rank): at least 32 tokens'
    outputs (all of them up to 32) and every row of 16 touched experts, among them the four
    with the most rows (at 512+ tokens those fill token tiles past 32 rows, the cp.async
    gather path; below, the four-row TMA gathers)."""
    cfg = synth.CONFIGS["dsv3_sweep"].with_T(T)
    inp, W, lay, y = _run_layer(cfg)
    ti = lay.bufs["topk_idx"].cpu().numpy()
    rng = np.random.default_rng(T)
    tokens = np.arange(T) if T <= 32 else np.sort(rng.choice(T, 32, replace=False))
    n = experts_by_rows(ti, cfg.E)
    touched = np.nonzero(n)[0]
    top = touched[np.argsort(-n[touched], kind="stable")][:4]
    rest = np.setdiff1d(touched, top)
    pick = np.concatenate([top, rng.choice(rest, min(12, rest.size), replace=False)])
    extra = [p for e in pick for p in hot_expert_pairs(ti, int(e))]
    res = check_layer(cfg, inp, W, lay.bufs, y, tokens, extra, tol=TOL_BF16)
    print(cfg.name, res)
    assert res["tokens"] >= min(T, 32) and res["experts"] >= 16


def _prefill_pairs(cfg, bufs, rng):
    """Expert rows for the large prefill checks: every row of the hottest expert, every row of an
    expert whose rows fill a token tile past 32 rows and of one with at most 32, and every row
    of two experts whose compact rows lie past the first 1024 (the schedule's grid-filled row
    list)."""
    ti = bufs["topk_idx"].cpu().numpy()
    n = experts_by_rows(ti, cfg.E)
    off = np.cumsum(n) - n
    hot = int(np.argmax(n))
    chosen = [hot]
    mid = np.nonzero((n > 32) & (n <= 64))[0]
    if mid.size:
        chosen.append(int(mid[0]))
    small = np.nonzero((n > 0) & (n <= 32))[0]
    if small.size:
        chosen.append(int(small[-1]))
    late = np.setdiff1d(np.nonzero((off >= 1024) & (n > 0))[0], chosen)
    chosen += [int(e) for e in rng.choice(late, min(2, late.size), replace=False)]
    return [p for e in chosen for p in hot_expert_pairs(ti, e)], hot, n


@pytest.mark.slow
def test_layer_skew_prefill_rows_and_tokens():
    """The Zipf-skewed prefill (T=4096, bf16): every row of the hottest expert (about 10x the
    mean load: many token tiles), of a 33..64-row expert, of a <=32-row one and of two experts
    past the first 1024 compact rows, plus 256 tokens' whole layer output; >= 1024 rows."""
    cfg = synth.CONFIGS["dsv3_skew_prefill"]
    inp, W, lay, y = _run_layer(cfg)
    rng = np.random.default_rng(cfg.seed)
    extra, hot, n = _prefill_pairs(cfg, lay.bufs, rng)
    assert n[hot] >= 8 * n.mean()
    tokens = np.sort(rng.choice(cfg.T, 256, replace=False))
    res = check_layer(cfg, inp, W, lay.bufs, y, tokens, extra, tol=TOL_BF16)
    print(cfg.name, res)
    assert res["rows"] >= 1024


def test_layer_equals_stage_calls_and_is_deterministic():
    cfg = SMALL
    inp, W = inputs(cfg)
    lay = moe().MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))
    y1 = lay(inp["x"]).clone()
    y2 = lay(inp["x"]).clone()
    assert torch.equal(y1, y2)
    r = _ffn(cfg, inp, W, run_stages(cfg, inp, W))
    y3 = torch.empty_like(y1)
    moe().combine(cfg, r["ebuf"], r["row_of"], r["topk_w"], r["shared_out"], y3)
    assert torch.equal(y1, y3)


@pytest.mark.parametrize("cfg", [SMALL, FP8_SMALL, P2_SMALL, synth.CONFIGS["dsv3_decode"]],
                         ids=lambda c: c.name)
def test_back_to_back_layers_match_single_calls(cfg):
    # Layer calls queued one after another on the stream with no synchronisation: within a call
    # every kernel after the first is launched programmatically and has to wait for its
    # predecessor before it reads anything. Each call gets other tokens, so a read of the
    # previous call's routing, schedule or activations would change its output.
    inp, W = inputs(cfg)
    lay = moe().MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))
    g = torch.Generator(device="cuda").manual_seed(cfg.seed + 7)
    xs = [inp["x"]] + [torch.randn(tuple(inp["x"].shape), generator=g, device="cuda")
                       .to(inp["x"].dtype) for _ in range(3)]
    ref = []
    for x in xs:
        ref.append(lay(x).clone())
        torch.cuda.synchronize()
    outs = [torch.empty_like(ref[0]) for _ in xs]
    for x, y in zip(xs, outs):
        lay(x, y)
    torch.cuda.synchronize()
    assert moe().read_status(lay.bufs["ws"]) == 0
    for a, b in zip(outs, ref):
        assert torch.equal(a, b)
    assert not torch.equal(ref[0], ref[1])


@pytest.mark.parametrize("cfg", [SMALL, FP8_SMALL, P2_SMALL, synth.CONFIGS["dsv3_decode"]],
                         ids=lambda c: c.name)
def test_layer_captured_in_a_cuda_graph_replays_like_eager_calls(cfg):
    # The layer enqueues kernel launches only (no allocation, no host sync), so it can be
    # captured once and replayed on new inputs written into the captured buffer; the
    # programmatic launches become programmatic edges of the graph.
    inp, W = inputs(cfg)
    lay = moe().MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))
    x_buf = inp["x"].clone()
    y_buf = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        lay(x_buf, y_buf)   # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        lay(x_buf, y_buf)
    g = torch.Generator(device="cuda").manual_seed(cfg.seed + 11)
    for i in range(3):
        x_new = inp["x"] if i == 0 else torch.randn(
            tuple(inp["x"].shape), generator=g, device="cuda").to(inp["x"].dtype)
        x_buf.copy_(x_new)
        graph.replay()
        torch.cuda.synchronize()
        ref = lay(x_new).clone()
        torch.cuda.synchronize()
        assert torch.equal(y_buf, ref)
    assert moe().read_status(lay.bufs["ws"]) == 0


GUARD = 4096   # canary bytes on each side of a guarded buffer (keeps the 16-byte alignment)


def _guarded(shape, dtype, store):
    """A tensor of the given shape and dtype inside a byte buffer whose first and last GUARD
    bytes hold the canary 0xA5; (buffer, payload bytes) is appended to store for the check."""
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    raw = torch.full((GUARD + n + GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
    store.append((raw, n))
    return raw[GUARD:GUARD + n].view(dtype).view(shape)


@pytest.mark.parametrize("cfg", [synth.CONFIGS["tiny"], SMALL, FP8_SMALL, P2_SMALL, PAIRED],
                         ids=lambda c: c.name)
def test_layer_writes_stay_inside_every_buffer(cfg):
    # Every buffer the layer writes (outputs, receive buffers, metadata, workspace) lies between
    # two guard bands of a canary byte; two layer calls later the bands are untouched.
    inp, W = inputs(cfg)
    m = moe()
    store, bufs = [], {}
    for key, t in m.Buffers(cfg).items():
        bufs[key] = None if t is None else _guarded(tuple(t.shape), t.dtype, store)
    bufs["ws"].zero_()
    y = _guarded((cfg.T, cfg.d), torch.bfloat16, store)
    for _ in range(2):
        m.layer(cfg, inp["x"], inp["w_gate"], inp["bias"], weight_dict(W), bufs, y)
    torch.cuda.synchronize()
    assert m.read_status(bufs["ws"]) == 0
    for raw, n in store:
        assert bool((raw[:GUARD] == 0xA5).all()) and bool((raw[GUARD + n:] == 0xA5).all())
    y_ref = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))(inp["x"])
    assert torch.equal(y, y_ref)


def test_layer_events_are_recorded_in_order():
    cfg = SMALL
    inp, W = inputs(cfg)
    lay = moe().MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(moe().MOE_LAYER_EVENTS)]
    for e in evs:
        e.record()
    torch.cuda.synchronize()
    lay(inp["x"], events=evs)
    torch.cuda.synchronize()
    times = [evs[0].elapsed_time(e) for e in evs]
    assert all(b >= a for a, b in zip(times, times[1:]))


@pytest.mark.parametrize("cfg", [synth.CONFIGS["tiny"], SMALL, ER64], ids=lambda c: c.name)
def test_gate_up_intermediate_and_schedule(cfg):
    """The expert schedule (compact rows expert-major, then source rank, then position) and the
    SwiGLU intermediate h of every compact row, before the down projection."""
    from gpu_util import ws_offsets
    inp, W = inputs(cfg)
    r = _ffn(cfg, inp, W, run_stages(cfg, inp, W))
    o = ws_offsets(cfg)
    ws = r["ws"]
    tk = cfg.T * cfg.k
    grp_n = ws[o["grp_n"]:o["grp_n"] + 4 * cfg.E].view(torch.int32).cpu().numpy()
    grp_off = ws[o["grp_off"]:o["grp_off"] + 4 * cfg.E].view(torch.int32).cpu().numpy()
    row_list = ws[o["row_list"]:o["row_list"] + 4 * tk].view(torch.int32).cpu().numpy()
    counts = r["counts"].cpu().numpy()
    assert np.array_equal(grp_n, counts.sum(0))
    assert np.array_equal(grp_off, np.cumsum(grp_n) - grp_n)
    src = r["src_tok"].cpu().numpy()
    ti = r["topk_idx"].cpu().numpy()
    # expected compact order: expert, then source rank, then token
    exp_rows = []
    for e in range(cfg.E):
        toks = [t for t in range(cfg.T) if e in ti[t]]
        ro = r["row_of"].cpu().numpy()
        exp_rows += [int(ro[t, list(ti[t]).index(e)]) for t in toks]
    assert np.array_equal(row_list, np.array(exp_rows, dtype=np.int32))
    h = ws[o["h"]:o["h"] + 2 * tk * cfg.d_ff].view(torch.bfloat16).view(tk, cfg.d_ff)
    h = bf16_to_f64(host_bits(h))
    x = host_bits(inp["x"])
    get = expert_getter(W, False)
    n_off = n_all = 0
    for e in range(cfg.E):
        Wt = get(e)
        for p in range(grp_n[e]):
            c = grp_off[e] + p
            t = src[row_list[c]]
            _, href = oracle.swiglu_row_bf16(x[t], Wt["w13"], Wt["w2"])
            # h is rounded to bf16 on both sides from sums taken in different orders (fp32
            # here, fp64 in the oracle): elements agree or sit one bf16 ulp apart.
            diff = np.abs(h[c] - href)
            bound = 2.0 ** -7 * np.abs(href) + 1e-6 * np.sqrt(np.mean(href * href))
            assert np.all(diff <= bound), (e, p, t, float((diff / np.maximum(bound, 1e-30)).max()))
            n_off += int((diff > 0).sum())
            n_all += diff.size
    assert n_off <= 0.01 * n_all, (n_off, n_all)


@pytest.mark.parametrize("cfg", [SMALL, HOT, PAIRED, PAIRED_RAGGED], ids=lambda c: c.name)
def test_schedule_lists_multi_tile_groups_first(cfg):
    """The schedule's tile lists (bn-row tiles and, for bf16 layers with 128-row tiles, 2 bn-row
    tiles): each group's rows in consecutive tiles of its own, the groups with two or more tiles
    first and then the one-tile groups, each part in group order, and the word after each
    list's tile count holding the size of its first part (which the GEMMs interleave with the
    second)."""
    from gpu_util import ws_offsets
    inp, W = inputs(cfg)
    r = _ffn(cfg, inp, W, run_stages(cfg, inp, W))
    assert moe().read_status(r["ws"]) == 0
    o = ws_offsets(cfg)
    ws = r["ws"]
    rows = r["counts"].cpu().numpy().sum(0)
    lists = [("n_tiles", "tiles", o["bn"])]
    if o["bn"] == 128 and cfg.act == "bf16":
        lists.append(("n_tiles2", "tiles2", 2 * o["bn"]))
    kinds = set()
    for count_name, list_name, bn in lists:
        head = ws[o[count_name]:o[count_name] + 8].view(torch.int32).cpu().numpy()
        nt = [int((n + bn - 1) // bn) for n in rows]
        multi = [g for g in range(cfg.E) if nt[g] >= 2]
        single = [g for g in range(cfg.E) if nt[g] == 1]
        expect = [(g, j * bn, min(bn, int(rows[g]) - j * bn), nt[g])
                  for g in multi + single for j in range(nt[g])]
        assert int(head[0]) == len(expect), (list_name, head, len(expect))
        assert int(head[1]) == sum(nt[g] for g in multi), (list_name, head)
        got = ws[o[list_name]:o[list_name] + 16 * len(expect)].view(torch.int32).view(-1, 4)
        assert [tuple(int(v) for v in t) for t in got.cpu().numpy()] == expect, list_name
        kinds.add((bool(multi), bool(single)))
    # the configurations reach both kinds together in at least one list
    if cfg.name in ("paired", "paired_ragged", "hot"):
        assert (True, True) in kinds, kinds


# ------------------------------------------------------------------------------------------
# e4m3 path
# ------------------------------------------------------------------------------------------
TOL_FP8 = 6e-2
FP8_HOT = dataclasses.replace(HOT, name="hot_fp8", act="fp8", w="fp8", d=256, d_ff=256,
                              d_ff_shared=256)
# d = 3 x 128: the down projection takes one 128-column output tile per unit (d not a multiple
# of 256), the other shapes two
FP8_ODD = dataclasses.replace(SMALL, name="odd_fp8", act="fp8", w="fp8", d=384, d_ff=256,
                              d_ff_shared=256)


@pytest.mark.parametrize("cfg", [FP8_SMALL, FP8_HOT, FP8_ODD], ids=lambda c: c.name)
def test_fp8_expert_rows_and_layer(cfg):
    inp, W = inputs(cfg)
    m = moe()
    lay = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))
    y = lay(inp["x"])
    assert m.read_status(lay.bufs["ws"]) == 0
    b = lay.bufs
    ti = b["topk_idx"].cpu().numpy()
    ro = b["row_of"].cpu().numpy()
    idx, _ = oracle_route(cfg, inp)
    assert np.array_equal(ti, idx)
    x = host_bits(inp["x"])
    xq, xs = oracle.quant_rows_e4m3(oracle.bf16_to_f32(x))
    get = expert_getter(W, True)
    eb = host_bits(b["ebuf"])
    worst = 0.0
    for e in np.unique(ti):
        Wt = get(int(e))
        for t, i in zip(*np.nonzero(ti == e)):
            ref, _ = oracle.swiglu_row_fp8(xq[t], xs[t], Wt["w13"], Wt["w13_s"], Wt["w2"], Wt["w2_s"])
            worst = max(worst, rel_max_err(bf16_to_f64(eb[ro[t, i]]), bf16_to_f64(ref)))
    assert worst <= TOL_FP8, worst
    S = shared_host(W, True)
    sh = host_bits(b["shared_out"])
    for t in range(0, cfg.T, 7):
        ref, _ = oracle.swiglu_row_fp8(xq[t], xs[t], S["ws13"], S["ws13_s"], S["ws2"], S["ws2_s"])
        assert rel_max_err(bf16_to_f64(sh[t]), bf16_to_f64(ref)) <= TOL_FP8
    assert _layer_tokens_check(cfg, np.arange(cfg.T), inp, W, y) <= TOL_FP8


@pytest.mark.slow
def test_fp8_prefill_rows_and_tokens():
    """The FP8 prefill (T=16384, e4m3 activations and weights): every row of the hottest expert,
    of a <=32-row and a 33..64-row expert where they exist, and of two experts past the first
    1024 compact rows, plus 256 tokens' whole layer output; >= 1024 rows."""
    cfg = synth.CONFIGS["dsv3_fp8_prefill"]
    inp, W, lay, y = _run_layer(cfg)
    rng = np.random.default_rng(cfg.seed)
    extra, hot, n = _prefill_pairs(cfg, lay.bufs, rng)
    tokens = np.sort(np.concatenate([[0, cfg.T - 1],
                                     rng.choice(np.arange(1, cfg.T - 1), 254, replace=False)]))
    res = check_layer(cfg, inp, W, lay.bufs, y, tokens, extra, tol=TOL_FP8)
    print(cfg.name, res)
    assert res["rows"] >= 1024


# ------------------------------------------------------------------------------------------
# e4m3 with power-of-two block scales (the block-scaled MMA's recipe)
# ------------------------------------------------------------------------------------------
P2_HOT = dataclasses.replace(FP8_HOT, name="hot_fp8p2", scales="pow2")
# several k-steps in both GEMMs (d = 4 x 128, d_ff = 3 x 128), ragged token tiles, 4 ranks
P2_WIDE = dataclasses.replace(SMALL, name="wide_fp8p2", act="fp8", w="fp8", scales="pow2",
                              T=200, d=512, d_ff=384, d_ff_shared=384, E=16, k=4, n_group=4,
                              topk_group=2, R=4, seed=91)


def test_dispatch_pow2_codes_and_scales_bit_exact():
    cfg = P2_SMALL
    inp = synth.make_router_inputs(cfg, "cuda")
    m = moe()
    b = m.Buffers(cfg)
    m.route(cfg, inp["x"], inp["w_gate"], inp["bias"], b["topk_idx"], b["topk_w"], b["ws"])
    m.dispatch(cfg, inp["x"], b["topk_idx"], b["recv"], b["recv_scales"], b["counts"],
               b["row_of"], None)
    idx, _ = oracle_route(cfg, inp)
    _, _, row_of, src_tok = oracle.dispatch_index(idx, cfg.E, cfg.R)
    q, sc = oracle.dispatch_payload(host_bits(inp["x"]), row_of, src_tok.size, fp8=True,
                                    pow2=True)
    filled = src_tok >= 0
    assert np.array_equal(b["recv"].cpu().numpy()[filled], q[filled])
    assert np.array_equal(b["recv_scales"].cpu().numpy().T[filled], sc[filled])
    m_, _ = np.frexp(sc[filled])
    assert np.all(m_ == 0.5)


@pytest.mark.parametrize("cfg", [P2_SMALL, P2_HOT, P2_WIDE], ids=lambda c: c.name)
def test_fp8_pow2_expert_rows_and_layer(cfg):
    """Every routed row and every 3rd shared row against the oracle's reading R-l, the whole
    layer output of every token, the gate/up intermediate's codes and scales close to the
    oracle's and its scales powers of two."""
    inp, W = inputs(cfg)
    m = moe()
    lay = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))
    y = lay(inp["x"])
    assert m.read_status(lay.bufs["ws"]) == 0
    b = lay.bufs
    ti = b["topk_idx"].cpu().numpy()
    ro = b["row_of"].cpu().numpy()
    idx, _ = oracle_route(cfg, inp)
    assert np.array_equal(ti, idx)
    xq, xs = oracle.quant_rows_e4m3(oracle.bf16_to_f32(host_bits(inp["x"])), pow2=True)
    get = expert_getter(W, True)
    eb = host_bits(b["ebuf"])
    worst = 0.0
    n = 0
    for e in np.unique(ti):
        Wt = get(int(e))
        for t, i in zip(*np.nonzero(ti == e)):
            ref, _ = oracle.swiglu_row_fp8(xq[t], xs[t], Wt["w13"], Wt["w13_s"], Wt["w2"],
                                           Wt["w2_s"], pow2=True)
            worst = max(worst, rel_max_err(bf16_to_f64(eb[ro[t, i]]), bf16_to_f64(ref)))
            n += 1
    assert n == cfg.T * cfg.k
    assert worst <= TOL_FP8, worst
    S = shared_host(W, True)
    sh = host_bits(b["shared_out"])
    for t in range(0, cfg.T, 3):
        ref, _ = oracle.swiglu_row_fp8(xq[t], xs[t], S["ws13"], S["ws13_s"], S["ws2"], S["ws2_s"],
                                       pow2=True)
        assert rel_max_err(bf16_to_f64(sh[t]), bf16_to_f64(ref)) <= TOL_FP8
    assert _layer_tokens_check(cfg, np.arange(cfg.T), inp, W, y) <= TOL_FP8


@pytest.mark.parametrize("cfg", [P2_SMALL, P2_WIDE], ids=lambda c: c.name)
def test_fp8_pow2_variants_equal_the_layer(cfg):
    """Gather mode, the shared expert on a side stream, a placement and back-to-back calls give
    the pow2 layer's output bit for bit; the amax/448 recipe gives a different one."""
    inp, W = inputs(cfg)
    m = moe()
    y0 = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))(inp["x"]).clone()
    for v in (dict(gather=True), dict(side_stream=True), dict(gather=True, side_stream=True)):
        y = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W), **v)(inp["x"])
        torch.cuda.synchronize()
        assert torch.equal(y, y0), v
    pl, _ = _placement_for(cfg, inp, 2, 31)
    lay = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W), placement=pl)
    assert torch.equal(lay(inp["x"]), y0)
    assert torch.equal(lay(inp["x"]), y0)
    assert m.read_status(lay.bufs["ws"]) == 0
    amax_cfg = dataclasses.replace(cfg, scales="amax")
    W8 = synth.make_expert_weights(amax_cfg, "cuda")
    y8 = m.MoELayer(amax_cfg, inp["w_gate"], inp["bias"], weight_dict(W8))(inp["x"])
    assert not torch.equal(y8, y0)


def _e4m3_step(v, scale):
    """The e4m3 grid spacing at |v| for values quantised with block scale `scale`: 2^(e - 3)
    in binade [2^e, 2^(e+1)) of |v| / scale (e >= -6; the subnormal spacing 2^-9 below)."""
    a = np.abs(v) / scale
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return 2.0 ** (e - 3) * scale


@pytest.mark.parametrize("cfg", [P2_SMALL, P2_WIDE], ids=lambda c: c.name)
def test_fp8_pow2_intermediate_is_the_oracles(cfg):
    """The re-quantised SwiGLU intermediate h of every compact row against the oracle's reading
    R-l: each 128-column block's power-of-two scale (the GPU's scale byte) equals the oracle's
    except where the two sides' amax fall on opposite sides of a binade edge 448 * 2^e (fp32
    sums here, fp64 there), and inside a block with the same scale every element is the
    oracle's or one e4m3 step from it. (An edge crossing re-quantises the whole block at half
    or twice the step, which is why this recipe's outputs sit further from the oracle than
    the amax/448 recipe's.)"""
    from gpu_util import ws_offsets
    inp, W = inputs(cfg)
    r = _ffn(cfg, inp, W, run_stages(cfg, inp, W))
    assert moe().read_status(r["ws"]) == 0
    o = ws_offsets(cfg)
    ws = r["ws"]
    tk, F = cfg.T * cfg.k, cfg.d_ff
    hq = ws[o["h"]:o["h"] + tk * F].view(tk, F).cpu().numpy()
    sfb = ws[o["sf_h"]:o["sf_h"] + 64 * tk].view(tk, 64).cpu().numpy()
    grp_off = ws[o["grp_off"]:o["grp_off"] + 4 * cfg.E].view(torch.int32).cpu().numpy()
    ti = r["topk_idx"].cpu().numpy()
    xq, xs = oracle.quant_rows_e4m3(oracle.bf16_to_f32(host_bits(inp["x"])), pow2=True)
    get = expert_getter(W, True)
    blocks = same = off = n = 0
    for e in range(cfg.E):
        Wt = get(e)
        for p_, t in enumerate([t for t in range(cfg.T) if e in ti[t]]):
            c = grp_off[e] + p_
            _, href = oracle.swiglu_row_fp8(xq[t], xs[t], Wt["w13"], Wt["w13_s"], Wt["w2"],
                                            Wt["w2_s"], pow2=True)
            g_sc = np.ldexp(1.0, sfb[c, :F // 128].astype(np.int64) - 127)
            gdeq = oracle.e4m3_to_f32(hq[c]).astype(np.float64) * np.repeat(g_sc, 128)
            for b in range(F // 128):
                sl = slice(128 * b, 128 * (b + 1))
                ho, hg = href[sl].astype(np.float64), gdeq[sl]
                amax_o = float(np.abs(ho).max())
                blocks += 1
                # the scales differ by at most one binade
                assert amax_o <= 2 * 448.0 * g_sc[b] + 1e-30 and \
                    (amax_o == 0 or amax_o >= 224.0 * g_sc[b] / 2), (e, t, b)
                # the oracle's scale: its quantised amax lies in [224 s, 448 s]
                if amax_o == 0 or 224.0 * g_sc[b] <= amax_o <= 448.0 * g_sc[b]:
                    same += 1
                    d = np.abs(hg - ho)
                    assert np.all(d <= _e4m3_step(np.maximum(np.abs(ho), np.abs(hg)), g_sc[b])
                                  * 1.0001), (e, t, b)
                    off += int((d > 0).sum())
                    n += d.size
    assert same >= 0.97 * blocks, (same, blocks)
    assert off <= 0.05 * n, (off, n)


def test_fp8_pow2_reports_a_weight_scale_that_is_not_a_power_of_two():
    """Weights with one block scale off the power-of-two grid: the GEMM reports MOE_DEV_SCALE
    in the status word and keeps running; the context stays usable."""
    cfg = P2_SMALL
    inp, W = inputs(cfg)
    m = moe()
    Wbad = dict(weight_dict(W))
    Wbad["w13_s"] = W["w13_s"].clone()
    Wbad["w13_s"][:, 0, 0] *= 1.5   # every routed expert's first gate block
    lay = m.MoELayer(cfg, inp["w_gate"], inp["bias"], Wbad)
    lay(inp["x"])
    torch.cuda.synchronize()
    st = m.read_status(lay.bufs["ws"])
    assert st & m.MOE_DEV_SCALE and not st & m.MOE_DEV_TIMEOUT
    ok = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))
    ok(inp["x"])
    assert m.read_status(ok.bufs["ws"]) == 0


@pytest.mark.slow
def test_fp8_pow2_prefill_rows_and_tokens():
    """The FP8 prefill with power-of-two scales (T=16384): every row of the hottest expert, of a
    <=32-row and a 33..64-row expert where they exist, of two experts past the first 1024
    compact rows, and 256 tokens' whole layer output; >= 1024 rows."""
    cfg = synth.CONFIGS["dsv3_fp8_pow2_prefill"]
    inp, W, lay, y = _run_layer(cfg)
    rng = np.random.default_rng(cfg.seed)
    extra, hot, n = _prefill_pairs(cfg, lay.bufs, rng)
    tokens = np.sort(np.concatenate([[0, cfg.T - 1],
                                     rng.choice(np.arange(1, cfg.T - 1), 254, replace=False)]))
    res = check_layer(cfg, inp, W, lay.bufs, y, tokens, extra, tol=TOL_FP8)
    print(cfg.name, res)
    assert res["rows"] >= 1024


# ------------------------------------------------------------------------------------------
# Layer variants: gather mode (no receive-buffer copy) and the shared expert on a side stream
# ------------------------------------------------------------------------------------------
VARIANTS = [dict(gather=True), dict(side_stream=True), dict(gather=True, side_stream=True),
            dict(side_stream=True, side_ctas=3)]


@pytest.mark.parametrize("cfg", [SMALL, FP8_SMALL, HOT, FP8_HOT, synth.CONFIGS["dsv3_decode"],
                                 PAIRED], ids=lambda c: c.name)
def test_layer_variants_equal_the_layer(cfg):
    """Every variant computes the same rows with the same kernels in the same K order, so its
    output equals moe_layer's bit for bit (and the gate weights, indices and counts too)."""
    inp, W = inputs(cfg)
    m = moe()
    base = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))
    y0 = base(inp["x"]).clone()
    torch.cuda.synchronize()
    for v in VARIANTS:
        lay = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W), **v)
        for _ in range(2):   # twice: the second call reuses the workspace and the side stream
            y = lay(inp["x"])
            torch.cuda.synchronize()
            assert m.read_status(lay.bufs["ws"]) == 0, v
            assert torch.equal(y, y0), v
        assert torch.equal(lay.bufs["counts"], base.bufs["counts"])
        assert torch.equal(lay.bufs["row_of"], base.bufs["row_of"])
        if v.get("gather"):
            assert lay.bufs["recv"] is None


@pytest.mark.parametrize("cfg", [SMALL, FP8_SMALL, E192_R64], ids=lambda c: c.name)
def test_gather_stage_calls_equal_the_copying_ones(cfg):
    inp, W = inputs(cfg)
    m = moe()
    r = _ffn(cfg, inp, W, run_stages(cfg, inp, W))
    b = m.Buffers(cfg, with_recv=False)
    st = torch.empty(b.sizes["recv_rows"], dtype=torch.int32, device="cuda")
    m.dispatch_index(cfg, r["topk_idx"], b["counts"], b["row_of"], st)
    assert torch.equal(b["counts"], r["counts"]) and torch.equal(b["row_of"], r["row_of"])
    assert torch.equal(st, r["src_tok"])
    m.expert_ffn_gather(cfg, inp["x"], b["counts"], st, weight_dict(W), b["ebuf"],
                        b["shared_out"], b["ws"])
    torch.cuda.synchronize()
    assert m.read_status(b["ws"]) == 0
    filled = (r["src_tok"] >= 0).nonzero().squeeze(1)
    assert torch.equal(b["ebuf"][filled], r["ebuf"][filled])
    if cfg.d_ff_shared:
        assert torch.equal(b["shared_out"], r["shared_out"])


@pytest.mark.slow
@pytest.mark.parametrize("name", ["dsv3_skew_prefill", "dsv3_fp8_prefill"])
def test_gather_mode_equals_the_layer_at_prefill(name):
    cfg = synth.CONFIGS[name]
    inp, W = inputs(cfg)
    m = moe()
    y0 = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))(inp["x"]).clone()
    lay = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W), gather=True)
    y = lay(inp["x"])
    torch.cuda.synchronize()
    assert m.read_status(lay.bufs["ws"]) == 0
    assert torch.equal(y, y0)


def test_layer_ex_rejects_bad_options():
    import ctypes
    m = moe()
    cfg = SMALL
    inp, W = inputs(cfg)
    b = m.Buffers(cfg)
    y = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.MoEError) as e:   # an unknown flag
        m.layer_ex(cfg, m.LayerOpts(flags=8), inp["x"], inp["w_gate"], inp["bias"],
                   weight_dict(W), b, y)
    assert e.value.code == 1
    with pytest.raises(m.MoEError) as e:   # side stream asked for without a stream or events
        m.layer_ex(cfg, m.LayerOpts(flags=m.MOE_OPT_SHARED_SIDE_STREAM), inp["x"],
                   inp["w_gate"], inp["bias"], weight_dict(W), b, y)
    assert e.value.code == 1
    with pytest.raises(m.MoEError) as e:   # no receive buffer without gather mode
        bb = dict(b)
        bb["recv"] = None
        m.layer_ex(cfg, m.LayerOpts(flags=0), inp["x"], inp["w_gate"], inp["bias"],
                   weight_dict(W), bb, y)
    assert e.value.code == 1


# ------------------------------------------------------------------------------------------
# Redundant experts placed on slots
# ------------------------------------------------------------------------------------------
def _placement_for(cfg, inp, spare_per_rank, seed):
    """A placement planned from the loads of another batch of the same workload (the routing of
    other tokens stands for past traffic), as a deployment would plan it."""
    m = moe()
    other = synth.normal_bf16(cfg.seed + seed, synth.TAG_X, (cfg.T, cfg.d), cfg.x_std, "cuda")
    b = m.Buffers(cfg)
    m.route(cfg, other, inp["w_gate"], inp["bias"], b["topk_idx"], b["topk_w"], b["ws"])
    load = np.bincount(b["topk_idx"].cpu().numpy().reshape(-1), minlength=cfg.E)
    S = cfg.E // cfg.R + spare_per_rank
    return m.Placement.from_loads(load.astype(np.float64), cfg.R, S, max_copies=16), S


PLACED = [(SMALL, 2), (HOT, 3), (E192_R64, 1), (synth.CONFIGS["dsv3_decode"], 4),
          (FP8_SMALL, 2), (PAIRED, 2)]


@pytest.mark.parametrize("cfg,spare", PLACED, ids=lambda v: getattr(v, "name", str(v)))
def test_placed_layer_dispatch_is_the_oracles_and_output_is_the_layers(cfg, spare):
    inp, W = inputs(cfg)
    m = moe()
    pl, S = _placement_for(cfg, inp, spare, 31)
    y0 = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))(inp["x"]).clone()
    for gather in (False, True):
        lay = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W), placement=pl,
                         gather=gather)
        y = lay(inp["x"])
        torch.cuda.synchronize()
        assert m.read_status(lay.bufs["ws"]) == 0
        ti = lay.bufs["topk_idx"].cpu().numpy()
        counts, row_of, _ = oracle.dispatch_index_placed(
            ti, cfg.E, cfg.R, S, pl.n_copies.cpu().numpy(), pl.copy_slot.cpu().numpy())
        assert np.array_equal(lay.bufs["counts"].cpu().numpy(), counts)
        assert np.array_equal(lay.bufs["row_of"].cpu().numpy(), row_of)
        # the same rows through the same weights: the output equals the unplaced layer's
        assert torch.equal(y, y0)


@pytest.mark.slow
def test_placed_skew_prefill_lowers_the_imbalance_and_keeps_the_output():
    cfg = synth.CONFIGS["dsv3_skew_prefill"]
    inp, W = inputs(cfg)
    m = moe()
    pl, S = _placement_for(cfg, inp, 4, 17)
    base = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))
    y0 = base(inp["x"]).clone()
    lay = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W), placement=pl)
    y = lay(inp["x"])
    torch.cuda.synchronize()
    assert m.read_status(lay.bufs["ws"]) == 0
    assert torch.equal(y, y0)
    ti = lay.bufs["topk_idx"].cpu().numpy()
    counts, row_of, _ = oracle.dispatch_index_placed(
        ti, cfg.E, cfg.R, S, pl.n_copies.cpu().numpy(), pl.copy_slot.cpu().numpy())
    assert np.array_equal(lay.bufs["counts"].cpu().numpy(), counts)
    assert np.array_equal(lay.bufs["row_of"].cpu().numpy(), row_of)
    before = oracle.imbalance_factor(np.bincount(ti.reshape(-1), minlength=cfg.E), cfg.R)
    loads = oracle.rank_loads(counts, cfg.R)
    after = loads.max() / loads.mean()
    print("skew prefill rank IF: contiguous %.3f, placed %.3f" % (before, after))
    assert after < before and after < 1.1


# ------------------------------------------------------------------------------------------
# The fused expert stage: both GEMMs and the combine in one persistent launch (bf16)
# ------------------------------------------------------------------------------------------
FUSED_CFGS = [synth.CONFIGS["tiny"], SMALL, HOT, ER64, E192_R64,
              synth.CONFIGS["dsv3_sweep"].with_T(8), synth.CONFIGS["dsv3_decode"],
              synth.CONFIGS["dsv3_sweep"].with_T(256)]


@pytest.mark.parametrize("cfg", FUSED_CFGS, ids=lambda c: c.name)
def test_fused_expert_stage_equals_the_layer(cfg):
    """The same rows through the same GEMM units and the combine's arithmetic: bit for bit the
    output of moe_layer, alone and with gather mode, on three calls in a row (the dependency
    counters are reset by every call)."""
    inp, W = inputs(cfg)
    m = moe()
    y0 = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))(inp["x"]).clone()
    torch.cuda.synchronize()
    for v in (dict(fused=True), dict(fused=True, gather=True)):
        lay = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W), **v)
        for _ in range(3):
            y = lay(inp["x"])
        torch.cuda.synchronize()
        assert m.read_status(lay.bufs["ws"]) == 0, v
        assert torch.equal(y, y0), v


def test_fused_expert_stage_with_placed_experts_and_events():
    cfg = synth.CONFIGS["dsv3_decode"]
    inp, W = inputs(cfg)
    m = moe()
    y0 = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))(inp["x"]).clone()
    pl, _ = _placement_for(cfg, inp, 4, 31)
    lay = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W), placement=pl, fused=True,
                     gather=True)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(m.MOE_LAYER_EVENTS)]
    for e in evs:
        e.record()
    y = lay(inp["x"], events=evs)
    torch.cuda.synchronize()
    assert m.read_status(lay.bufs["ws"]) == 0
    assert torch.equal(y, y0)
    times = [evs[0].elapsed_time(e) for e in evs]
    assert all(b >= a for a, b in zip(times, times[1:]))


def test_fused_back_to_back_and_in_a_cuda_graph():
    cfg = SMALL
    inp, W = inputs(cfg)
    m = moe()
    lay = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W), fused=True, gather=True)
    ref = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))
    g = torch.Generator(device="cuda").manual_seed(5)
    xs = [torch.randn(tuple(inp["x"].shape), generator=g, device="cuda").to(inp["x"].dtype)
          for _ in range(3)]
    outs = [lay(x).clone() for x in xs]          # queued back to back, no synchronisation
    torch.cuda.synchronize()
    for x, y in zip(xs, outs):
        assert torch.equal(y, ref(x))
    x_buf = xs[0].clone()
    y_buf = torch.empty_like(outs[0])
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        lay(x_buf, y_buf)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        lay(x_buf, y_buf)
    for x in xs:
        x_buf.copy_(x)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(y_buf, ref(x))
    assert m.read_status(lay.bufs["ws"]) == 0


def test_fused_rejects_fp8_and_the_side_stream():
    m = moe()
    inp, W = inputs(FP8_SMALL)
    with pytest.raises(m.MoEError) as e:
        m.MoELayer(FP8_SMALL, inp["w_gate"], inp["bias"], weight_dict(W), fused=True)(inp["x"])
    assert e.value.code == 2
    inp, W = inputs(SMALL)
    with pytest.raises(m.MoEError) as e:
        m.MoELayer(SMALL, inp["w_gate"], inp["bias"], weight_dict(W), fused=True,
                   side_stream=True)(inp["x"])
    assert e.value.code == 1
