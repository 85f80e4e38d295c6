"""Pins of the CPU oracle against things other than itself: library conversions, error bounds,
brute force on tiny inputs, invariants, textbook special cases and values printed on the pages.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _ulp32(x):
    x = np.abs(np.asarray(x, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(x, np.finfo(np.float32).tiny)))
    return np.exp2(e - 23)


# ------------------------------------------------------------------------------------------
# Number formats
# ------------------------------------------------------------------------------------------
def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    v = rng.standard_normal(200000).astype(np.float32) * np.float32(3.0)
    # exact ties: bf16 value plus half an ulp, both parities
    base = torch.from_numpy(v[:1000]).to(torch.bfloat16).float().numpy()
    ties = (base.view(np.uint32) + np.uint32(0x8000)).view(np.float32)
    v = np.concatenate([v, ties, np.float32([0.0, -0.0, 1e-40, -1e-40, 3.4e38])])
    ours = oracle.f32_to_bf16(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f32(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert nan.sum() == 2 and ours[0x7e] == 448.0 and ours[0x01] == 2.0 ** -9


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(2)
    v = np.concatenate([
        rng.uniform(-448, 448, 100000), rng.standard_normal(100000) * 0.01,
        rng.standard_normal(50000) * 1e-3]).astype(np.float32)
    # midpoints between neighbouring finite codes exercise ties-to-even
    vals = np.sort(oracle.e4m3_to_f32(np.arange(0, 0x7f, dtype=np.uint8)))
    mids = ((vals[1:].astype(np.float64) + vals[:-1]) / 2).astype(np.float32)
    v = np.concatenate([v, mids, -mids, np.float32([0.0, -0.0, 448.0, -448.0])])
    ours = oracle.f32_to_e4m3(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_saturates_and_round_trips():
    big = np.float32([449.0, 464.0, 1e6, -500.0, np.inf, -np.inf])
    q = oracle.f32_to_e4m3(big)
    assert list(q) == [0x7e, 0x7e, 0x7e, 0xfe, 0x7e, 0xfe]
    finite = np.array([c for c in range(256) if (c & 0x7f) != 0x7f], dtype=np.uint8)
    assert np.array_equal(oracle.f32_to_e4m3(oracle.e4m3_to_f32(finite)), finite)


def test_exp_within_two_ulp_of_fp64():
    z = np.linspace(-87.0, 87.0, 400001, dtype=np.float64).astype(np.float32)
    ours = oracle.exp(z).astype(np.float64)
    ref = np.exp(z.astype(np.float64))
    err = np.abs(ours - ref) / _ulp32(ref)
    assert err.max() <= 2.0, err.max()
    assert oracle.exp(np.float32([0.0]))[0] == 1.0


def test_sigmoid_within_three_ulp_of_fp64():
    z = np.linspace(-30.0, 30.0, 200001).astype(np.float32)
    ours = oracle.sigmoid(z).astype(np.float64)
    ref = 1.0 / (1.0 + np.exp(-z.astype(np.float64)))
    err = np.abs(ours - ref) / _ulp32(ref)
    assert err.max() <= 3.0, err.max()
    assert oracle.sigmoid(np.float32([0.0]))[0] == 0.5


# ------------------------------------------------------------------------------------------
# Router: logits, selection, weights
# ------------------------------------------------------------------------------------------
def test_logit_within_fp32_dot_error_bound():
    cfg = synth.CONFIGS["dsv3_decode"]
    x = synth.bf16_bits(synth.normal_bf16(11, synth.TAG_X, (4, cfg.d), 1.0))
    w = synth.normal_f32(11, synth.TAG_WGATE, (8, cfg.d), 0.02).numpy()
    u = 2.0 ** -24
    gamma = cfg.d * u / (1 - cfg.d * u)
    xf = oracle.bf16_to_f32(x).astype(np.float64)
    for t in range(4):
        for e in range(8):
            z = oracle.logit(x[t], w[e])
            ref = float(xf[t] @ w[e].astype(np.float64))
            assert abs(z - ref) <= gamma * float(np.abs(xf[t] * w[e]).sum()) + 1e-30


def test_logit_picks_the_right_operands():
    d = 256
    w = np.arange(d, dtype=np.float32) * np.float32(0.5) + np.float32(1.0)
    for j in (0, 15, 16, 100, 255):       # one-hot x selects one weight exactly
        x = np.zeros(d, dtype=np.float32)
        x[j] = 1.0
        assert oracle.logit(oracle.f32_to_bf16(x), w) == w[j]
    ones = oracle.f32_to_bf16(np.ones(d, dtype=np.float32))
    assert oracle.logit(ones, np.full(d, 0.25, dtype=np.float32)) == 64.0


def _brute_force_route(s, bias, k, n_group, topk_group, scale):
    """Selection by enumeration: the kept groups and chosen experts are the unique subsets
    whose every member ranks before every non-member ((key desc, index asc) order)."""
    E = s.size
    gs = E // n_group
    v = (s + bias).astype(np.float32)

    def before(a, ia, b, ib):
        return a > b or (a == b and ia < ib)

    gscore = []
    for g in range(n_group):
        vals = sorted(v[g * gs:(g + 1) * gs].tolist(), reverse=True)
        gscore.append(np.float32(vals[0]) + np.float32(vals[1]) if gs > 1 else np.float32(vals[0]))
    kept = [S for S in itertools.combinations(range(n_group), topk_group)
            if all(before(gscore[a], a, gscore[b], b)
                   for a in S for b in range(n_group) if b not in S)]
    assert len(kept) == 1
    elig = [e for e in range(E) if e // gs in kept[0]]
    chosen = [S for S in itertools.combinations(elig, k)
              if all(before(v[a], a, v[b], b) for a in S for b in elig if b not in S)]
    assert len(chosen) == 1
    order = sorted(chosen[0], key=lambda e: (-float(v[e]), e))
    tot = np.float32(0.0)
    for e in order:
        tot = np.float32(tot + s[e])
    w = [np.float32(np.float32(s[e] / tot) * np.float32(scale)) for e in order]
    return order, w


@pytest.mark.parametrize("E,k,n_group,topk_group", [(8, 3, 4, 2), (16, 4, 4, 2), (12, 2, 3, 1),
                                                    (16, 5, 8, 3), (10, 3, 1, 1)])
def test_route_matches_brute_force(E, k, n_group, topk_group):
    d = 64
    for seed in range(6):
        x = synth.bf16_bits(synth.normal_bf16(seed, synth.TAG_X, (5, d), 1.0))
        wg = synth.normal_f32(seed, synth.TAG_WGATE, (E, d), 0.1).numpy()
        b = synth.uniform_sym_f32(seed, synth.TAG_BIAS, E, 0.3).numpy()
        if seed == 5:   # force exact ties: duplicate gate rows and bias
            wg[E - 1] = wg[0]
            b[E - 1] = b[0]
            wg[1] = wg[2]
            b[1] = b[2]
        idx, w, z, s = oracle.route(x, wg, b, k, n_group, topk_group, 2.5, want_scores=True)
        for t in range(5):
            order, ww = _brute_force_route(s[t], b, k, n_group, topk_group, 2.5)
            assert list(idx[t]) == order
            assert np.array_equal(w[t], np.array(ww, dtype=np.float32))


def test_route_single_group_is_plain_topk_and_weights_sum_to_scale():
    cfg = synth.CONFIGS["tiny"]
    inp = synth.make_router_inputs(cfg)
    x = synth.bf16_bits(inp["x"])
    idx, w, z, s = oracle.route(x, inp["w_gate"].numpy(), inp["bias"].numpy(), cfg.k, 1, 1,
                                cfg.route_scale, want_scores=True)
    v = s + inp["bias"].numpy()
    for t in range(cfg.T):
        ref = np.lexsort((np.arange(cfg.E), -v[t]))[:cfg.k]   # independent sort
        assert list(idx[t]) == list(ref)
    assert np.allclose(w.sum(1), cfg.route_scale, rtol=1e-6, atol=0)
    # the bias steers selection: a large bias forces an expert in for every token
    b2 = inp["bias"].numpy().copy()
    b2[5] = 10.0
    idx2, _ = oracle.route(x, inp["w_gate"].numpy(), b2, cfg.k, 1, 1, 1.0)
    assert (idx2[:, 0] == 5).all()


def test_route_weights_use_raw_scores_not_bias():
    d, E = 32, 8
    x = synth.bf16_bits(synth.normal_bf16(3, synth.TAG_X, (3, d), 1.0))
    wg = synth.normal_f32(3, synth.TAG_WGATE, (E, d), 0.1).numpy()
    b0 = np.zeros(E, dtype=np.float32)
    b1 = np.full(E, 0.05, dtype=np.float32)      # uniform shift: same selection, same weights
    i0, w0 = oracle.route(x, wg, b0, 2, 1, 1, 1.0)
    i1, w1 = oracle.route(x, wg, b1, 2, 1, 1, 1.0)
    assert np.array_equal(i0, i1) and np.array_equal(w0, w1)


def test_route_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oracle.route(np.zeros((1, 24), np.uint16), np.zeros((8, 24), np.float32),
                     np.zeros(8, np.float32), 2, 1, 1, 1.0)      # d % 16 != 0
    with pytest.raises(ValueError):
        oracle.route(np.zeros((1, 32), np.uint16), np.zeros((8, 32), np.float32),
                     np.zeros(8, np.float32), 5, 4, 2, 1.0)      # k > topk_group * E/n_group


# ------------------------------------------------------------------------------------------
# Dispatch
# ------------------------------------------------------------------------------------------
def _random_topk(T, E, k, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,k,R", [(16, 16, 2, 2), (24, 12, 3, 4), (64, 256, 8, 8), (8, 8, 8, 8),
                                     (6, 4, 1, 1)])
def test_dispatch_index_matches_sorted_enumeration(T, E, k, R):
    ti = _random_topk(T, E, k, T * 7 + E)
    counts, offsets, row_of, src_tok = oracle.dispatch_index(ti, E, R)
    Ts, Er = T // R, E // R
    cap = Ts * min(k, Er)
    # enumeration: sort (dest rank, source rank, expert, token) and lay rows out segment by segment
    entries = sorted(((int(e) // Er, t // Ts, int(e), t, i) for t in range(T)
                      for i, e in enumerate(ti[t])))
    fill = {}
    for r, s, e, t, i in entries:
        n = fill.get((r, s), 0)
        assert row_of[t, i] == (r * R + s) * cap + n
        fill[(r, s)] = n + 1
    # invariants
    assert counts.sum() == T * k
    assert len(set(row_of.reshape(-1).tolist())) == T * k            # injective
    for t in range(T):
        for i in range(k):
            assert src_tok[row_of[t, i]] == t
    assert (src_tok >= 0).sum() == T * k
    assert max(fill.values()) <= cap
    # per-destination send counts equal a bincount of destination ranks per source
    for s in range(R):
        dst = (ti[s * Ts:(s + 1) * Ts].reshape(-1) // Er)
        assert np.array_equal(counts[s].reshape(R, Er).sum(1), np.bincount(dst, minlength=R))
    # offsets are exclusive sums inside each destination rank
    for s in range(R):
        for r in range(R):
            c = counts[s, r * Er:(r + 1) * Er]
            assert np.array_equal(offsets[s, r * Er:(r + 1) * Er], np.cumsum(c) - c)


def test_dispatch_payload_bf16_and_fp8():
    T, d, E, k, R = 16, 256, 16, 2, 2
    x = synth.bf16_bits(synth.normal_bf16(5, synth.TAG_X, (T, d), 1.0))
    ti = _random_topk(T, E, k, 9)
    _, _, row_of, src_tok = oracle.dispatch_index(ti, E, R)
    n_rows = src_tok.size
    recv, _ = oracle.dispatch_payload(x, row_of, n_rows)
    for r in range(n_rows):
        if src_tok[r] >= 0:
            assert np.array_equal(recv[r], x[src_tok[r]])
    q, sc = oracle.dispatch_payload(x, row_of, n_rows, fp8=True)
    xf = oracle.bf16_to_f32(x)
    for t in range(T):
        blk = xf[t].reshape(d // 128, 128)
        scale = (np.abs(blk).max(1) / np.float32(448.0)).astype(np.float32)
        ref = torch.from_numpy((blk / scale[:, None]).astype(np.float32)).to(
            torch.float8_e4m3fn).view(torch.uint8).numpy().reshape(-1)
        for i in range(k):
            assert np.array_equal(q[row_of[t, i]], ref)
            assert np.array_equal(sc[row_of[t, i]], scale)


def _is_pow2_scale_of(amax, scale):
    """Reading R-l's defining properties: scale = 2^e, -126 <= e <= 127, amax <= 448 * 2^e, and
    no smaller power of two would do (or e is at its floor); 1 for amax 0."""
    amax, scale = float(amax), float(scale)
    if amax == 0.0:
        return scale == 1.0
    m, e = math.frexp(scale)           # scale = m * 2^e, m in [0.5, 1)
    if m != 0.5 or not (-126 <= e - 1 <= 127):
        return False
    return amax <= 448.0 * scale and (e - 1 == -126 or amax > 224.0 * scale)


def test_pow2_scale_definition_at_block_boundaries():
    """The power-of-two scale at and around the edges of each binade of 448 * 2^e, at zero, for
    fp32 subnormals and near the top of the range; the generator's independent torch form
    (log2 estimate + exact corrections) gives the same scales."""
    vals = [0.0, 1e-45, 1e-40, 1.17e-38, 1e-20, 0.001, 1.0, 3.0, 447.99, 448.0, 448.00003, 500.0,
            896.0, 1e6, 3e38]
    for k in range(-130, 120, 7):
        b = np.float32(448.0 * 2.0 ** k) if 448.0 * 2.0 ** k < 3.4e38 else None
        if b is None or b == 0:
            continue
        vals += [float(b), float(np.nextafter(b, np.float32(np.inf))),
                 float(np.nextafter(b, np.float32(0)))]
    amax = np.asarray(vals, dtype=np.float32)
    got = np.array([oracle.pow2_scale(a) for a in amax], dtype=np.float32)
    for a, sc in zip(amax, got):
        assert _is_pow2_scale_of(a, sc), (a, sc)
    ref = synth.pow2_block_scale(torch.from_numpy(amax)).numpy()
    assert np.array_equal(got, ref)
    # 448 * 2^k itself takes 2^k; one step above it takes 2^(k+1)
    assert oracle.pow2_scale(np.float32(448.0)) == 1.0
    assert oracle.pow2_scale(np.nextafter(np.float32(448.0), np.float32(1e9))) == 2.0


def test_quant_pow2_rows_and_payload():
    """Reading R-l on rows: every block's scale has the defining properties, the codes are
    torch's e4m3 conversion of value / scale (exact division), nothing saturates, and the
    dispatch payload carries the same codes and scales."""
    T, d, E, k, R = 16, 512, 16, 2, 2
    x = synth.bf16_bits(synth.normal_bf16(5, synth.TAG_X, (T, d), 1.0))
    xf = oracle.bf16_to_f32(x)
    xf[3, :128] *= 1e-30          # a block with a tiny amax
    xf[4, 128:256] = 0.0           # an all-zero block
    q, sc = oracle.quant_rows_e4m3(xf, pow2=True)
    for t in range(T):
        blk = xf[t].reshape(d // 128, 128)
        amax = np.abs(blk).max(1)
        for b in range(d // 128):
            assert _is_pow2_scale_of(amax[b], sc[t, b])
        v = (blk / sc[t][:, None]).astype(np.float32)
        assert np.all(np.abs(v) <= 448.0)
        assert np.array_equal(v * sc[t][:, None], blk)   # the division by 2^e was exact
        ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy().reshape(-1)
        assert np.array_equal(q[t], ref)
    # the amax/448 recipe differs from it on these rows
    q0, sc0 = oracle.quant_rows_e4m3(xf)
    assert not np.array_equal(sc0, sc)
    ti = _random_topk(T, E, k, 9)
    _, _, row_of, src_tok = oracle.dispatch_index(ti, E, R)
    xb = oracle.f32_to_bf16(xf)
    q2, s2 = oracle.quant_rows_e4m3(oracle.bf16_to_f32(xb), pow2=True)
    recv, rsc = oracle.dispatch_payload(xb, row_of, src_tok.size, fp8=True, pow2=True)
    for t in range(T):
        for i in range(k):
            assert np.array_equal(recv[row_of[t, i]], q2[t])
            assert np.array_equal(rsc[row_of[t, i]], s2[t])


# ------------------------------------------------------------------------------------------
# Experts and combine
# ------------------------------------------------------------------------------------------
def _torch_swiglu(x, w13, w2, F):
    """Dense SwiGLU MLP in fp64 torch ops with the same bf16 rounding points."""
    g = x @ w13[:F].T
    u = x @ w13[F:].T
    h = (torch.nn.functional.silu(g) * u).float().to(torch.bfloat16).double()
    return (h @ w2.T).float().to(torch.bfloat16), h


def test_swiglu_bf16_is_a_dense_mlp_when_one_expert():
    d, F = 256, 128
    x = synth.normal_bf16(7, synth.TAG_X, (6, d), 1.0)
    w13 = synth.normal_bf16(7, synth.TAG_W13, (2 * F, d), 0.05)
    w2 = synth.normal_bf16(7, synth.TAG_W2, (d, F), 0.05)
    ref, href = _torch_swiglu(x.double(), w13.double(), w2.double(), F)
    ref = synth.bf16_bits(ref)
    mism = 0
    for t in range(6):
        out, h = oracle.swiglu_row_bf16(synth.bf16_bits(x[t]), synth.bf16_bits(w13), synth.bf16_bits(w2))
        assert np.allclose(h, href[t].numpy(), rtol=2 ** -8, atol=0)
        diff = np.abs(out.astype(np.int32) - ref[t].astype(np.int32))
        assert diff.max() <= 1
        mism += int((diff > 0).sum())
    assert mism <= 3


def test_swiglu_bf16_exact_output_is_the_unrounded_down_projection():
    """The fp64 output before rounding: the fp64 torch down projection of the same bf16 h (the
    sums agree to fp64 rounding order), and its rounding (fp64 -> fp32 -> bf16) is the bf16
    output bit for bit."""
    d, F = 256, 128
    x = synth.normal_bf16(8, synth.TAG_X, (4, d), 1.0)
    w13 = synth.normal_bf16(8, synth.TAG_W13, (2 * F, d), 0.05)
    w2 = synth.normal_bf16(8, synth.TAG_W2, (d, F), 0.05)
    for t in range(4):
        out, h, ox = oracle.swiglu_row_bf16(synth.bf16_bits(x[t]), synth.bf16_bits(w13),
                                            synth.bf16_bits(w2), exact=True)
        ref = (torch.from_numpy(h.astype(np.float64)) @ w2.double().T).numpy()
        assert np.allclose(ox, ref, rtol=1e-12, atol=1e-12)
        rounded = torch.from_numpy(ox).float().to(torch.bfloat16).view(torch.int16).numpy()
        assert np.array_equal(rounded.view(np.uint16), out)


def test_swiglu_bf16_gate_and_up_are_not_swapped():
    d, F = 128, 128
    x = np.full(d, 0x3f80, dtype=np.uint16)            # ones
    w13 = np.zeros((2 * F, d), dtype=np.uint16)
    w13[:F] = 0x3f80      # gate rows: 1.0 -> g = d
    w13[F:] = 0x0000      # up rows: 0 -> h = 0 regardless of g
    w2 = np.full((d, F), 0x3f80, dtype=np.uint16)
    out, h = oracle.swiglu_row_bf16(x, w13, w2)
    assert not h.any() and not out.any()
    w13[:F], w13[F:] = 0, 0x3f80                        # gate 0 -> silu(0) = 0
    out, h = oracle.swiglu_row_bf16(x, w13, w2)
    assert not h.any()


def test_swiglu_fp8_matches_torch_dequantised_mlp():
    cfg = synth.MoEConfig("t", T=4, d=256, E=2, k=1, n_group=1, topk_group=1, d_ff=256,
                          d_ff_shared=0, R=1, route_scale=1.0, act="fp8", w="fp8", seed=3)
    W = synth.expert_weight_slice(cfg, 1)
    x = synth.normal_bf16(3, synth.TAG_X, (4, cfg.d), 1.0)
    xq, xs = oracle.quant_rows_e4m3(oracle.bf16_to_f32(synth.bf16_bits(x)))
    F, d = cfg.d_ff, cfg.d

    def deq(q, s):
        v = torch.from_numpy(q.numpy() if torch.is_tensor(q) else q).view(torch.float8_e4m3fn).double()
        s = torch.as_tensor(s).double()
        return v * s.repeat_interleave(128, 0).repeat_interleave(128, 1)

    w13 = deq(W["w13"], W["w13_s"])
    w2 = deq(W["w2"], W["w2_s"])
    for t in range(4):
        xv = torch.from_numpy(xq[t]).view(torch.float8_e4m3fn).double() * \
            torch.from_numpy(xs[t]).double().repeat_interleave(128)
        g = w13[:F] @ xv
        u = w13[F:] @ xv
        hf = (torch.nn.functional.silu(g) * u).float()
        blk = hf.view(F // 128, 128)
        sc = blk.abs().amax(1) / 448.0
        hq = (blk / sc[:, None]).to(torch.float8_e4m3fn).double() * sc[:, None].double()
        ref = (w2 @ hq.reshape(-1)).float()
        out, h, ox = oracle.swiglu_row_fp8(xq[t], xs[t], W["w13"].numpy(), W["w13_s"].numpy(),
                                           W["w2"].numpy(), W["w2_s"].numpy(), exact=True)
        o = oracle.bf16_to_f32(out)
        assert np.abs(o - ref.numpy()).max() <= 2 ** -7 * np.abs(ref.numpy()).max() + 1e-6
        # the unrounded output: the fp64 down projection of the oracle's own dequantised h,
        # which rounds to the bf16 output
        assert np.allclose(ox, (w2 @ torch.from_numpy(h.astype(np.float64))).numpy(),
                           rtol=1e-12, atol=1e-12)
        rounded = torch.from_numpy(ox).float().to(torch.bfloat16).view(torch.int16).numpy()
        assert np.array_equal(rounded.view(np.uint16), out)


def test_swiglu_fp8_pow2_matches_torch_dequantised_mlp():
    """Reading R-l through one expert: power-of-two weight block scales from the generator and
    the intermediate re-quantised with power-of-two scales, against fp64 torch."""
    cfg = synth.MoEConfig("t", T=4, d=256, E=2, k=1, n_group=1, topk_group=1, d_ff=256,
                          d_ff_shared=0, R=1, route_scale=1.0, act="fp8", w="fp8",
                          scales="pow2", seed=3)
    W = synth.expert_weight_slice(cfg, 1)
    for s_ in (W["w13_s"], W["w2_s"]):
        m, _ = np.frexp(s_.numpy())
        assert np.all(m == 0.5)
    x = synth.normal_bf16(3, synth.TAG_X, (4, cfg.d), 1.0)
    xq, xs = oracle.quant_rows_e4m3(oracle.bf16_to_f32(synth.bf16_bits(x)), pow2=True)
    F = cfg.d_ff

    def deq(q, s):
        v = torch.from_numpy(q.numpy()).view(torch.float8_e4m3fn).double()
        s = torch.as_tensor(s).double()
        return v * s.repeat_interleave(128, 0).repeat_interleave(128, 1)

    w13 = deq(W["w13"], W["w13_s"])
    w2 = deq(W["w2"], W["w2_s"])
    for t in range(4):
        xv = torch.from_numpy(xq[t]).view(torch.float8_e4m3fn).double() * \
            torch.from_numpy(xs[t]).double().repeat_interleave(128)
        hf = (torch.nn.functional.silu(w13[:F] @ xv) * (w13[F:] @ xv)).float()
        blk = hf.view(F // 128, 128)
        sc = synth.pow2_block_scale(blk.abs().amax(1))
        for b in range(F // 128):
            assert _is_pow2_scale_of(blk[b].abs().max().item(), sc[b].item())
        hq = (blk / sc[:, None]).to(torch.float8_e4m3fn).double() * sc[:, None].double()
        ref = (w2 @ hq.reshape(-1)).float()
        out, h = oracle.swiglu_row_fp8(xq[t], xs[t], W["w13"].numpy(), W["w13_s"].numpy(),
                                       W["w2"].numpy(), W["w2_s"].numpy(), pow2=True)
        assert np.abs(oracle.bf16_to_f32(out) - ref.numpy()).max() <= \
            2 ** -7 * np.abs(ref.numpy()).max() + 1e-6
        assert np.allclose(h, hq.reshape(-1).float().numpy(), rtol=0, atol=0)


def test_combine_identity_experts_return_scaled_x():
    """Dispatch followed by identity experts and the combine gives route_scale * x."""
    cfg = synth.CONFIGS["tiny"]
    inp = synth.make_router_inputs(cfg)
    x = synth.bf16_bits(inp["x"])
    idx, w = oracle.route(x, inp["w_gate"].numpy(), inp["bias"].numpy(), cfg.k, cfg.n_group,
                          cfg.topk_group, 1.75)
    _, _, row_of, src_tok = oracle.dispatch_index(idx, cfg.E, cfg.R)
    recv, _ = oracle.dispatch_payload(x, row_of, src_tok.size)
    y = oracle.combine(recv, row_of, w)
    ref = oracle.bf16_to_f32(x).astype(np.float64) * 1.75
    yf = oracle.bf16_to_f32(y)
    assert np.all(np.abs(yf - ref) <= 2 ** -8 * np.abs(ref) + 1e-30)


def test_combine_matches_numpy_weighted_sum():
    rng = np.random.default_rng(4)
    T, d, k, n = 5, 128, 3, 20
    eb = oracle.f32_to_bf16(rng.standard_normal((n, d)).astype(np.float32))
    sh = oracle.f32_to_bf16(rng.standard_normal((T, d)).astype(np.float32))
    ro = rng.permutation(n)[:T * k].reshape(T, k).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    y = oracle.combine(eb, ro, w, sh)
    ref = np.einsum("tk,tkd->td", w.astype(np.float64), oracle.bf16_to_f32(eb)[ro].astype(np.float64))
    ref += oracle.bf16_to_f32(sh)
    refb = torch.from_numpy(ref).float().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.abs(y.astype(np.int32) - refb.astype(np.int32)).max() <= 1
    # the unrounded sums: numpy's fp64 weighted sum (to fp64 rounding order), rounding to y
    y2, yx = oracle.combine(eb, ro, w, sh, exact=True)
    assert np.array_equal(y2, y)
    assert np.allclose(yx, ref, rtol=1e-13, atol=1e-13)
    rounded = torch.from_numpy(yx).float().to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(rounded.view(np.uint16), y)


# ------------------------------------------------------------------------------------------
# The pages' metrics
# ------------------------------------------------------------------------------------------
def test_imbalance_factor_exercise_three():
    g = _golden("exercise3_imbalance.json")
    c = np.array(g["expert_counts"])
    assert oracle.imbalance_factor(c, g["G"]) == g["imbalance_factor"]
    assert list(c.reshape(g["G"], -1).sum(1)) == g["rank_loads"]


def test_imbalance_factor_demo_ranges():
    g = _golden("skew_demo.json")
    rng = np.random.default_rng(12)
    E, G, T, k = g["E"], g["G"], g["T"], g["k"]
    uni = np.bincount(rng.integers(0, E, size=T * k), minlength=E)
    assert 1.0 <= oracle.imbalance_factor(uni, G) <= 1.15
    p = np.ones(E)
    p[g["hot_experts"]] *= g["hot_weight"]
    p /= p.sum()
    sk = np.bincount(rng.choice(E, size=T * k, p=p), minlength=E)
    assert oracle.imbalance_factor(sk, G) > g["skewed_if_above"]


def test_distinct_experts_closed_form():
    g = _golden("distinct_experts.json")
    E, k, B = g["E"], g["k"], g["B"]
    closed = E * (1 - (1 - k / E) ** B)
    assert round(closed) == g["printed_value"]
    assert abs(closed / E - g["printed_fraction"]) < 0.005
    trials = [oracle.distinct_experts(_random_topk(B, E, k, 100 + s)) for s in range(64)]
    assert abs(np.mean(trials) - closed) <= 3 * 4.58 / math.sqrt(64)


def test_router_touches_about_the_closed_form_count():
    """With no bias, sigmoid routing on random weights is uniform over experts, so a batch of
    64 touches about E(1-(1-k/E)^B) = 222 experts. With the workload's U(-0.1, 0.1) bias the
    bias dominates the near-saturated top scores and fewer experts are touched."""
    cfg = synth.CONFIGS["dsv3_decode"]
    inp = synth.make_router_inputs(cfg)
    x = synth.bf16_bits(inp["x"])
    closed = cfg.E * (1 - (1 - cfg.k / cfg.E) ** cfg.T)
    idx0, _ = oracle.route(x, inp["w_gate"].numpy(), np.zeros(cfg.E, np.float32), cfg.k,
                           cfg.n_group, cfg.topk_group, cfg.route_scale)
    assert abs(oracle.distinct_experts(idx0) - closed) <= 0.1 * closed
    idx, _ = oracle.route(x, inp["w_gate"].numpy(), inp["bias"].numpy(), cfg.k, cfg.n_group,
                          cfg.topk_group, cfg.route_scale)
    assert oracle.distinct_experts(idx) < oracle.distinct_experts(idx0)


def test_layer_tokens_composes_route_experts_combine():
    cfg = synth.CONFIGS["tiny"]
    inp = synth.make_router_inputs(cfg)
    W = synth.make_expert_weights(cfg)
    w13 = synth.bf16_bits(W["w13"])
    w2 = synth.bf16_bits(W["w2"])
    x = synth.bf16_bits(inp["x"])
    out = oracle.layer_tokens(cfg, x, inp["w_gate"].numpy(), inp["bias"].numpy(),
                              lambda e: dict(w13=w13[e], w2=w2[e]), None, [3, 0, 15])
    idx, w = oracle.route(x, inp["w_gate"].numpy(), inp["bias"].numpy(), cfg.k, 1, 1, 1.0)
    assert np.array_equal(out["topk_idx"], idx[[3, 0, 15]])
    t = 15
    ref = np.zeros(cfg.d)
    for i in range(cfg.k):
        o, _ = oracle.swiglu_row_bf16(x[t], w13[idx[t, i]], w2[idx[t, i]])
        ref += float(w[t, i]) * oracle.bf16_to_f32(o)
    yb = torch.from_numpy(ref).float().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.abs(out["y"][2].astype(np.int32) - yb.astype(np.int32)).max() <= 1


# ------------------------------------------------------------------------------------------
# Redundant experts and their placement (reading R-k)
# ------------------------------------------------------------------------------------------
def _placement_ok(slot_expert, n_copies, copy_slot, E, R, S):
    assert slot_expert.shape == (R * S,)
    assert (n_copies >= 1).all() and n_copies.sum() == R * S
    assert np.array_equal(np.bincount(slot_expert, minlength=E), n_copies)
    for e in range(E):
        slots = copy_slot[e, :n_copies[e]]
        assert (copy_slot[e, n_copies[e]:] == -1).all()
        assert np.all(np.diff(slots) > 0) and (slot_expert[slots] == e).all()
    for r in range(R):                      # a rank's slots in (expert, copy) order
        assert np.all(np.diff(slot_expert[r * S:(r + 1) * S]) >= 0)


def test_placement_of_equal_loads_without_spares_is_round_robin():
    """Equal loads and no spare slot: LPT deals the experts out in index order, expert e to rank
    e mod R, so rank r holds r, r+R, r+2R, ..."""
    E, R = 24, 4
    se, nc, cs = oracle.place_experts(np.ones(E), R, E // R)
    _placement_ok(se, nc, cs, E, R, E // R)
    assert np.array_equal(se.reshape(R, -1), np.arange(E).reshape(-1, R).T)


def test_placement_spare_copies_go_to_the_heaviest_shares():
    # one heavy expert among equals takes every spare slot while its share stays the largest
    E, R, S = 8, 6, 2
    load = np.ones(E)
    load[5] = 40.0
    se, nc, cs = oracle.place_experts(load, R, S)
    _placement_ok(se, nc, cs, E, R, S)
    assert nc[5] == 1 + (R * S - E) and (np.delete(nc, 5) == 1).all()
    # its copies land on distinct ranks (each is larger than any other expert's load)
    assert len({int(p) // S for p in cs[5, :nc[5]]}) == nc[5]


def _brute_force_makespan(shares, R, S):
    """Smallest possible maximum rank load over every assignment of the shares to R ranks of at
    most S shares each."""
    import itertools
    best = np.inf
    for assign in itertools.product(range(R), repeat=len(shares)):
        if max(np.bincount(assign, minlength=R)) > S:
            continue
        loads = np.zeros(R)
        for a, l in zip(assign, shares):
            loads[a] += l
        best = min(best, loads.max())
    return best


@pytest.mark.parametrize("seed", range(8))
def test_placement_is_within_grahams_lpt_bound(seed):
    """With slots to spare on every rank (no slot limit binds) the placement is LPT, whose
    largest rank load is at most (4/3 - 1/(3R)) of the optimum (Graham, 1969); the optimum
    comes from brute force over every assignment."""
    rng = np.random.default_rng(seed)
    E, R = 6, 3
    S = 4                                   # 12 slots: 6 experts + 6 copies, <= 4 per rank
    load = rng.integers(1, 60, E).astype(np.float64)
    se, nc, cs = oracle.place_experts(load, R, S)
    _placement_ok(se, nc, cs, E, R, S)
    shares = np.concatenate([[load[e] / nc[e]] * nc[e] for e in range(E)])
    rank_load = np.zeros(R)
    for p, e in enumerate(se):
        rank_load[p // S] += load[e] / nc[e]
    opt = _brute_force_makespan(shares, R, S)
    assert rank_load.max() <= (4 / 3 - 1 / (3 * R)) * opt + 1e-9
    assert np.isclose(rank_load.sum(), load.sum())


def _chapter_skewed_batch():
    """The skewed decode batch of "Serving Mixture-of-Experts", Hot-Expert Skew section: 256
    experts on 32 GPUs, 2048 tokens, top-8, experts 0..7 four times as popular (drawn with the
    same seeded generator the chapter names)."""
    rng = np.random.default_rng(0)
    E, G, T, k = 256, 32, 2048, 8
    rng.integers(0, E, size=(T, k))          # the chapter draws its uniform batch first
    p = np.ones(E)
    p[:8] *= 4
    p /= p.sum()
    return rng.choice(E, size=(T, k), p=p), E, G


def test_replication_lowers_the_imbalance_of_the_chapters_skewed_batch():
    """The chapter's claim (exercise 5): replicating the hot experts drops IF on its skewed
    example. Contiguous placement IF > 1.5 (the chapter's printed bound); the LPT placement with
    one spare slot per GPU, loads from that same batch, brings it close to 1."""
    ids, E, G = _chapter_skewed_batch()
    counts = np.bincount(ids.reshape(-1), minlength=E)
    base = oracle.imbalance_factor(counts, G)
    assert base > 1.5
    S = E // G + 1
    se, nc, cs = oracle.place_experts(counts.astype(np.float64), G, S)
    _placement_ok(se, nc, cs, E, G, S)
    assert (nc[:8] >= 2).all()               # every hot expert got a copy
    rank = np.zeros(G)
    for p, e in enumerate(se):
        rank[p // S] += counts[e] / nc[e]
    placed = rank.max() / rank.mean()
    assert placed < base and placed < 1.1


def test_placed_dispatch_with_one_copy_each_is_the_rank_major_layout():
    """One copy per expert in expert order (slot e = expert e): the placed dispatch is the
    dispatch of reading R-g, bit for bit."""
    cfg = synth.CONFIGS["tiny"]
    rng = np.random.default_rng(11)
    ti = np.stack([rng.permutation(cfg.E)[:cfg.k] for _ in range(cfg.T)]).astype(np.int32)
    nc = np.ones(cfg.E, np.int32)
    cs = np.full((cfg.E, 4), -1, np.int32)
    cs[:, 0] = np.arange(cfg.E)
    c1, r1, s1 = oracle.dispatch_index_placed(ti, cfg.E, cfg.R, cfg.E // cfg.R, nc, cs)
    c0, _, r0, s0 = oracle.dispatch_index(ti, cfg.E, cfg.R)
    assert np.array_equal(c1, c0) and np.array_equal(r1, r0) and np.array_equal(s1, s0)


def test_placed_dispatch_splits_each_sources_tokens_evenly_over_the_copies():
    T, E, k, R, S = 64, 16, 4, 4, 6          # 24 slots: 8 copies to spare
    rng = np.random.default_rng(3)
    p = np.ones(E)
    p[[2, 9]] = 12.0
    p /= p.sum()
    ti = np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    load = np.bincount(ti.reshape(-1), minlength=E).astype(np.float64)
    se, nc, cs = oracle.place_experts(load, R, S)
    counts, row_of, src_tok = oracle.dispatch_index_placed(ti, E, R, S, nc, cs)
    cap = (T // R) * min(k, S)
    assert counts.sum() == T * k
    assert len(np.unique(row_of)) == T * k and row_of.min() >= 0 and row_of.max() < R * R * cap
    tok = np.repeat(np.arange(T), k)
    assert np.array_equal(src_tok[row_of.reshape(-1)], tok)
    Ts = T // R
    for s in range(R):
        for e in range(E):
            got = counts[s, cs[e, :nc[e]]]
            assert got.max() - got.min() <= 1          # even within one source
            n_se = int((ti[s * Ts:(s + 1) * Ts] == e).sum())
            assert got.sum() == n_se
            # the j-th token of source s for expert e went to copy (j + s) mod copies
            js = [(t, i) for t in range(s * Ts, (s + 1) * Ts) for i in range(k) if ti[t, i] == e]
            for j, (t, i) in enumerate(js):
                slot = cs[e, (j + s) % nc[e]]
                seg = row_of[t, i] // cap
                assert seg == (slot // S) * R + s
    # rows land in the segment of the slot's rank, packed from 0
    seg_fill = np.bincount(row_of.reshape(-1) // cap, minlength=R * R)
    assert np.array_equal(seg_fill.reshape(R, R).T.reshape(-1),
                          counts.reshape(R, R, S).sum(2).reshape(-1))
    # replication lowered the rank-level imbalance of this batch
    contiguous = oracle.imbalance_factor(load, R)
    placed = oracle.rank_loads(counts, R)
    assert placed.max() / placed.mean() < contiguous
