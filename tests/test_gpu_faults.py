"""Stage calls fed metadata that breaks their contract, built on the host (the layer itself never
produces such input): duplicate or out-of-range experts to the dispatch, rows past the receive
buffer to the combine, counts that do not sum to T*k to the expert FFNs. Each call must skip the
bad entries, report MOE_DEV_BOUNDS in the status word, and write nothing outside its buffers
(checked with canary guard bands around every buffer the call writes). Nothing here faults or
hangs the GPU: every index the kernels derive from such input is bounded before use."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import bf16_to_f64, host_bits, weight_dict

pytestmark = pytest.mark.gpu

GUARD = 4096
SMALL = synth.MoEConfig("small", T=96, d=384, E=12, k=3, n_group=4, topk_group=2, d_ff=640,
                        d_ff_shared=640, R=3, route_scale=2.5, seed=77)


def moe():
    import combine_grouped_gemm_gb300 as m
    return m


def _guarded(shape, dtype, store, fill=0xA5):
    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    raw = torch.full((GUARD + n + GUARD,), fill, dtype=torch.uint8, device="cuda")
    store.append((raw, n))
    return raw[GUARD:GUARD + n].view(dtype).view(shape)


def _bands_intact(store):
    return all(bool((raw[:GUARD] == 0xA5).all()) and bool((raw[GUARD + n:] == 0xA5).all())
               for raw, n in store)


def _corrupt_choices(cfg, seed):
    """Distinct random choices per token, then some repeated and some out of range. A choice is
    valid when its expert is in [0, E) and differs from the token's earlier choices."""
    rng = np.random.default_rng(seed)
    ti = np.stack([rng.permutation(cfg.E)[:cfg.k] for _ in range(cfg.T)]).astype(np.int32)
    for t in rng.choice(cfg.T, 12, replace=False):
        ti[t, 2] = ti[t, 0]                    # a repeat of the token's first choice
    for t in rng.choice(cfg.T, 6, replace=False):
        ti[t, int(rng.integers(cfg.k))] = [cfg.E, cfg.E + 77, -1, -5000][int(rng.integers(4))]
    valid = np.zeros_like(ti, dtype=bool)
    for t in range(cfg.T):
        for i in range(cfg.k):
            valid[t, i] = 0 <= ti[t, i] < cfg.E and ti[t, i] not in ti[t, :i]
    assert (~valid).sum() >= 12
    return ti, ~valid


def _expected_layout(cfg, ti, valid):
    """Receive row of each valid choice: the stable rank-major layout of the valid choices
    (destination rank, source rank, local expert ascending, token ascending)."""
    T, E, R, k = cfg.T, cfg.E, cfg.R, cfg.k
    Ts, Er, cap = cfg.T_s, cfg.E_r, cfg.cap
    counts = np.zeros((R, E), np.int64)
    for t in range(T):
        for i in range(k):
            if valid[t, i]:
                counts[t // Ts, ti[t, i]] += 1
    first = np.cumsum(counts.reshape(R, R, Er), axis=2) - counts.reshape(R, R, Er)
    first = first.reshape(R, E)
    run = np.zeros((R, E), np.int64)
    rows = np.full((T, k), -1, np.int64)
    for t in range(T):
        s = t // Ts
        for i in range(k):
            if valid[t, i]:
                e = ti[t, i]
                rows[t, i] = ((e // Er) * R + s) * cap + first[s, e] + run[s, e]
                run[s, e] += 1
    return counts, rows


@pytest.mark.parametrize("act", ["bf16", "fp8"])
def test_dispatch_skips_and_reports_repeated_and_out_of_range_experts(act):
    import dataclasses
    cfg = SMALL if act == "bf16" else dataclasses.replace(SMALL, name="small_fp8", act="fp8",
                                                          w="fp8", d=512, d_ff=256,
                                                          d_ff_shared=256)
    m = moe()
    ti, bad = _corrupt_choices(cfg, 5)
    valid = ~bad
    s = m.query_sizes(cfg)
    store = []
    fp8 = cfg.act == "fp8"
    recv = _guarded((s["recv_rows"], cfg.d), torch.uint8 if fp8 else torch.bfloat16, store)
    rsc = _guarded((cfg.d // 128, s["recv_rows"]), torch.float32, store) if fp8 else None
    counts = _guarded((cfg.R, cfg.E), torch.int32, store)
    row_of = _guarded((cfg.T, cfg.k), torch.int32, store)
    src_tok = _guarded((s["recv_rows"],), torch.int32, store)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    x = synth.normal_bf16(cfg.seed, synth.TAG_X, (cfg.T, cfg.d), 1.0, "cuda")
    m.dispatch(cfg, x, torch.from_numpy(ti).cuda(), recv, rsc, counts, row_of, src_tok,
               status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == m.MOE_DEV_BOUNDS
    assert _bands_intact(store)
    exp_counts, exp_rows = _expected_layout(cfg, ti, valid)
    assert np.array_equal(counts.cpu().numpy(), exp_counts)
    assert np.array_equal(row_of.cpu().numpy(), exp_rows)
    st = src_tok.cpu().numpy()
    tok = np.repeat(np.arange(cfg.T), cfg.k).reshape(cfg.T, cfg.k)
    assert np.array_equal(st[exp_rows[valid]], tok[valid])
    assert (st >= 0).sum() == valid.sum()
    # the payload of the valid rows is the token's row (bf16) or its e4m3 codes and scales
    xb = host_bits(x)
    if fp8:
        q, sc = oracle.quant_rows_e4m3(oracle.bf16_to_f32(xb))
        got = recv.cpu().numpy()
        assert np.array_equal(got[exp_rows[valid]], q[tok[valid]])
        assert np.array_equal(rsc.cpu().numpy().T[exp_rows[valid]], sc[tok[valid]])
    else:
        assert np.array_equal(host_bits(recv)[exp_rows[valid]], xb[tok[valid]])
    # the index-only pass reports the same way and agrees
    st2 = torch.empty_like(src_tok)
    c2 = torch.empty_like(counts)
    r2 = torch.empty_like(row_of)
    status.zero_()
    m.dispatch_index(cfg, torch.from_numpy(ti).cuda(), c2, r2, st2, status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == m.MOE_DEV_BOUNDS
    assert torch.equal(c2, counts) and torch.equal(r2, row_of) and torch.equal(st2, src_tok)


def test_combine_skips_and_reports_rows_past_the_receive_buffer():
    cfg = SMALL
    m = moe()
    s = m.query_sizes(cfg)
    g = torch.Generator().manual_seed(9)
    ebuf = (torch.randn((s["recv_rows"], cfg.d), generator=g) * 0.5).to(torch.bfloat16).cuda()
    sh = torch.randn((cfg.T, cfg.d), generator=g).to(torch.bfloat16).cuda()
    rng = np.random.default_rng(2)
    ro = rng.choice(s["recv_rows"], cfg.T * cfg.k, replace=False).reshape(cfg.T, cfg.k)
    ro = ro.astype(np.int32)
    w = rng.random((cfg.T, cfg.k)).astype(np.float32)
    ro[3, 1] = s["recv_rows"]              # one past the end
    ro[10, 0] = s["recv_rows"] + 123456    # far past
    ro[20, 2] = 2 ** 31 - 1
    ro[30, 0] = -1                         # skipped silently (a choice the dispatch skipped)
    store = []
    y = _guarded((cfg.T, cfg.d), torch.bfloat16, store)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    m.combine(cfg, ebuf, torch.from_numpy(ro).cuda(), torch.from_numpy(w).cuda(), sh, y,
              status=status)
    torch.cuda.synchronize()
    assert int(status[0]) == m.MOE_DEV_BOUNDS
    assert _bands_intact(store)
    # expected: the skipped choices contribute nothing (an appended zero row stands for them)
    eb = np.concatenate([host_bits(ebuf), np.zeros((1, cfg.d), np.uint16)])
    ro_ok = np.where((ro < 0) | (ro >= s["recv_rows"]), s["recv_rows"], ro).astype(np.int32)
    ref = oracle.combine(eb, ro_ok, w, host_bits(sh))
    assert np.abs(host_bits(y).astype(np.int32) - ref.astype(np.int32)).max() <= 1


@pytest.mark.parametrize("how", ["total", "segment"])
def test_expert_ffn_reports_counts_that_break_their_sum(how):
    """counts that do not sum to T*k (or overflow a receive segment) are reported and every
    derived index stays inside its buffer."""
    cfg = SMALL
    m = moe()
    inp = synth.make_router_inputs(cfg, "cuda")
    W = synth.make_expert_weights(cfg, "cuda")
    b = m.Buffers(cfg)
    m.route(cfg, inp["x"], inp["w_gate"], inp["bias"], b["topk_idx"], b["topk_w"], b["ws"])
    m.dispatch(cfg, inp["x"], b["topk_idx"], b["recv"], None, b["counts"], b["row_of"])
    torch.cuda.synchronize()
    counts = b["counts"].clone()
    if how == "total":
        counts[1, 4] += 37
    else:
        counts[2, 0] = cfg.cap + 5
    s = m.query_sizes(cfg)
    store = []
    ebuf = _guarded((s["recv_rows"], cfg.d), torch.bfloat16, store)
    shared_out = _guarded((cfg.T, cfg.d), torch.bfloat16, store)
    ws = _guarded((s["ws_bytes"],), torch.uint8, store)
    ws.zero_()
    m.expert_ffn(cfg, b["recv"], None, counts, inp["x"], weight_dict(W), ebuf, shared_out, ws)
    torch.cuda.synchronize()
    st = m.read_status(ws)
    assert st & m.MOE_DEV_BOUNDS and not st & m.MOE_DEV_TIMEOUT
    assert _bands_intact(store)
    # the context is still usable and a clean call is right
    lay = m.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W))
    y = lay(inp["x"])
    assert m.read_status(lay.bufs["ws"]) == 0
    ref = oracle.layer_tokens(cfg, host_bits(inp["x"]), inp["w_gate"].cpu().numpy(),
                              inp["bias"].cpu().numpy(),
                              lambda e: dict(w13=host_bits(W["w13"][e]), w2=host_bits(W["w2"][e])),
                              dict(ws13=host_bits(W["ws13"]), ws2=host_bits(W["ws2"])),
                              np.arange(8))
    got = bf16_to_f64(host_bits(y)[:8])
    assert np.abs(got - ref["y_exact"]).max() / np.sqrt(np.mean(ref["y_exact"] ** 2)) <= 2e-2
