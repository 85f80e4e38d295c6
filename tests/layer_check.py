"""Oracle check of one layer call on DeepSeek-V3-sized workloads, expert by expert.

The checked set is a list of tokens (whose whole layer output y[t] is compared) plus any extra
(token, choice) pairs (whose expert-output rows are compared). Work is grouped by expert: each
touched expert's weights are copied to the host once, and the oracle's row functions for that
expert's rows run on a host thread. The oracle itself stays single-threaded; several calls into
it run at once because ctypes releases the GIL for the duration of each C call.

Comparisons (the workload's rules): routing indices and gate weights of every checked token bit
for bit; the checked expert-output rows, the shared-expert rows and the layer outputs each within
the given tolerance of max |error| / rms(reference). The reference is the oracle's fp64 value
before its rounding to bf16, the RMS is taken over the checked set, and each bf16 output is
allowed its own rounding (half the bf16 gap below it) before the error is measured: a bf16
output cannot be closer to the exact value than that, and at 4-5 RMS one bf16 step is already
about 2e-2 of the RMS.
"""
from __future__ import annotations

import collections
import concurrent.futures as cf
import os

import numpy as np
import torch

import oracle
from gpu_util import bf16_to_f64, format_err, host_bits, rel_max_err


def _threads():
    return max(1, min(32, os.cpu_count() or 1))


def _rows_of(t_dev, rows):
    """Host copy of the listed rows of a device tensor."""
    idx = torch.as_tensor(np.asarray(rows, dtype=np.int64), device=t_dev.device)
    return host_bits(t_dev.index_select(0, idx))


def check_layer(cfg, inp, W, bufs, y, tokens, extra_pairs=(), tol=2e-2):
    """Returns a dict of the worst errors; asserts every rule on the way."""
    fp8 = cfg.w == "fp8"
    p2 = getattr(cfg, "scales", "amax") == "pow2"   # e4m3 with power-of-two block scales
    k = cfg.k
    tokens = np.asarray(sorted(set(int(t) for t in tokens)), dtype=np.int64)
    x = host_bits(inp["x"])
    ti = bufs["topk_idx"].cpu().numpy()
    tw = bufs["topk_w"].cpu().numpy()
    ro = bufs["row_of"].cpu().numpy()
    pairs = {(int(t), i) for t in tokens for i in range(k)} | {(int(t), int(i))
                                                                for t, i in extra_pairs}
    toks_all = np.asarray(sorted({t for t, _ in pairs}), dtype=np.int64)

    # routing of every checked token, bit for bit
    idx_o, w_o = oracle.route(x[toks_all], inp["w_gate"].cpu().numpy(), inp["bias"].cpu().numpy(),
                              cfg.k, cfg.n_group, cfg.topk_group, cfg.route_scale)
    assert np.array_equal(ti[toks_all], idx_o), "routing differs from the oracle"
    assert np.array_equal(tw[toks_all], w_o), "gate weights differ from the oracle"

    # oracle inputs per token (e4m3: the dispatch's 1x128 quantisation of x)
    pos = {int(t): j for j, t in enumerate(toks_all)}
    if fp8:
        xq, xsc = oracle.quant_rows_e4m3(oracle.bf16_to_f32(x[toks_all]), pow2=p2)

    by_e = collections.defaultdict(list)
    for t, i in sorted(pairs):
        by_e[int(ti[t, i])].append((t, i))

    # each job returns (bf16 output, fp64 output before its rounding) per row
    def expert_job(e, Wt, plist):
        out = {}
        for t, i in plist:
            j = pos[t]
            if fp8:
                o, _, ox = oracle.swiglu_row_fp8(xq[j], xsc[j], Wt["w13"], Wt["w13_s"], Wt["w2"],
                                                 Wt["w2_s"], exact=True, pow2=p2)
            else:
                o, _, ox = oracle.swiglu_row_bf16(x[t], Wt["w13"], Wt["w2"], exact=True)
            out[(t, i)] = (o, ox)
        return out

    def shared_job(S, tl):
        out = {}
        for t in tl:
            j = pos[t]
            if fp8:
                o, _, ox = oracle.swiglu_row_fp8(xq[j], xsc[j], S["ws13"], S["ws13_s"], S["ws2"],
                                                 S["ws2_s"], exact=True, pow2=p2)
            else:
                o, _, ox = oracle.swiglu_row_bf16(x[t], S["ws13"], S["ws2"], exact=True)
            out[t] = (o, ox)
        return out

    ref = {}
    sh_ref = {}
    nthr = _threads()
    with cf.ThreadPoolExecutor(max_workers=nthr) as ex:
        futs = []
        if cfg.d_ff_shared:
            S = dict(ws13=host_bits(W["ws13"]), ws2=host_bits(W["ws2"]))
            if fp8:
                S["ws13_s"] = W["ws13_s"].cpu().numpy()
                S["ws2_s"] = W["ws2_s"].cpu().numpy()
            chunk = max(1, len(tokens) // nthr + 1)
            for c0 in range(0, len(tokens), chunk):
                futs.append(("s", ex.submit(shared_job, S, [int(t) for t in tokens[c0:c0 + chunk]])))
        # the largest experts first so the pool ends evenly; big experts split in pieces
        for e in sorted(by_e, key=lambda e: -len(by_e[e])):
            Wt = dict(w13=host_bits(W["w13"][e]), w2=host_bits(W["w2"][e]))
            if fp8:
                Wt["w13_s"] = W["w13_s"][e].cpu().numpy()
                Wt["w2_s"] = W["w2_s"][e].cpu().numpy()
            pl = by_e[e]
            piece = max(8, len(pl) // nthr + 1)
            for p0 in range(0, len(pl), piece):
                futs.append(("e", ex.submit(expert_job, e, Wt, pl[p0:p0 + piece])))
        for kind, f in futs:
            (sh_ref if kind == "s" else ref).update(f.result())

    # Every computed expert-output row against ebuf at its receive row. The workload's rule
    # (max |error| relative to the output RMS) is applied to each stage's bf16 output against
    # the oracle's exact value (before the oracle's own rounding to bf16), after allowing the
    # output its own rounding to bf16 (format_err); the RMS is taken over the checked set. The
    # plain max |error| / RMS against the exact and the rounded oracle values is reported too.
    plist = sorted(pairs)
    got_rows = bf16_to_f64(_rows_of(bufs["ebuf"], [ro[t, i] for t, i in plist]))
    ref_rows = np.stack([ref[p][1] for p in plist])
    res = {"rows": len(plist), "tokens": len(tokens), "experts": len(by_e),
           "rows_err": format_err(got_rows, ref_rows),
           "rows_plain": rel_max_err(got_rows, ref_rows),
           "rows_vs_rounded": rel_max_err(got_rows,
                                          bf16_to_f64(np.stack([ref[p][0] for p in plist]))),
           "shared_err": 0.0, "shared_plain": 0.0, "y_err": 0.0, "y_plain": 0.0,
           "y_vs_rounded": 0.0}
    assert res["rows_err"] <= tol, res
    if len(tokens) == 0:
        return res
    sh = None
    if cfg.d_ff_shared:
        got_sh = bf16_to_f64(_rows_of(bufs["shared_out"], tokens))
        sh = np.stack([sh_ref[int(t)][0] for t in tokens])
        sh_exact = np.stack([sh_ref[int(t)][1] for t in tokens])
        res["shared_err"] = format_err(got_sh, sh_exact)
        res["shared_plain"] = rel_max_err(got_sh, sh_exact)
        assert res["shared_err"] <= tol, res
    # the layer output of the checked tokens: the oracle's combine of the oracle's rows
    eo = np.stack([ref[(int(t), i)][0] for t in tokens for i in range(k)])
    rows = np.arange(len(tokens) * k, dtype=np.int32).reshape(len(tokens), k)
    y_ref, y_exact = oracle.combine(eo, rows, tw[tokens], sh, exact=True)
    got_y = bf16_to_f64(_rows_of(y, tokens))
    res["y_err"] = format_err(got_y, y_exact)
    res["y_plain"] = rel_max_err(got_y, y_exact)
    res["y_vs_rounded"] = rel_max_err(got_y, bf16_to_f64(y_ref))
    assert res["y_err"] <= tol, res
    return res


def hot_expert_pairs(ti, e):
    """Every (token, choice) routed to expert e."""
    t, i = np.nonzero(ti == e)
    return list(zip(t.tolist(), i.tolist()))


def experts_by_rows(ti, E):
    """Rows per expert."""
    return np.bincount(ti.reshape(-1), minlength=E)
