"""Helpers shared by the GPU tests: inputs on the device from the seeded generator, the
library's stages run through the C ABI, and host copies for the oracle."""
import numpy as np
import torch

import synth


def device_inputs(cfg, device="cuda"):
    inp = synth.make_router_inputs(cfg, device)
    W = synth.make_expert_weights(cfg, device)
    return inp, W


def weight_dict(W):
    return dict(w13=W["w13"], w13_s=W["w13_s"], w2=W["w2"], w2_s=W["w2_s"], ws13=W["ws13"],
                ws13_s=W["ws13_s"], ws2=W["ws2"], ws2_s=W["ws2_s"])


def host_bits(t):
    """Host numpy view of a device tensor: bf16 -> uint16 bits, uint8 stays uint8."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def expert_getter(W, fp8):
    """Callable e -> host weights of routed expert e, for oracle.layer_tokens."""
    def get(e):
        if fp8:
            return dict(w13=host_bits(W["w13"][e]), w2=host_bits(W["w2"][e]),
                        w13_s=W["w13_s"][e].cpu().numpy(), w2_s=W["w2_s"][e].cpu().numpy())
        return dict(w13=host_bits(W["w13"][e]), w2=host_bits(W["w2"][e]))
    return get


def shared_host(W, fp8):
    if W["ws13"] is None:
        return None
    if fp8:
        return dict(ws13=host_bits(W["ws13"]), ws2=host_bits(W["ws2"]),
                    ws13_s=W["ws13_s"].cpu().numpy(), ws2_s=W["ws2_s"].cpu().numpy())
    return dict(ws13=host_bits(W["ws13"]), ws2=host_bits(W["ws2"]))


def rel_max_err(got, ref):
    """max |got - ref| / rms(ref) over float arrays."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(np.abs(got - ref).max()) / max(rms, 1e-30)


def bf16_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ws_offsets(cfg):
    """Byte offsets inside the workspace, mirroring the library's layout (for diagnostics:
    the tests read the SwiGLU intermediate h through them)."""
    def up(v):
        return (v + 255) // 256 * 256
    tk = cfg.T * cfg.k
    ab = 1 if cfg.act == "fp8" else 2
    bn = 128 if (cfg.act == "fp8" or tk >= 16 * cfg.E) else 64
    max_tiles = cfg.E + (tk + bn - 1) // bn
    o = {}
    cur = 0
    for name, size in [("status", 16), ("partials", 4 * 16 * cfg.T * cfg.E), ("grp_n", 4 * cfg.E),
                       ("grp_off", 4 * cfg.E), ("n_tiles", 8), ("tiles", 16 * max_tiles),
                       ("row_list", 4 * tk), ("h", ab * tk * cfg.d_ff)]:
        o[name] = cur
        cur = up(cur + size)
    fp8 = cfg.act == "fp8"
    p2 = fp8 and getattr(cfg, "scales", "amax") == "pow2"
    cur = up(cur + (4 * tk * (cfg.d_ff // 128) if fp8 else 0))          # h_scales
    cap = (cfg.T // cfg.R) * min(cfg.k, cfg.E // cfg.R)
    shared_tiles = (cfg.T + bn - 1) // bn if cfg.d_ff_shared else 0
    for name, size in [("hs", ab * cfg.T * cfg.d_ff_shared),
                       ("hs_scales", 4 * cfg.T * (cfg.d_ff_shared // 128) if fp8 else 0),
                       ("xq", cfg.T * cfg.d if fp8 else 0),
                       ("xq_scales", 4 * cfg.T * (cfg.d // 128) if fp8 else 0),
                       ("run_start", 4 * cfg.R * cfg.E), ("run_pre", 4 * cfg.R * cfg.E),
                       ("src_tok", 4 * cfg.R * cfg.R * cap), ("tok_list", 4 * tk),
                       ("grp_order", 4 * cfg.E),
                       ("fused_done", 4 * (max_tiles + shared_tiles + 2)),
                       ("sf_gu", 64 * tk if p2 else 0), ("sf_x", 64 * cfg.T if p2 else 0),
                       ("sf_h", 64 * tk if p2 else 0), ("sf_hs", 64 * cfg.T if p2 else 0),
                       ("n_tiles2", 8), ("tiles2", 16 * (cfg.E + (tk + 2 * bn - 1) // (2 * bn)))]:
        o[name] = cur
        cur = up(cur + size)
    o["total"] = cur
    o["bn"] = bn
    return o


def half_gap_below_bf16(v):
    """Half the distance from |v| down to the next smaller bf16 value (v bf16 values as
    floats): the largest error the rounding of an exact value to v can have made."""
    v = np.abs(np.asarray(v, dtype=np.float64)).astype(np.float32)
    bits = v.view(np.uint32) >> 16
    below = ((np.maximum(bits, 1) - 1).astype(np.uint32) << 16).view(np.float32)
    return (v.astype(np.float64) - below.astype(np.float64)) / 2.0


def format_err(got, exact):
    """Error of bf16 outputs `got` (as floats) against the exact reference values, relative to
    the reference RMS, after allowing each output its own rounding to bf16:
    max(0, |got - exact| - half the bf16 gap below |got|) / rms(exact)."""
    got = np.asarray(got, dtype=np.float64)
    exact = np.asarray(exact, dtype=np.float64)
    rms = float(np.sqrt(np.mean(exact * exact)))
    excess = np.maximum(0.0, np.abs(got - exact) - half_gap_below_bf16(got))
    return float(excess.max()) / max(rms, 1e-30)
