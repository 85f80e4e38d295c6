"""Benchmark of the MoE layer hot path on GB300.

One step = one pass of the whole layer (router -> dispatch -> expert FFNs -> combine) over one
batch of seeded synthetic input with resident random-init weights. Default workload: the
DeepSeek-V3-shaped decode layer (T=64 tokens, d=7168, 256 routed experts of d_ff 2048 + one
shared expert, top-8 of 8 groups keeping 4, 8 logical ranks), bf16.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line (rank 0). Under torchrun (N > 1) every rank runs an independent replica
of the layer on its own batch (no collective on the data path: the expert-parallel ranks of
this method are logical partitions of one GPU), and the timing is the max over ranks.
--impl reference times the CPU oracle (the plain C definition of the method) on the host
cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE layer µs & tokens/s vs tokens (1–16K); % of HBM / tensor roofline"
# route x2, dispatch x2, ffn schedule x2 (plan, row list), gate/up GEMM, down GEMM, combine
# (+ the shared expert's input quantisation on the e4m3 path)
def kernels_per_step(cfg, mode="layer"):
    """Library kernels one layer step launches: route 2, dispatch 2 (1 in gather mode: no copy),
    schedule 2 (1 when the plan kernel fills the row list itself, up to 1024 rows), gate/up,
    down, combine; for e4m3 the quantisation of x when a shared expert or gather mode needs it;
    with power-of-two e4m3 scales the gate/up GEMM's scale-byte pass (one per gate/up launch);
    with the shared expert on a side stream, its two GEMMs as launches of their own."""
    gather = "gather" in mode
    side = "side" in mode and cfg.d_ff_shared > 0
    fused = "fused" in mode
    sched = 1 if cfg.T * cfg.k <= 1024 else 2
    quant = 1 if cfg.act == "fp8" and (cfg.d_ff_shared or gather) else 0
    sfpass = (2 if side else 1) if cfg.act == "fp8" and cfg.scales == "pow2" else 0
    return (7 + sched + quant + sfpass - (1 if gather else 0) + (2 if side else 0)
            - (2 if fused else 0))
L2_BYTES = 129 * 2 ** 20
CPU_SAMPLE_SECONDS = 12.0   # target CPU time of the oracle sample behind cpu_baseline


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default="dsv3_decode")
    p.add_argument("--T", type=int, default=0, help="override the token count (sweep points)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-sample", type=int, default=0, help="tokens in the oracle sample")
    p.add_argument("--no-extras", dest="extras", action="store_false",
                   help="time the named workload only (default with dsv3_decode at N=1: also "
                        "the sweep, the skewed prefill and the FP8 prefill)")
    p.add_argument("--extra-steps", type=int, default=10, help="timed steps per extra workload")
    p.add_argument("--mode", default="layer", choices=sorted(MODES),
                   help="the layer variant of the main workload's timed steps")
    p.add_argument("--route-only", action="store_true",
                   help="time the router stage alone on the workload's shapes (router inputs "
                        "and workspace only, no expert weights): for profiling its kernels")
    return p.parse_args()


def workload(args):
    cfg = synth.CONFIGS[args.workload]
    if args.T:
        cfg = cfg.with_T(args.T)
    return cfg


def describe(cfg):
    return {"workload": cfg.name, "T": cfg.T, "d": cfg.d, "E": cfg.E, "k": cfg.k,
            "n_group": cfg.n_group, "topk_group": cfg.topk_group, "d_ff": cfg.d_ff,
            "d_ff_shared": cfg.d_ff_shared, "R_logical": cfg.R, "route_scale": cfg.route_scale,
            "act": cfg.act, "weights": cfg.w, "bias": cfg.bias}


# ------------------------------------------------------------------------------------------
# Algorithmic bytes / flops per stage (what the method must move; expert counts are the
# routing's own)
# ------------------------------------------------------------------------------------------
def algorithmic(cfg, counts):
    T, d, E, k, F, Fs = cfg.T, cfg.d, cfg.E, cfg.k, cfg.d_ff, cfg.d_ff_shared
    bw = 1 if cfg.w == "fp8" else 2
    ba = 1 if cfg.act == "fp8" else 2
    tk = T * k
    touched = int((counts.sum(0) > 0).sum())
    sc_w13 = (2 * F // 128) * (d // 128) * 4 if cfg.w == "fp8" else 0
    sc_w2 = (d // 128) * (F // 128) * 4 if cfg.w == "fp8" else 0
    sc_act = (d // 128) * 4 if cfg.act == "fp8" else 0
    sc_h = (F // 128) * 4 if cfg.act == "fp8" else 0
    rows_sh = T if Fs else 0
    b = {}
    b["route"] = 2 * T * d + 4 * E * d + 4 * E + 8 * tk
    b["dispatch"] = 2 * T * d + tk * (d * ba + sc_act) + 12 * tk
    b["ffn_gate_up"] = (touched * (2 * F * d * bw + sc_w13) + (2 * Fs * d * bw + sc_w13 if Fs else 0)
                        + (tk + rows_sh) * (d * ba + sc_act) + (tk + rows_sh) * (F * ba + sc_h))
    b["ffn_down"] = (touched * (d * F * bw + sc_w2) + (d * Fs * bw + sc_w2 if Fs else 0)
                     + (tk + rows_sh) * (F * ba + sc_h) + (tk + rows_sh) * d * 2)
    b["combine"] = tk * d * 2 + (T * d * 2 if Fs else 0) + T * d * 2 + 8 * tk
    # schedule: counts in, per-expert tables and the row list out (+ the shared expert's input
    # quantised on the e4m3 path)
    b["ffn_setup"] = 4 * cfg.R * E * 3 + 8 * E + 4 * tk + (
        T * d * 2 + T * d + T * (d // 128) * 4 if cfg.act == "fp8" and Fs else 0)
    f = {"route": 2 * T * d * E, "ffn_gate_up": 2 * (tk + rows_sh) * 2 * F * d,
         "ffn_down": 2 * (tk + rows_sh) * F * d}
    return b, f, touched


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm": float(p["hbm_gbs"]), "bf16": float(p["bf16_tflops"]),
                "bf16_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


KERNEL_NAMES = {"ffn_gate_up": "ffn_gemm_{}_kernel<0> (gate/up + SwiGLU)",
                "ffn_down": "ffn_gemm_{}_kernel<1> (down)",
                "route": "route_partials[_resident]_kernel + route_select[_cta]_kernel",
                "dispatch": "dispatch_index_kernel + dispatch_copy_kernel",
                "combine": "combine_kernel", "ffn_setup": "ffn_plan_kernel + ffn_rows_kernel"}


# The router's dot products are exact-order fp32 FMAs on the CUDA cores (no tensor cores), so its
# compute roof is the fp32 FMA rate: 152 SMs x 128 FMA lanes x 2 flops x 2.07 GHz (the maximum
# SM clock; a packed fp32x2 FMA occupies two lanes).
ALU_FP32_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def roofline(cfg, stage, ms, bytes_, flops, pk):
    """Roofline entry of one stage: the binding roof is the one whose ideal time is longest —
    HBM (algorithmic bytes / measured copy bandwidth), the tensor cores for the expert GEMMs
    (flops / the dtype's peak: measured bf16 burst, e4m3 = 2x that by the nominal ratio) or the
    fp32 FMA rate for the router."""
    tc_peak = pk["bf16"] * (2.0 if cfg.w == "fp8" else 1.0)
    t_hbm = bytes_[stage] / (pk["hbm"] * 1e9)
    t_tc = flops.get(stage, 0) / (tc_peak * 1e12) if stage in ("ffn_gate_up", "ffn_down") else 0.0
    t_alu = flops.get(stage, 0) / (ALU_FP32_TFLOPS * 1e12) if stage == "route" else 0.0
    kind = "bf16" if cfg.w != "fp8" else ("mx8" if cfg.scales == "pow2" else "e4m3")
    name = KERNEL_NAMES[stage].format(kind)
    traffic, note = measured_traffic(stage, cfg.name, bytes_[stage])
    base = {"kernel": name, "launch_ms": round(ms, 4), "traffic": traffic,
            "algorithmic_bytes_per_launch": bytes_[stage],
            "algorithmic_flops_per_launch": flops.get(stage, 0)}
    if note:
        base["traffic_source"] = note
    if t_alu > t_hbm:
        ach = flops[stage] / (ms * 1e-3) / 1e12
        return {**base, "bound": "alu", "achieved": round(ach, 1), "peak": round(ALU_FP32_TFLOPS, 1),
                "unit": "TFLOP/s", "frac": round(ach / ALU_FP32_TFLOPS, 4),
                "peak_source": "derived: fp32 FMA lanes x 2 x max SM clock"}
    if t_tc > t_hbm:
        ach = flops[stage] / (ms * 1e-3) / 1e12
        return {**base, "bound": "tensor", "achieved": round(ach, 1), "peak": tc_peak,
                "unit": "TFLOP/s", "frac": round(ach / tc_peak, 4),
                "peak_source": f"{pk['source']} bf16_tflops" + (" x2 (e4m3 nominal ratio)"
                                                                 if cfg.w == "fp8" else "")}
    ach = bytes_[stage] / (ms * 1e-3) / 1e9
    return {**base, "bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm"], "unit": "GB/s",
            "frac": round(ach / pk["hbm"], 4), "peak_source": f"{pk['source']} hbm_gbs"}


# The 32-expert stand-ins whose DRAM counters stand for each full workload: the same per-expert
# shapes and kernels, a few GB on the device (ncu captures of full-size launches are avoided).
# (The skewed prefill has none: 32 experts cannot hold its 10x hot expert, whose token tiles
# are what its excess traffic comes from.)
TRAFFIC_STANDIN = {"dsv3_decode": "dsv3_decode_e32", "dsv3_fp8_prefill": "dsv3_fp8_e32",
                   "dsv3_fp8_pow2_prefill": "dsv3_fp8_pow2_e32"}


def sources_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel, workload_name, algorithmic_bytes):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from the committed
    ncu summary: the launch's own capture when there is one, else the stand-in's measured
    traffic / algorithmic ratio times this launch's algorithmic bytes. None when absent, or
    when a kernel source changed since the counters were taken. Returns (bytes, note)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            tab = json.load(fh)
    except Exception:
        return None, None
    for key, direct in ((f"{kernel}@{workload_name}", True),
                        (f"{kernel}@{TRAFFIC_STANDIN.get(workload_name, '')}", False)):
        ent = tab.get(key)
        if not ent:
            continue
        try:
            if sources_hash(ent["sources"]) != ent["sources_sha256_16"]:
                return None, f"{key}: kernel source changed since the capture"
        except Exception:
            return None, None
        if direct:
            return int(ent["dram_bytes_per_launch"]), f"{key} (captured)"
        ratio = ent["dram_bytes_per_launch"] / ent["algorithmic_bytes_per_launch"]
        return int(round(ratio * algorithmic_bytes)), (
            f"scaled from {key}: traffic / algorithmic = {ratio:.4f} on the stand-in")
    return None, None


# ------------------------------------------------------------------------------------------
# Clocks during the timed region
# ------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.3)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            return None
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i]
                          and "Not" not in r[5 + i]})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def max_over_ranks(value: float, device) -> float:
    """The largest value over all ranks (the job is as slow as its slowest replica)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(T: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank processes its own T tokens per step."""
    return T * world / (ms_per_step * 1e-3)


# ------------------------------------------------------------------------------------------
# Our arm
# ------------------------------------------------------------------------------------------
def weight_dict(W):
    return dict(w13=W["w13"], w13_s=W["w13_s"], w2=W["w2"], w2_s=W["w2_s"], ws13=W["ws13"],
                ws13_s=W["ws13_s"], ws2=W["ws2"], ws2_s=W["ws2_s"])


MODES = {"layer": {}, "gather": {"gather": True}, "side": {"side_stream": True},
         "gather+side": {"gather": True, "side_stream": True},
         "side32": {"side_stream": True, "side_ctas": 32},
         "side64": {"side_stream": True, "side_ctas": 64},
         "fused": {"fused": True}, "gather+fused": {"gather": True, "fused": True}}


def setup(cfg, dev, rank=0, world=1, W=None, mode="layer"):
    """Inputs, weights (made here unless given) and a layer object on dev. Under torchrun every
    rank holds the same weights and its own batch of tokens. mode: one of MODES (moe_layer, or
    moe_layer_ex with gather mode and/or the shared expert on a side stream)."""
    import combine_grouped_gemm_gb300 as moe

    inp = synth.make_router_inputs(cfg, dev)
    if world > 1:
        inp["x"] = synth.normal_bf16(cfg.seed + 7919 * rank, synth.TAG_X, (cfg.T, cfg.d),
                                     cfg.x_std, dev)
    if W is None:
        W = synth.make_expert_weights(cfg, dev)
    lay = moe.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W), dev, **MODES[mode])
    return inp, W, lay


def time_modes(cfg, dev, W, steps, warm, modes=("gather", "side", "gather+side")):
    """Layer time of each variant on the same inputs and weights (the variants' outputs equal
    moe_layer's bit for bit; the tests check that)."""
    out = {}
    for mode in modes:
        inp, _, lay = setup(cfg, dev, W=W, mode=mode)
        r = time_layer(cfg, inp, lay, steps, warm, dev)
        out[mode] = {"layer_us": round(r["ms"] * 1e3, 2),
                     "tokens_per_s": round(job_tokens_per_s(cfg.T, 1, r["ms"]), 1),
                     "stages_us": {n: round(v * 1e3, 2) for n, v in r["stage_ms"].items()},
                     "e2e_tokens_per_s": round(job_tokens_per_s(cfg.T, 1, r["ms_e2e"]), 1),
                     "gpu_launches": kernels_per_step(cfg, mode) * steps}
        del lay, inp
    return out


def time_layer(cfg, inp, lay, steps, warmup, dev, rank=0, world=1, local_rank=0):
    """W untimed steps, then K back-to-back steps timed with CUDA events on the launching stream
    (barrier + synchronize on both sides, clocks sampled meanwhile); then K steps with stage
    events; then K end-to-end steps through MoELayer.run_host (pinned host buffers, both copies
    inside the timed region)."""
    import combine_grouped_gemm_gb300 as moe

    y = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.MOE_LAYER_EVENTS)]
           for _ in range(steps)]
    for row in evs:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize(dev)

    for _ in range(warmup):
        lay(inp["x"], y)
    torch.cuda.synchronize(dev)
    moe.clear_status(lay.bufs["ws"])

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    clocks = ClockSampler(local_rank) if rank == 0 else None
    barrier()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        lay(inp["x"], y)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop() if clocks else None
    ms = t0.elapsed_time(t1) / steps
    status = moe.read_status(lay.bufs["ws"])
    if status:
        raise RuntimeError(f"device status {status} after the timed region")

    # Per-stage times: the same steps again with an event between the stages. The events make
    # each stage start after the previous one has finished (no programmatic overlap of the
    # launches), so the stages add up to a little more than the step time above.
    for i in range(steps):
        lay(inp["x"], y, events=evs[i])
    torch.cuda.synchronize(dev)
    stage_ms = {n: 0.0 for n in moe.STAGE_NAMES}
    for row in evs:
        for j, n in enumerate(moe.STAGE_NAMES):
            stage_ms[n] += row[j].elapsed_time(row[j + 1]) / steps
    ms_max = max_over_ranks(ms, dev)

    # end to end through the public API: pinned host buffers, copies inside the timed region
    x_host = inp["x"].cpu().pin_memory()
    y_host = torch.empty_like(x_host).pin_memory()
    for _ in range(2):
        lay.run_host(x_host, y_host, stream)
    torch.cuda.synchronize(dev)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        lay.run_host(x_host, y_host, stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / steps, dev)

    counts = lay.bufs["counts"].cpu().numpy()
    return dict(ms=ms_max, ms_local=ms, stage_ms=stage_ms, clocks=clk, ms_e2e=ms_e2e,
                counts=counts, steps=steps, warmup=warmup)


def imbalance(cfg, counts):
    """Rank-level imbalance factor of one step's routing (max rank load / mean rank load)."""
    return round(float(counts.sum(0).reshape(cfg.R, -1).sum(1).max() / (cfg.T * cfg.k / cfg.R)), 4)


def summarise(cfg, r, pk, world=1, full=True):
    """The per-configuration fields of the JSON line."""
    b, f, touched = algorithmic(cfg, r["counts"])
    layer_bytes = sum(b.values())
    out = {
        "workload": cfg.name, "T": cfg.T, "act": cfg.act,
        "steps": r["steps"], "warmup": r["warmup"],
        "layer_us": round(r["ms"] * 1e3, 2),
        "tokens_per_s": round(job_tokens_per_s(cfg.T, world, r["ms"]), 1),
        "layer_hbm_frac": round(layer_bytes / (r["ms"] * 1e-3) / 1e9 / pk["hbm"], 4),
        "stages_us": {n: round(v * 1e3, 2) for n, v in r["stage_ms"].items()},
        "stages_roofline": {n: {k2: v2 for k2, v2 in
                                roofline(cfg, n, r["stage_ms"][n], b, f, pk).items()
                                if k2 in ("bound", "achieved", "unit", "frac")}
                            for n in ("route", "dispatch", "ffn_gate_up", "ffn_down", "combine")},
        "experts_touched": touched,
        "imbalance_factor": imbalance(cfg, r["counts"]),
        "gpu_launches": kernels_per_step(cfg, r.get("mode", "layer")) * r["steps"],
        "e2e": {"value": round(job_tokens_per_s(cfg.T, world, r["ms_e2e"]), 1),
                "unit": "tokens/s", "h2d_bytes_per_step": cfg.T * cfg.d * 2,
                "d2h_bytes_per_step": cfg.T * cfg.d * 2, "ms_per_step": round(r["ms_e2e"], 5)},
        "clocks": r["clocks"],
    }
    if full:
        out["gemm_roofline"] = {n: roofline(cfg, n, r["stage_ms"][n], b, f, pk)
                                for n in ("ffn_gate_up", "ffn_down")}
    return out


def time_placed(cfg, dev, W, steps, warm, spare_per_rank=4, seed=17):
    """The layer with redundant experts (32 spare slots at 8 ranks): a placement planned by
    moe_place_experts from the routing of another batch of the same workload (standing for past
    traffic), then timed on this batch. Reports the logical ranks' imbalance factor before
    (contiguous experts) and after (placed copies) on the timed batch."""
    import combine_grouped_gemm_gb300 as moe

    inp = synth.make_router_inputs(cfg, dev)
    other = synth.normal_bf16(cfg.seed + seed, synth.TAG_X, (cfg.T, cfg.d), cfg.x_std, dev)
    b = moe.Buffers(cfg, dev)
    moe.route(cfg, other, inp["w_gate"], inp["bias"], b["topk_idx"], b["topk_w"], b["ws"])
    load = np.bincount(b["topk_idx"].cpu().numpy().reshape(-1), minlength=cfg.E)
    del b
    S = cfg.E // cfg.R + spare_per_rank
    pl = moe.Placement.from_loads(load.astype(np.float64), cfg.R, S, max_copies=16, device=dev)
    lay = moe.MoELayer(cfg, inp["w_gate"], inp["bias"], weight_dict(W), dev, placement=pl)
    r = time_layer(cfg, inp, lay, steps, warm, dev)
    counts = r["counts"]                      # [R][slots] of the timed batch
    ti = lay.bufs["topk_idx"].cpu().numpy()
    per_expert = np.bincount(ti.reshape(-1), minlength=cfg.E)
    before = per_expert.reshape(cfg.R, -1).sum(1)
    after = counts.sum(0).reshape(cfg.R, -1).sum(1)
    nc = pl.n_copies.cpu().numpy()
    out = {"slots_per_rank": S, "redundant": int(cfg.R * S - cfg.E),
           "copies_of_hottest": int(nc[int(np.argmax(per_expert))]),
           "layer_us": round(r["ms"] * 1e3, 2),
           "tokens_per_s": round(job_tokens_per_s(cfg.T, 1, r["ms"]), 1),
           "stages_us": {n: round(v * 1e3, 2) for n, v in r["stage_ms"].items()},
           "imbalance_factor_contiguous": round(float(before.max() / before.mean()), 4),
           "imbalance_factor_placed": round(float(after.max() / after.mean()), 4),
           "slots_touched": int((counts.sum(0) > 0).sum()),
           "planned_from": "routing of another batch of the workload (seed + %d)" % seed}
    del lay, inp
    return out


def run_extras(args, dev, W_decode, pk):
    """The rest of the metric's token range in the same process: the decode sweep (the decode
    layer's weights at T = 8 .. 1024), the Zipf-skewed bf16 prefill (T = 4096) and the FP8
    prefill (T = 16384) with amax/448 and with power-of-two block scales. Each prefill's
    weights are made, timed and freed before the next."""
    steps = max(3, args.extra_steps)
    warm = max(3, args.warmup)
    out = {"sweep": []}
    dec = synth.CONFIGS["dsv3_decode"]
    out["variants"] = {dec.name: time_modes(dec, dev, W_decode, steps, warm,
                                            ("gather", "side", "side32", "side64",
                                             "gather+side", "fused", "gather+fused"))}
    for T in (8, 256, 1024):   # the fused stage across the sweep
        out["variants"][dec.with_T(T).name] = time_modes(dec.with_T(T), dev, W_decode, steps, warm,
                                                         ("layer", "gather", "fused",
                                                          "gather+fused"))
    out["placed"] = {dec.name: time_placed(dec, dev, W_decode, steps, warm)}
    for T in synth.SWEEP_T:
        cfg = dec.with_T(T)
        inp, _, lay = setup(cfg, dev, W=W_decode)
        r = time_layer(cfg, inp, lay, steps, warm, dev)
        s = summarise(cfg, r, pk, full=False)
        out["sweep"].append({k: s[k] for k in ("T", "layer_us", "tokens_per_s", "layer_hbm_frac",
                                               "stages_us", "experts_touched", "e2e",
                                               "gpu_launches")}
                            | {"sm_mhz": (r["clocks"] or {}).get("sm_mhz")})
        del lay, inp
    for key, name in (("skew_prefill", "dsv3_skew_prefill"), ("fp8_prefill", "dsv3_fp8_prefill"),
                      ("fp8_pow2_prefill", "dsv3_fp8_pow2_prefill")):
        cfg = synth.CONFIGS[name]
        torch.cuda.empty_cache()
        inp, W, lay = setup(cfg, dev)
        r = time_layer(cfg, inp, lay, steps, warm, dev)
        out[key] = summarise(cfg, r, pk)
        del lay, inp
        out["variants"][cfg.name] = time_modes(
            cfg, dev, W, steps, warm,
            ("gather", "side", "gather+side") + (("fused", "gather+fused") if cfg.act == "bf16"
                                                 else ()))
        out["placed"][cfg.name] = time_placed(cfg, dev, W, steps, warm)
        del W
        torch.cuda.empty_cache()
    return out


def oracle_sample(cfg, inp, W, tokens):
    """Times the oracle's steps on the given tokens, single-threaded: the router, the dispatch
    index, every routed expert row, the shared expert and the combine. Weight slices are copied
    to the host before the clock starts. Returns {stage: seconds}."""
    import oracle

    def bits(t):
        t = t.detach().cpu().contiguous()
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()

    x = bits(inp["x"])[tokens]
    wg = inp["w_gate"].cpu().numpy()
    b = inp["bias"].cpu().numpy()
    idx, _ = oracle.route(x, wg, b, cfg.k, cfg.n_group, cfg.topk_group, cfg.route_scale)
    fp8 = cfg.w == "fp8"
    experts = {}
    for e in np.unique(idx):
        e = int(e)
        experts[e] = dict(w13=bits(W["w13"][e]), w2=bits(W["w2"][e]))
        if fp8:
            experts[e]["w13_s"] = W["w13_s"][e].cpu().numpy()
            experts[e]["w2_s"] = W["w2_s"][e].cpu().numpy()
    S = None
    if cfg.d_ff_shared:
        S = dict(ws13=bits(W["ws13"]), ws2=bits(W["ws2"]))
        if fp8:
            S["ws13_s"] = W["ws13_s"].cpu().numpy()
            S["ws2_s"] = W["ws2_s"].cpu().numpy()
    n, k = len(tokens), cfg.k
    sec = {}
    t = time.perf_counter()
    idx, w = oracle.route(x, wg, b, cfg.k, cfg.n_group, cfg.topk_group, cfg.route_scale)
    sec["route"] = time.perf_counter() - t
    t = time.perf_counter()
    if fp8:
        xq, xs = oracle.quant_rows_e4m3(oracle.bf16_to_f32(x))
    sec["dispatch"] = time.perf_counter() - t   # the index pass below is negligible
    eo = np.empty((n, k, cfg.d), dtype=np.uint16)
    t = time.perf_counter()
    for j in range(n):
        for i in range(k):
            Wt = experts[int(idx[j, i])]
            if fp8:
                eo[j, i], _ = oracle.swiglu_row_fp8(xq[j], xs[j], Wt["w13"], Wt["w13_s"],
                                                    Wt["w2"], Wt["w2_s"])
            else:
                eo[j, i], _ = oracle.swiglu_row_bf16(x[j], Wt["w13"], Wt["w2"])
    sec["experts"] = time.perf_counter() - t
    sh = None
    t = time.perf_counter()
    if S is not None:
        sh = np.empty((n, cfg.d), dtype=np.uint16)
        for j in range(n):
            if fp8:
                sh[j], _ = oracle.swiglu_row_fp8(xq[j], xs[j], S["ws13"], S["ws13_s"], S["ws2"],
                                                 S["ws2_s"])
            else:
                sh[j], _ = oracle.swiglu_row_bf16(x[j], S["ws13"], S["ws2"])
    sec["shared"] = time.perf_counter() - t
    t = time.perf_counter()
    oracle.combine(eo.reshape(n * k, cfg.d), np.arange(n * k, dtype=np.int32).reshape(n, k), w, sh)
    sec["combine"] = time.perf_counter() - t
    return sec


def run_route_only(args, cfg):
    """The router stage (moe_route) alone: W untimed calls, then K calls timed back to back with
    CUDA events. The gate weight (7.3 MB for DSV3) stays in L2 between calls, unlike in the
    layer, where the expert GEMMs stream gigabytes between router calls."""
    import combine_grouped_gemm_gb300 as moe
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    inp = synth.make_router_inputs(cfg, dev)
    ws = torch.zeros(moe.query_sizes(cfg)["ws_bytes"], dtype=torch.uint8, device=dev)
    idx = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=dev)
    w = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev)
    for _ in range(max(1, args.warmup)):
        moe.route(cfg, inp["x"], inp["w_gate"], inp["bias"], idx, w, ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        moe.route(cfg, inp["x"], inp["w_gate"], inp["bias"], idx, w, ws)
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / args.steps
    flops = 2.0 * cfg.T * cfg.d * cfg.E
    print(json.dumps({"metric": "router stage us", "value": round(us, 2), "unit": "us",
                      "higher_is_better": False, "steps": args.steps, "warmup": args.warmup,
                      "config": describe(cfg),
                      "alu_frac": round(flops / (us * 1e-6) / (ALU_FP32_TFLOPS * 1e12), 4)}),
          flush=True)
    return 0


def main():
    args = parse()
    cfg = workload(args)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.gpus > 1 and world == 1:
        print(json.dumps({"error": "--gpus > 1 needs torchrun (one process per GPU)"}))
        return 2

    if args.impl == "reference":
        return run_reference(args, cfg, rank, world, local_rank)
    if args.route_only:
        return run_route_only(args, cfg)

    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)

    inp, W, lay = setup(cfg, dev, rank, world, mode=args.mode)
    r = time_layer(cfg, inp, lay, args.steps, args.warmup, dev, rank, world, local_rank)
    r["mode"] = args.mode
    if rank == 0:
        b, f, touched = algorithmic(cfg, r["counts"])
        pk = peaks()
        dom = max(r["stage_ms"], key=lambda n: r["stage_ms"][n])
        roof = roofline(cfg, dom, r["stage_ms"][dom], b, f, pk)
        s = summarise(cfg, r, pk, world)
        out = {
            "metric": METRIC, "value": s["tokens_per_s"], "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(r["ms"], 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": cfg.act,
            "data": "synthetic: seeded counter-based generator, random-init weights",
            "config": {**describe(cfg), "parallelism": f"replicas x{world}", "mode": args.mode,
                       "l2": "inputs larger than L2: ~%.1f GB of expert weights streamed per "
                             "step vs 129 MB L2" % (b["ffn_gate_up"] / 1e9 + b["ffn_down"] / 1e9)},
            **{k2: s[k2] for k2 in ("layer_us", "stages_us", "layer_hbm_frac", "stages_roofline",
                                    "experts_touched", "imbalance_factor", "gemm_roofline")},
            "roofline": roof,
            "gpu_launches": s["gpu_launches"],
            "clocks": r["clocks"],
            "e2e": s["e2e"],
        }
        if world == 1 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(cfg, inp, W, args.cpu_sample)
        else:
            out["cpu_baseline"] = None
        if world == 1 and args.extras and cfg.name == "dsv3_decode":
            del lay
            out.update(run_extras(args, dev, W, pk))
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


def cpu_baseline(cfg, inp, W, n_tokens=0, seconds=CPU_SAMPLE_SECONDS):
    """The oracle on a bounded sample of the workload's tokens, single-threaded: a 4-token probe
    sizes the sample to about `seconds` of CPU work (n_tokens > 0 fixes it instead). The sample
    runs in batches of 8 tokens, each copying only its own experts' weights to the host outside
    the clock, so host memory holds one batch's experts at a time."""
    rng = np.random.default_rng(0)
    n0 = min(cfg.T, 4)
    if n_tokens > 0:
        n = min(cfg.T, n_tokens)
    else:
        sec0 = sum(oracle_sample(cfg, inp, W, np.sort(rng.choice(cfg.T, n0, replace=False)))
                   .values())
        per_token = max(sec0, 1e-6) / n0
        n = int(min(cfg.T, max(n0, round(seconds / per_token))))
    tokens = np.sort(np.random.default_rng(1).choice(cfg.T, n, replace=False))
    stage = {}
    for i in range(0, n, 8):
        for key, v in oracle_sample(cfg, inp, W, tokens[i:i + 8]).items():
            stage[key] = stage.get(key, 0.0) + v
    sec = sum(stage.values())
    return {"value": round(n / sec, 4), "unit": "tokens/s", "cores": 1,
            "host_cores": os.cpu_count(), "kind": "oracle",
            "us_per_token": {key: round(v / n * 1e6, 1) for key, v in stage.items()},
            "sample": f"{n} of {cfg.T} tokens of {cfg.name}: route + k experts + shared + "
                      f"combine per token, {sec:.1f} s single-threaded"
                      + (f" (sized from a {n0}-token probe)" if n_tokens <= 0 else "")}


def run_reference(args, cfg, rank, world, local_rank):
    """The reference arm: the CPU oracle timed on this host's cores, each step a bounded
    sample (one token of the workload through the whole layer)."""
    if rank != 0:
        return 0
    dev = torch.device("cuda", local_rank) if torch.cuda.is_available() else torch.device("cpu")
    inp = synth.make_router_inputs(cfg, dev)
    W = synth.make_expert_weights(cfg, dev)
    rng = np.random.default_rng(1)
    for _ in range(args.warmup):
        oracle_sample(cfg, inp, W, rng.choice(cfg.T, 1))
    total = 0.0
    for _ in range(args.steps):
        total += sum(oracle_sample(cfg, inp, W, rng.choice(cfg.T, 1)).values())
    v = args.steps / total
    out = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "tokens/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": cfg.act,
           "data": "synthetic: seeded counter-based generator, random-init weights",
           "config": {**describe(cfg), "parallelism": "cpu oracle, 1 thread"},
           "cpu_baseline": {"value": round(v, 4), "unit": "tokens/s", "cores": 1,
                            "kind": "oracle",
                            "sample": f"1 token of {cfg.name} per step through the whole layer"},
           "e2e": {"value": round(v, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
