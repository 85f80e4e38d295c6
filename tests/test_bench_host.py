"""bench.py's host-side arithmetic on CPU: kernels counted per step, the binding roof of each
stage with its achieved/peak/fraction fields, and the DRAM-traffic lookup that goes stale with
its kernel source."""
import hashlib
import json

import numpy as np
import pytest

import bench
import synth

C = synth.CONFIGS
PEAKS = {"hbm": 6781.1, "bf16": 1907.9, "bf16_sustained": 1700.0, "source": "measured"}


def test_kernels_per_step_follows_the_launch_structure():
    # route 2, dispatch 2, plan (+ row-list kernel beyond 1024 rows), gate/up, down, combine
    assert bench.kernels_per_step(C["tiny"]) == 8
    assert bench.kernels_per_step(C["dsv3_decode"]) == 8                 # 512 rows
    assert bench.kernels_per_step(C["dsv3_sweep"].with_T(128)) == 8      # 1024 rows
    assert bench.kernels_per_step(C["dsv3_sweep"].with_T(256)) == 9      # 2048 rows
    assert bench.kernels_per_step(C["dsv3_skew_prefill"]) == 9
    # + the e4m3 quantisation of the shared expert's input
    assert bench.kernels_per_step(C["dsv3_fp8_prefill"]) == 10
    # the power-of-two recipe adds the scale-byte pass before each gate/up launch
    assert bench.kernels_per_step(C["dsv3_fp8_pow2_prefill"]) == 11
    assert bench.kernels_per_step(C["dsv3_fp8_pow2_prefill"], "side") == 14


def test_kernels_per_step_of_the_layer_variants():
    dec, f8 = C["dsv3_decode"], C["dsv3_fp8_prefill"]
    assert bench.kernels_per_step(dec, "gather") == 7          # no copy kernel
    assert bench.kernels_per_step(dec, "side") == 10           # + the shared expert's 2 GEMMs
    assert bench.kernels_per_step(dec, "fused") == 6           # GEMMs and combine in one launch
    assert bench.kernels_per_step(dec, "gather+fused") == 5
    assert bench.kernels_per_step(C["tiny"], "side") == 8      # no shared expert: nothing moves
    # e4m3: the quantisation of x runs for the shared expert and for gather mode alike
    assert bench.kernels_per_step(f8, "gather") == 9
    # without a shared expert gather mode swaps the dispatch's e4m3 copy for the quantisation
    assert bench.kernels_per_step(dataclasses_replace(f8, d_ff_shared=0), "gather") == 9
    assert bench.kernels_per_step(dataclasses_replace(f8, d_ff_shared=0), "layer") == 9


def dataclasses_replace(cfg, **kw):
    import dataclasses
    return dataclasses.replace(cfg, **kw)


def _counts(cfg, touched):
    c = np.zeros((cfg.R, cfg.E), dtype=np.int64)
    c[0, :touched] = 1
    return c


def test_touched_experts_scale_the_weight_bytes():
    cfg = C["dsv3_decode"]
    b1, _, t1 = bench.algorithmic(cfg, _counts(cfg, 100))
    b2, _, t2 = bench.algorithmic(cfg, _counts(cfg, 101))
    assert (t1, t2) == (100, 101)
    # one more touched expert streams one more expert's gate/up and down weights
    assert b2["ffn_gate_up"] - b1["ffn_gate_up"] == 2 * cfg.d_ff * cfg.d * 2
    assert b2["ffn_down"] - b1["ffn_down"] == cfg.d * cfg.d_ff * 2
    # e4m3 weights: half the bytes plus one fp32 scale per 128x128 block
    f8 = C["dsv3_fp8_prefill"]
    b8a, _, _ = bench.algorithmic(f8, _counts(f8, 100))
    b8b, _, _ = bench.algorithmic(f8, _counts(f8, 101))
    assert b8b["ffn_gate_up"] - b8a["ffn_gate_up"] == (2 * f8.d_ff * f8.d
                                                       + (2 * f8.d_ff // 128) * (f8.d // 128) * 4)


def test_binding_roof_per_stage():
    dec = C["dsv3_decode"]
    b, f, _ = bench.algorithmic(dec, _counts(dec, 135))
    r = bench.roofline(dec, "ffn_gate_up", 1.15, b, f, PEAKS)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == PEAKS["hbm"]
    assert r["achieved"] == pytest.approx(b["ffn_gate_up"] / 1.15e-3 / 1e9, rel=1e-4)
    assert r["frac"] == pytest.approx(r["achieved"] / PEAKS["hbm"], rel=1e-3)
    # the router: reading W_g binds at T=8, its fp32 FMAs from T of a few dozen on
    small = C["dsv3_sweep"].with_T(8)
    bs, fs, _ = bench.algorithmic(small, _counts(small, 50))
    assert bench.roofline(small, "route", 0.02, bs, fs, PEAKS)["bound"] == "hbm"
    ra = bench.roofline(dec, "route", 0.03, b, f, PEAKS)
    assert ra["bound"] == "alu" and ra["peak"] == pytest.approx(80.5, abs=0.1)
    assert ra["achieved"] == pytest.approx(f["route"] / 0.03e-3 / 1e12, abs=0.05)   # 0.1 rounding
    # FP8 prefill GEMMs: the tensor roof, e4m3 = 2 x the measured bf16 burst
    f8 = C["dsv3_fp8_prefill"]
    b8, f8l, _ = bench.algorithmic(f8, _counts(f8, 256))
    rt = bench.roofline(f8, "ffn_gate_up", 5.0, b8, f8l, PEAKS)
    assert rt["bound"] == "tensor" and rt["peak"] == pytest.approx(2 * PEAKS["bf16"])
    assert rt["frac"] == pytest.approx(f8l["ffn_gate_up"] / 5e-3 / 1e12 / (2 * PEAKS["bf16"]),
                                       rel=1e-3)


def test_traffic_lookup_goes_stale_with_its_kernel_source(tmp_path, monkeypatch):
    src = tmp_path / "kernel.cu"
    hdr = tmp_path / "kernel.cuh"
    src.write_text("first version\n")
    hdr.write_text("header\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.sources_hash(["kernel.cu", "kernel.cuh"])
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"ffn_gate_up@w": {"sources": ["kernel.cu", "kernel.cuh"], "sources_sha256_16": h,
                           "dram_bytes_per_launch": 123},
         "ffn_down@dsv3_decode_e32": {"sources": ["kernel.cu", "kernel.cuh"],
                                      "sources_sha256_16": h, "dram_bytes_per_launch": 1100,
                                      "algorithmic_bytes_per_launch": 1000}}))
    assert bench.measured_traffic("ffn_gate_up", "w", 999)[0] == 123      # its own capture
    assert bench.measured_traffic("ffn_down", "w", 999)[0] is None        # none at all
    # the full decode launch scaled from its stand-in: 1.1 x its own algorithmic bytes
    t, note = bench.measured_traffic("ffn_down", "dsv3_decode", 50000)
    assert t == 55000 and "dsv3_decode_e32" in note
    hdr.write_text("second version\n")                                   # any source changes
    assert bench.measured_traffic("ffn_gate_up", "w", 999)[0] is None
    assert bench.measured_traffic("ffn_down", "dsv3_decode", 50000)[0] is None


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_under_two_ranks(rank):
    # bench.py --impl reference as torchrun would start it with two ranks: rank 0 times the
    # oracle and prints one JSON line, the other rank exits 0 without work
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank),
               MASTER_ADDR="127.0.0.1", MASTER_PORT="29533")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--workload", "tiny", "--steps", "2", "--warmup", "1"],
                       cwd=root, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    if rank:
        assert lines == []
        return
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["value"] > 0 and out["unit"] == "tokens/s"
    assert out["cpu_baseline"]["kind"] == "oracle" and out["cpu_baseline"]["value"] == out["value"]
    assert out["e2e"] == {"value": out["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}


def test_cpu_baseline_sizes_its_sample_from_the_probe():
    cfg = C["tiny"]
    inp = synth.make_router_inputs(cfg, "cpu")
    W = synth.make_expert_weights(cfg, "cpu")
    # a tiny layer: a second of oracle work covers every token
    out = bench.cpu_baseline(cfg, inp, W, seconds=1.0)
    assert out["kind"] == "oracle" and out["cores"] == 1 and out["value"] > 0
    assert out["sample"].startswith(f"{cfg.T} of {cfg.T} tokens")
    # a fixed size is taken as given, in batches of 8
    out = bench.cpu_baseline(cfg, inp, W, n_tokens=11)
    assert out["sample"].startswith(f"11 of {cfg.T} tokens")


@pytest.mark.gpu
def test_route_only_mode_times_the_router_and_prints_one_line():
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--workload", "tiny",
                        "--route-only", "--steps", "3", "--warmup", "1"],
                       cwd=root, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    out = json.loads(lines[0])
    assert out["metric"] == "router stage us" and out["value"] > 0
    assert out["config"]["workload"] == "tiny"
