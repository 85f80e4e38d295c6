"""Seeded synthetic inputs for the MoE layer.

This module is shared by the CPU oracle's tests, the CUDA path's tests and the bench. It holds
no step of the MoE method (no routing, dispatch, expert or combine arithmetic): only a
counter-based random number generator, the value distributions of the workloads, and the
workload shapes themselves.

Generator definition:

* ``key(seed, tag)`` derives two 32-bit keys from the seed and a per-tensor tag.
* 32-bit word number ``c`` (a 64-bit counter) of a stream is
  ``mix(mix(lo32(c) ^ k0) ^ mix(hi32(c) ^ k1))`` where ``mix`` is the "lowbias32" integer hash
  (C. Wellons, 2018: xor-shift 16, multiply 0x7feb352d, xor-shift 15, multiply 0x846ca68b,
  xor-shift 16). All of it is integer arithmetic on int64 tensors kept below 2**63, so the words
  are the same on every device.
* Element ``i`` of a normal tensor uses words ``2i`` and ``2i+1`` as two uniforms,
  ``u1 = (w0 + 1) / 2**32`` in (0, 1] and ``u2 = w1 / 2**32`` in [0, 1), and takes the cosine
  branch of the Box-Muller transform (G. Box and M. Muller, 1958),
  ``z = sqrt(-2 ln u1) * cos(2 pi u2)``, a standard normal draw (|z| <= 6.66 at 32-bit
  resolution). ``z * std`` is computed in fp64 and rounded once to fp32. The fp64 log, sqrt and
  cos come from the device's math library, whose last bit can differ between devices; after
  the rounding to fp32 such a difference survives only for the rare draws within a few fp64
  ulps of an fp32 rounding boundary. Every check gives the oracle the host copy of the very
  tensor the CUDA path reads, so none depends on it.
* Uniform draws use the top 24 bits of word ``i`` (exact on every device).
* bf16 values are the fp32 value rounded to nearest even (torch's conversion); e4m3 weights
  are block-quantised from fp32 draws (see ``fp8_block_weights``).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch

M32 = 0xFFFFFFFF

# Per-tensor stream tags.
TAG_X, TAG_WGATE, TAG_BIAS, TAG_W13, TAG_W2, TAG_WS13, TAG_WS2, TAG_PERM = 1, 2, 3, 4, 5, 6, 7, 8

# Elements generated per torch call; bounds the temporaries (a few int64 tensors of this size).
_CHUNK = 1 << 26


# --------------------------------------------------------------------------------------------
# Workload shapes
# --------------------------------------------------------------------------------------------
@dataclass(frozen=True)
class MoEConfig:
    """Shape and value recipe of one MoE layer workload."""

    name: str
    T: int                # tokens
    d: int                # model width
    E: int                # routed experts
    k: int                # experts per token
    n_group: int          # expert groups for group-limited routing
    topk_group: int       # groups kept per token
    d_ff: int             # routed expert SwiGLU width
    d_ff_shared: int      # shared expert SwiGLU width (0 = no shared expert)
    R: int                # logical expert-parallel ranks
    route_scale: float    # scale applied to the renormalised gate weights
    act: str = "bf16"     # dispatched activation format: "bf16" or "fp8"
    w: str = "bf16"       # expert weight format: "bf16" or "fp8"
    bias: str = "uniform" # "uniform": U(-0.1, 0.1); "zipf": skewed popularity
    scales: str = "amax"  # e4m3 block scales: "amax" (amax/448) or "pow2" (its power of two)
    seed: int = 0
    x_std: float = 1.0
    w_std: float = 0.02
    wg_std: float = 0.02
    bias_range: float = 0.1

    def with_T(self, T: int) -> "MoEConfig":
        return replace(self, T=T, name=f"{self.name}_T{T}")

    def with_seed(self, seed: int) -> "MoEConfig":
        return replace(self, seed=seed)

    @property
    def E_r(self) -> int:
        return self.E // self.R

    @property
    def T_s(self) -> int:
        return self.T // self.R

    @property
    def cap(self) -> int:
        """Receive-segment capacity: the most rows one source rank can send one destination."""
        return self.T_s * min(self.k, self.E_r)


_DSV3 = dict(d=7168, E=256, k=8, n_group=8, topk_group=4, d_ff=2048, d_ff_shared=2048, R=8,
             route_scale=2.5)

CONFIGS = {
    # T=16, d=256, E=16, top-2, one group, d_ff=128, no shared expert, 2 logical ranks, seed 0.
    "tiny": MoEConfig("tiny", T=16, d=256, E=16, k=2, n_group=1, topk_group=1, d_ff=128,
                      d_ff_shared=0, R=2, route_scale=1.0, seed=0),
    # DeepSeek-V3-shaped decode layer, 64 tokens (8 per logical rank).
    "dsv3_decode": MoEConfig("dsv3_decode", T=64, seed=1000, **_DSV3),
    # The same layer swept over 1..128 tokens per logical rank.
    "dsv3_sweep": MoEConfig("dsv3_sweep", T=64, seed=2000, **_DSV3),
    # The same layer at 4096 tokens with Zipf(1.2)-skewed expert popularity.
    "dsv3_skew_prefill": MoEConfig("dsv3_skew_prefill", T=4096, bias="zipf", seed=3000, **_DSV3),
    # The same layer at 16384 tokens with e4m3 activations (1x128 scales) and e4m3 weights
    # (128x128 scales).
    "dsv3_fp8_prefill": MoEConfig("dsv3_fp8_prefill", T=16384, act="fp8", w="fp8", seed=4000,
                                  **_DSV3),
    # The FP8 prefill layer with power-of-two block scales (the block-scaled MMA's recipe).
    "dsv3_fp8_pow2_prefill": MoEConfig("dsv3_fp8_pow2_prefill", T=16384, act="fp8", w="fp8",
                                       scales="pow2", seed=4000, **_DSV3),
    # Profiling stand-in for the decode layer: the same per-expert shapes, 32 experts (E/R = 4
    # per logical rank, groups of 4), so one capture holds about 3 GB on the device.
    "dsv3_decode_e32": MoEConfig("dsv3_decode_e32", T=64, d=7168, E=32, k=8, n_group=8,
                                 topk_group=4, d_ff=2048, d_ff_shared=2048, R=8,
                                 route_scale=2.5, seed=1000),
    # Profiling stand-in for the bf16 prefill layer: the same per-expert shapes, 32 experts and
    # 512 tokens (128 rows per expert, as at T=4096 with 256 experts), ~2.9 GB of weights.
    "dsv3_prefill_e32": MoEConfig("dsv3_prefill_e32", T=512, d=7168, E=32, k=8, n_group=8,
                                  topk_group=4, d_ff=2048, d_ff_shared=2048, R=8,
                                  route_scale=2.5, seed=3000),
    # Profiling stand-in for the FP8 prefill layer: the same per-expert shapes, 32 experts and
    # 2048 tokens (512 rows per expert, as at T=16384 with 256 experts), ~1.5 GB of weights.
    "dsv3_fp8_e32": MoEConfig("dsv3_fp8_e32", T=2048, d=7168, E=32, k=8, n_group=8, topk_group=4,
                              d_ff=2048, d_ff_shared=2048, R=8, route_scale=2.5, act="fp8",
                              w="fp8", seed=4000),
    "dsv3_fp8_pow2_e32": MoEConfig("dsv3_fp8_pow2_e32", T=2048, d=7168, E=32, k=8, n_group=8,
                                   topk_group=4, d_ff=2048, d_ff_shared=2048, R=8,
                                   route_scale=2.5, act="fp8", w="fp8", scales="pow2",
                                   seed=4000),
}
SWEEP_T = [8 * m for m in (1, 2, 4, 8, 16, 32, 64, 128)]

# Bias strength for the skewed workload: b_e = ZIPF_ALPHA * (ln p_e - mean ln p) with
# p_e proportional to rank(e)^-ZIPF_S. Frozen from a bisection written by
# oracle/calibrate_skew.py (it runs the oracle router at T=4096 and targets a hottest-expert
# load of about 10x the mean).
ZIPF_S = 1.2
ZIPF_ALPHA = None  # filled in below by the calibration result


# --------------------------------------------------------------------------------------------
# Counter-based generator
# --------------------------------------------------------------------------------------------
def _mix32_int(h: int) -> int:
    h &= M32
    h ^= h >> 16
    h = (h * 0x7FEB352D) & M32
    h ^= h >> 15
    h = (h * 0x846CA68B) & M32
    h ^= h >> 16
    return h


def key(seed: int, tag: int) -> tuple[int, int]:
    """Two 32-bit stream keys for (seed, tag)."""
    a = _mix32_int((seed * 0x9E3779B9 + tag * 0x632BE5AB + 0x5BD1E995) & M32)
    b = _mix32_int(a ^ ((seed >> 32) & M32) ^ (tag * 0x85EBCA6B & M32) ^ 0x27D4EB2F)
    return a, b


def _mul32(x: torch.Tensor, c: int) -> torch.Tensor:
    """(x * c) mod 2**32 for x in [0, 2**32), without int64 overflow."""
    lo, hi = c & 0xFFFF, c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & M32


def _mix32(h: torch.Tensor) -> torch.Tensor:
    h = h ^ (h >> 16)
    h = _mul32(h, 0x7FEB352D)
    h = h ^ (h >> 15)
    h = _mul32(h, 0x846CA68B)
    h = h ^ (h >> 16)
    return h


def word(c: torch.Tensor, k0: int, k1: int) -> torch.Tensor:
    """32-bit word for each 64-bit counter in ``c`` (int64, non-negative)."""
    lo = c & M32
    hi = c >> 32
    return _mix32(_mix32(lo ^ k0) ^ _mix32(hi ^ k1))


def word_int(c: int, k0: int, k1: int) -> int:
    """Scalar restatement of ``word`` on Python ints (used to pin the tensor version)."""
    return _mix32_int(_mix32_int((c & M32) ^ k0) ^ _mix32_int(((c >> 32) & M32) ^ k1))


def _normal_f64(idx: torch.Tensor, k0: int, k1: int) -> torch.Tensor:
    """Standard normal draws for element indices ``idx`` (Box-Muller, cosine branch, fp64)."""
    u1 = (word(idx * 2, k0, k1) + 1).to(torch.float64) * 2.0 ** -32
    u2 = word(idx * 2 + 1, k0, k1).to(torch.float64) * 2.0 ** -32
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def _normal_f32_range(seed, tag, start, n, std, device):
    k0, k1 = key(seed, tag)
    idx = torch.arange(start, start + n, dtype=torch.int64, device=device)
    return (_normal_f64(idx, k0, k1) * float(std)).to(torch.float32)


def normal_f32(seed: int, tag: int, shape, std: float, device="cpu", start: int = 0):
    """fp32 tensor of normal draws with mean 0 and standard deviation ``std``.

    ``start`` offsets the element counter, so a slice of a large tensor can be made alone."""
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=torch.float32, device=device)
    for o in range(0, n, _CHUNK):
        m = min(_CHUNK, n - o)
        out[o:o + m] = _normal_f32_range(seed, tag, start + o, m, std, device)
    return out.view(*shape)


def normal_bf16(seed: int, tag: int, shape, std: float, device="cpu", start: int = 0):
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=torch.bfloat16, device=device)
    for o in range(0, n, _CHUNK):
        m = min(_CHUNK, n - o)
        out[o:o + m] = _normal_f32_range(seed, tag, start + o, m, std, device).to(torch.bfloat16)
    return out.view(*shape)


def uniform_sym_f32(seed: int, tag: int, n: int, a: float, device="cpu"):
    """fp32 draws on [-a, a): (2*u24 - 2**24) * (a / 2**24), one fp32 rounding."""
    k0, k1 = key(seed, tag)
    idx = torch.arange(n, dtype=torch.int64, device=device)
    u24 = word(idx, k0, k1) >> 8
    c = torch.tensor(np.float32(a / float(1 << 24)), dtype=torch.float32, device=device)
    return (2 * u24 - (1 << 24)).to(torch.float32) * c


def permutation(seed: int, tag: int, n: int) -> np.ndarray:
    """A seeded permutation of range(n): indices sorted by their random word."""
    k0, k1 = key(seed, tag)
    w = word(torch.arange(n, dtype=torch.int64), k0, k1).numpy()
    return np.argsort(w, kind="stable")


# --------------------------------------------------------------------------------------------
# Block-quantised e4m3 weights
# --------------------------------------------------------------------------------------------
def pow2_block_scale(amax: torch.Tensor) -> torch.Tensor:
    """The smallest power of two 2^e (-126 <= e <= 127) with amax <= 448 * 2^e, 1 where amax is
    0: a log2 estimate corrected by exact fp64 comparisons."""
    a = amax.double()
    e = torch.ceil(torch.log2(torch.where(a > 0, a, torch.ones_like(a)) / 448.0)).clamp(-126, 127)
    e = torch.where(a > 448.0 * torch.exp2(e), e + 1, e)
    e = torch.where((e > -126) & (a <= 448.0 * torch.exp2(e - 1)), e - 1, e).clamp(-126, 127)
    return torch.where(a > 0, torch.exp2(e), torch.ones_like(a)).float()


def fp8_block_weights(seed: int, tag: int, n_mat: int, rows: int, cols: int, std: float,
                      device="cpu", mat_start: int = 0, mat_count: int | None = None,
                      pow2: bool = False):
    """e4m3 weights [n_mat][rows][cols] (as uint8 codes) and fp32 scales
    [n_mat][rows/128][cols/128].

    Draws fp32 values, then per 128x128 block takes amax, scale = amax/448 (1 if amax is 0), or
    with pow2 the smallest power of two not below it, and codes = round-to-nearest-even e4m3
    of value/scale (torch's float8_e4m3fn conversion). Matrices
    ``mat_start .. mat_start+mat_count`` are made (a slice keeps the same values)."""
    if mat_count is None:
        mat_count = n_mat - mat_start
    assert rows % 128 == 0 and cols % 128 == 0
    q = torch.empty((mat_count, rows, cols), dtype=torch.uint8, device=device)
    s = torch.empty((mat_count, rows // 128, cols // 128), dtype=torch.float32, device=device)
    per = rows * cols
    for m in range(mat_count):
        w = normal_f32(seed, tag, (rows, cols), std, device, start=(mat_start + m) * per)
        blk = w.view(rows // 128, 128, cols // 128, 128)
        amax = blk.abs().amax(dim=(1, 3))
        if pow2:
            scale = pow2_block_scale(amax)
        else:
            scale = torch.where(amax > 0, amax / torch.tensor(448.0, device=device),
                                torch.ones_like(amax))
        qq = (blk / scale[:, None, :, None]).to(torch.float8_e4m3fn)
        q[m] = qq.view(torch.uint8).view(rows, cols)
        s[m] = scale
    return q, s


# --------------------------------------------------------------------------------------------
# Workload inputs
# --------------------------------------------------------------------------------------------
def zipf_bias(cfg: MoEConfig, alpha: float | None = None) -> torch.Tensor:
    """Per-expert bias giving Zipf(ZIPF_S) popularity over a seeded permutation."""
    if alpha is None:
        alpha = ZIPF_ALPHA
    perm = permutation(cfg.seed, TAG_PERM, cfg.E)
    lnp = -ZIPF_S * np.log(np.arange(1, cfg.E + 1, dtype=np.float64))
    b = np.empty(cfg.E, dtype=np.float64)
    b[perm] = alpha * (lnp - lnp.mean())
    return torch.from_numpy(b.astype(np.float32))


def make_router_inputs(cfg: MoEConfig, device="cpu"):
    x = normal_bf16(cfg.seed, TAG_X, (cfg.T, cfg.d), cfg.x_std, device)
    w_gate = normal_f32(cfg.seed, TAG_WGATE, (cfg.E, cfg.d), cfg.wg_std, device)
    if cfg.bias == "zipf":
        bias = zipf_bias(cfg).to(device)
    else:
        bias = uniform_sym_f32(cfg.seed, TAG_BIAS, cfg.E, cfg.bias_range, device)
    return dict(x=x, w_gate=w_gate, bias=bias)


def make_expert_weights(cfg: MoEConfig, device="cpu"):
    """Routed and shared expert weights in the library's K-major layout:
    w13 [E][2*d_ff][d] (rows 0..d_ff-1 gate, d_ff..2*d_ff-1 up), w2 [E][d][d_ff],
    ws13 [2*d_ff_shared][d], ws2 [d][d_ff_shared]; plus fp32 block scales for e4m3."""
    F, Fs, d, E = cfg.d_ff, cfg.d_ff_shared, cfg.d, cfg.E
    out = {}
    if cfg.w == "bf16":
        out["w13"] = normal_bf16(cfg.seed, TAG_W13, (E, 2 * F, d), cfg.w_std, device)
        out["w2"] = normal_bf16(cfg.seed, TAG_W2, (E, d, F), cfg.w_std, device)
        out["w13_s"] = out["w2_s"] = None
        if Fs:
            out["ws13"] = normal_bf16(cfg.seed, TAG_WS13, (2 * Fs, d), cfg.w_std, device)
            out["ws2"] = normal_bf16(cfg.seed, TAG_WS2, (d, Fs), cfg.w_std, device)
        out["ws13_s"] = out["ws2_s"] = None
    else:
        p2 = cfg.scales == "pow2"
        out["w13"], out["w13_s"] = fp8_block_weights(cfg.seed, TAG_W13, E, 2 * F, d, cfg.w_std,
                                                     device, pow2=p2)
        out["w2"], out["w2_s"] = fp8_block_weights(cfg.seed, TAG_W2, E, d, F, cfg.w_std, device,
                                                   pow2=p2)
        if Fs:
            q, s = fp8_block_weights(cfg.seed, TAG_WS13, 1, 2 * Fs, d, cfg.w_std, device, pow2=p2)
            out["ws13"], out["ws13_s"] = q[0], s[0]
            q, s = fp8_block_weights(cfg.seed, TAG_WS2, 1, d, Fs, cfg.w_std, device, pow2=p2)
            out["ws2"], out["ws2_s"] = q[0], s[0]
    if not Fs:
        out["ws13"] = out["ws2"] = out["ws13_s"] = out["ws2_s"] = None
    return out


def expert_weight_slice(cfg: MoEConfig, e: int, device="cpu"):
    """Weights of routed expert ``e`` alone (equal to slice ``e`` of make_expert_weights)."""
    F, d = cfg.d_ff, cfg.d
    if cfg.w == "bf16":
        w13 = normal_bf16(cfg.seed, TAG_W13, (2 * F, d), cfg.w_std, device, start=e * 2 * F * d)
        w2 = normal_bf16(cfg.seed, TAG_W2, (d, F), cfg.w_std, device, start=e * d * F)
        return dict(w13=w13, w2=w2, w13_s=None, w2_s=None)
    p2 = cfg.scales == "pow2"
    q13, s13 = fp8_block_weights(cfg.seed, TAG_W13, cfg.E, 2 * F, d, cfg.w_std, device,
                                 mat_start=e, mat_count=1, pow2=p2)
    q2, s2 = fp8_block_weights(cfg.seed, TAG_W2, cfg.E, d, F, cfg.w_std, device,
                               mat_start=e, mat_count=1, pow2=p2)
    return dict(w13=q13[0], w2=q2[0], w13_s=s13[0], w2_s=s2[0])


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


from synth._calibration import ZIPF_ALPHA as _ALPHA  # noqa: E402

ZIPF_ALPHA = _ALPHA
