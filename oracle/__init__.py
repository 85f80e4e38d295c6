"""CPU oracle for the MoE layer (test infrastructure).

A plain single-threaded C implementation (``moe_oracle.c``) of what the hot path computes,
loaded through ctypes, plus a few numpy helpers for the pages' metrics. Only the tests, the
smoke check and the bench's CPU-baseline leg use this package; the CUDA library never does.
It shares no code with the CUDA library: only the seeded input generator (``synth``) serves
both.

Every function takes and returns host numpy arrays. bf16 data travel as ``uint16`` bit
patterns and e4m3 data as ``uint8`` codes.

Parity pins: every function below is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle.py`` against something other than itself (brute force, closed forms,
invariants, textbook special cases, values printed on the pages).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmoe_oracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/_build (no -ffast-math, no contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_long
_F = ctypes.c_float

_SIGS = {
    "oracle_route": (_I, [_I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P, _P, _P, _P]),
    "oracle_select": (_I, [_I, _I, _I, _I, _I, _F, _P, _P, _P, _P]),
    "oracle_dispatch_index": (_I, [_I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "oracle_dispatch_payload": (None, [_I, _I, _I, _P, _P, _P, _P]),
    "oracle_dispatch_payload_ex": (None, [_I, _I, _I, _P, _P, _P, _P, _I]),
    "oracle_quant_row_e4m3": (None, [_P, _I, _P, _P]),
    "oracle_quant_row_e4m3_ex": (None, [_P, _I, _P, _P, _I]),
    "oracle_pow2_scale": (_F, [_F]),
    "oracle_swiglu_row_bf16": (None, [_I, _I, _P, _P, _P, _P, _P, _P]),
    "oracle_swiglu_row_fp8": (None, [_I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "oracle_swiglu_row_fp8_ex": (None, [_I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I]),
    "oracle_combine": (None, [_I, _I, _I, _P, _P, _P, _P, _P, _P]),
    "oracle_place_experts": (_I, [_I, _I, _I, _P, _I, _P, _P, _P]),
    "oracle_dispatch_index_placed": (_I, [_I, _I, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P]),
    "oracle_logit": (_F, [_P, _P, _I]),
    "oracle_exp_array": (None, [_L, _P, _P]),
    "oracle_sigmoid_array": (None, [_L, _P, _P]),
    "oracle_f32_to_e4m3_array": (None, [_L, _P, _P]),
    "oracle_e4m3_to_f32_array": (None, [_L, _P, _P]),
    "oracle_f32_to_bf16_array": (None, [_L, _P, _P]),
}


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------------------------------
# Number formats
# ------------------------------------------------------------------------------------------
def exp(z):
    z = _c(z, np.float32)
    out = np.empty_like(z)
    lib().oracle_exp_array(z.size, _ptr(z), _ptr(out))
    return out


def sigmoid(z):
    z = _c(z, np.float32)
    out = np.empty_like(z)
    lib().oracle_sigmoid_array(z.size, _ptr(z), _ptr(out))
    return out


def f32_to_e4m3(v):
    v = _c(v, np.float32)
    q = np.empty(v.shape, dtype=np.uint8)
    lib().oracle_f32_to_e4m3_array(v.size, _ptr(v), _ptr(q))
    return q


def e4m3_to_f32(q):
    q = _c(q, np.uint8)
    v = np.empty(q.shape, dtype=np.float32)
    lib().oracle_e4m3_to_f32_array(q.size, _ptr(q), _ptr(v))
    return v


def f32_to_bf16(v):
    v = _c(v, np.float32)
    h = np.empty(v.shape, dtype=np.uint16)
    lib().oracle_f32_to_bf16_array(v.size, _ptr(v), _ptr(h))
    return h


def bf16_to_f32(h):
    h = _c(h, np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


def quant_rows_e4m3(v, pow2=False):
    """1x128 block quantisation of each row of a float32 [n][m] array -> (codes, scales):
    scale amax/448 (reading R-i) or, with pow2, its power of two (reading R-l)."""
    v = _c(v, np.float32)
    n, m = v.shape
    q = np.empty((n, m), dtype=np.uint8)
    s = np.empty((n, m // 128), dtype=np.float32)
    for i in range(n):
        lib().oracle_quant_row_e4m3_ex(_ptr(v[i]), m, _ptr(q[i]), _ptr(s[i]), int(bool(pow2)))
    return q, s


def pow2_scale(amax):
    """Reading R-l's block scale for one amax (float32)."""
    return np.float32(lib().oracle_pow2_scale(float(np.float32(amax))))


# ------------------------------------------------------------------------------------------
# Router
# ------------------------------------------------------------------------------------------
def logit(x_row_bits, w_row):
    x = _c(x_row_bits, np.uint16)
    w = _c(w_row, np.float32)
    return float(lib().oracle_logit(_ptr(x), _ptr(w), x.size))


def route(x_bits, w_gate, bias, k, n_group, topk_group, route_scale, want_scores=False):
    """Router on every row of x. Returns (topk_idx int32 [T][k], topk_w f32 [T][k]) and, with
    want_scores, also (logits [T][E], sigmoid scores [T][E])."""
    x = _c(x_bits, np.uint16)
    wg = _c(w_gate, np.float32)
    b = _c(bias, np.float32)
    T, d = x.shape
    E = wg.shape[0]
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    z = np.empty((T, E), dtype=np.float32) if want_scores else None
    s = np.empty((T, E), dtype=np.float32) if want_scores else None
    rc = lib().oracle_route(T, d, E, k, n_group, topk_group, float(route_scale), _ptr(x),
                            _ptr(wg), _ptr(b), _ptr(idx), _ptr(w), _ptr(z), _ptr(s))
    if rc:
        raise ValueError("oracle_route: bad shape")
    return (idx, w, z, s) if want_scores else (idx, w)


def select(scores, bias, k, n_group, topk_group, route_scale):
    """Group-limited top-k from given sigmoid scores [T][E] (the router minus the gate GEMM)."""
    sc = _c(scores, np.float32)
    b = _c(bias, np.float32)
    T, E = sc.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    rc = lib().oracle_select(T, E, k, n_group, topk_group, float(route_scale), _ptr(sc), _ptr(b),
                             _ptr(idx), _ptr(w))
    if rc:
        raise ValueError("oracle_select: bad shape")
    return idx, w


# ------------------------------------------------------------------------------------------
# Dispatch
# ------------------------------------------------------------------------------------------
def dispatch_index(topk_idx, E, R):
    """Returns counts [R][E], offsets [R][E], row_of [T][k], src_tok [R*R*cap]."""
    ti = _c(topk_idx, np.int32)
    T, k = ti.shape
    Er = E // R
    cap = (T // R) * min(k, Er)
    counts = np.empty((R, E), dtype=np.int32)
    offsets = np.empty((R, E), dtype=np.int32)
    row_of = np.empty((T, k), dtype=np.int32)
    src_tok = np.empty(R * R * cap, dtype=np.int32)
    rc = lib().oracle_dispatch_index(T, E, k, R, _ptr(ti), _ptr(counts), _ptr(offsets),
                                     _ptr(row_of), _ptr(src_tok))
    if rc:
        raise ValueError("oracle_dispatch_index: bad shape")
    return counts, offsets, row_of, src_tok


def dispatch_payload(x_bits, row_of, n_rows, fp8=False, pow2=False):
    """Receive buffer [n_rows][d] (uint16 bf16 bits, or uint8 e4m3 codes plus f32 scales
    [n_rows][d/128], the scales of reading R-i or, with pow2, R-l); rows that receive nothing
    stay zero."""
    x = _c(x_bits, np.uint16)
    ro = _c(row_of, np.int32)
    T, d = x.shape
    k = ro.shape[1]
    if fp8:
        recv = np.zeros((n_rows, d), dtype=np.uint8)
        sc = np.zeros((n_rows, d // 128), dtype=np.float32)
    else:
        recv = np.zeros((n_rows, d), dtype=np.uint16)
        sc = None
    lib().oracle_dispatch_payload_ex(T, d, k, _ptr(x), _ptr(ro), _ptr(recv), _ptr(sc),
                                     int(bool(pow2)))
    return recv, sc


# ------------------------------------------------------------------------------------------
# Redundant experts (reading R-k)
# ------------------------------------------------------------------------------------------
def place_experts(load, R, S, max_copies=8):
    """Placement of E experts with R*S - E extra copies over R ranks of S slots, from estimated
    loads [E]. Returns (slot_expert [R*S], n_copies [E], copy_slot [E][max_copies])."""
    ld = _c(load, np.float64)
    E = ld.size
    se = np.empty(R * S, dtype=np.int32)
    nc = np.empty(E, dtype=np.int32)
    cs = np.empty((E, max_copies), dtype=np.int32)
    if lib().oracle_place_experts(E, R, S, _ptr(ld), max_copies, _ptr(se), _ptr(nc), _ptr(cs)):
        raise ValueError("oracle_place_experts: too few slots or too many copies")
    return se, nc, cs


def dispatch_index_placed(topk_idx, E, R, S, n_copies, copy_slot):
    """The dispatch index over the slots of a placement: counts [R][R*S], row_of [T][k],
    src_tok [R*R*cap] with cap = (T/R) * min(k, S)."""
    ti = _c(topk_idx, np.int32)
    nc = _c(n_copies, np.int32)
    cs = _c(copy_slot, np.int32)
    T, k = ti.shape
    cap = (T // R) * min(k, S)
    counts = np.empty((R, R * S), dtype=np.int32)
    row_of = np.empty((T, k), dtype=np.int32)
    src_tok = np.empty(R * R * cap, dtype=np.int32)
    if lib().oracle_dispatch_index_placed(T, E, k, R, S, _ptr(ti), _ptr(nc), _ptr(cs),
                                          cs.shape[1], _ptr(counts), _ptr(row_of),
                                          _ptr(src_tok)):
        raise ValueError("oracle_dispatch_index_placed: bad shape")
    return counts, row_of, src_tok


def rank_loads(counts, R):
    """Rows each rank receives: counts [sources][slots] summed per destination rank (slots in
    contiguous blocks of slots/R per rank)."""
    c = np.asarray(counts, dtype=np.int64).sum(axis=0)
    return c.reshape(R, -1).sum(axis=1)


# ------------------------------------------------------------------------------------------
# Experts and combine
# ------------------------------------------------------------------------------------------
def swiglu_row_bf16(x_row_bits, w13_bits, w2_bits, exact=False):
    """One bf16 row through one SwiGLU expert -> (out bf16 bits [d], h floats [F]); with exact,
    also the fp64 output before its rounding to bf16 [d]."""
    x = _c(x_row_bits, np.uint16)
    w13 = _c(w13_bits, np.uint16)
    w2 = _c(w2_bits, np.uint16)
    d = x.size
    F = w13.shape[0] // 2
    out = np.empty(d, dtype=np.uint16)
    h = np.empty(F, dtype=np.float32)
    ox = np.empty(d, dtype=np.float64) if exact else None
    lib().oracle_swiglu_row_bf16(d, F, _ptr(x), _ptr(w13), _ptr(w2), _ptr(out), _ptr(h), _ptr(ox))
    return (out, h, ox) if exact else (out, h)


def swiglu_row_fp8(xq, xs, w13q, w13s, w2q, w2s, exact=False, pow2=False):
    """One e4m3 row (codes + 1x128 scales) through one e4m3 expert -> (out bf16 [d], h [F]);
    with exact, also the fp64 output before its rounding to bf16 [d]. pow2: h is re-quantised
    with power-of-two scales (reading R-l)."""
    xq = _c(xq, np.uint8)
    xs = _c(xs, np.float32)
    w13q = _c(w13q, np.uint8)
    w13s = _c(w13s, np.float32)
    w2q = _c(w2q, np.uint8)
    w2s = _c(w2s, np.float32)
    d = xq.size
    F = w13q.shape[0] // 2
    out = np.empty(d, dtype=np.uint16)
    h = np.empty(F, dtype=np.float32)
    ox = np.empty(d, dtype=np.float64) if exact else None
    lib().oracle_swiglu_row_fp8_ex(d, F, _ptr(xq), _ptr(xs), _ptr(w13q), _ptr(w13s), _ptr(w2q),
                                   _ptr(w2s), _ptr(out), _ptr(h), _ptr(ox), int(bool(pow2)))
    return (out, h, ox) if exact else (out, h)


def combine(ebuf_bits, row_of, topk_w, shared_bits=None, exact=False):
    """y bf16 bits [T][d]; with exact, also the fp64 sums before their rounding [T][d]."""
    eb = _c(ebuf_bits, np.uint16)
    ro = _c(row_of, np.int32)
    w = _c(topk_w, np.float32)
    sh = None if shared_bits is None else _c(shared_bits, np.uint16)
    T, k = ro.shape
    d = eb.shape[1]
    y = np.empty((T, d), dtype=np.uint16)
    yx = np.empty((T, d), dtype=np.float64) if exact else None
    lib().oracle_combine(T, d, k, _ptr(eb), _ptr(ro), _ptr(w), _ptr(sh), _ptr(y), _ptr(yx))
    return (y, yx) if exact else y


# ------------------------------------------------------------------------------------------
# Metrics the pages define
# ------------------------------------------------------------------------------------------
def imbalance_factor(expert_counts, G):
    """Rank-level imbalance: max over ranks of the rank's load over the mean rank load, with
    expert e on rank e // (E/G) (Serving Mixture-of-Experts, Hot-Expert Skew section)."""
    c = np.asarray(expert_counts, dtype=np.float64).reshape(-1)
    loads = c.reshape(G, c.size // G).sum(axis=1)
    return float(loads.max() / loads.mean())


def distinct_experts(topk_idx):
    return int(np.unique(np.asarray(topk_idx).reshape(-1)).size)


# ------------------------------------------------------------------------------------------
# The layer, token by token
# ------------------------------------------------------------------------------------------
def layer_tokens(cfg, x_bits, w_gate, bias, expert_weights, shared_weights, tokens):
    """MoE layer output for the listed tokens.

    y[t] depends only on x[t] and the weights, so any subset of tokens can be computed alone.
    expert_weights: callable e -> dict(w13, w2, w13_s, w2_s) of host arrays (bf16 as uint16,
    e4m3 as uint8). shared_weights: dict(ws13, ws2, ws13_s, ws2_s) or None.
    Returns dict with topk_idx, topk_w, y (bf16 bits [n][d]), y_exact (the fp64 sums y is rounded
    from), expert_out (bf16 bits [n][k][d]) and shared_out (bf16 bits [n][d] or None)."""
    tokens = np.asarray(tokens, dtype=np.int64)
    xs = _c(x_bits[tokens], np.uint16)
    idx, w = route(xs, w_gate, bias, cfg.k, cfg.n_group, cfg.topk_group, cfg.route_scale)
    n, d = xs.shape
    fp8 = cfg.act == "fp8"
    p2 = getattr(cfg, "scales", "amax") == "pow2"
    if fp8:
        xq, xsc = quant_rows_e4m3(bf16_to_f32(xs), pow2=p2)
    cache = {}
    eo = np.empty((n, cfg.k, d), dtype=np.uint16)
    for j in range(n):
        for i in range(cfg.k):
            e = int(idx[j, i])
            if e not in cache:
                cache.clear()
                cache[e] = expert_weights(e)
            W = cache[e]
            if fp8:
                eo[j, i], _ = swiglu_row_fp8(xq[j], xsc[j], W["w13"], W["w13_s"], W["w2"], W["w2_s"],
                                             pow2=p2)
            else:
                eo[j, i], _ = swiglu_row_bf16(xs[j], W["w13"], W["w2"])
    sh = None
    if shared_weights is not None:
        sh = np.empty((n, d), dtype=np.uint16)
        for j in range(n):
            S = shared_weights
            if fp8:
                sh[j], _ = swiglu_row_fp8(xq[j], xsc[j], S["ws13"], S["ws13_s"], S["ws2"], S["ws2_s"],
                                          pow2=p2)
            else:
                sh[j], _ = swiglu_row_bf16(xs[j], S["ws13"], S["ws2"])
    rows = np.arange(n * cfg.k, dtype=np.int32).reshape(n, cfg.k)
    y, y_exact = combine(eo.reshape(n * cfg.k, d), rows, w, sh, exact=True)
    return dict(topk_idx=idx, topk_w=w, y=y, y_exact=y_exact, expert_out=eo, shared_out=sh)
