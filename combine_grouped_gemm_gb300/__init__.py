"""Python binding of libmoe, the GB300 (sm_103a) MoE-layer hot path.

Argument marshalling only: every function below passes device pointers of torch CUDA tensors
and the current CUDA stream to the C ABI declared in include/moe.h, and raises MoEError on a
non-zero return code. All the work runs in the library's CUDA kernels; there is no fallback.
If the shared library is missing, importing this package raises at once: build it with
``python combine_grouped_gemm_gb300/build.py``.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmoe.so")

MOE_BF16, MOE_FP8_E4M3, MOE_FP8_E4M3_POW2 = 0, 1, 2
MOE_DEV_TIMEOUT, MOE_DEV_BOUNDS, MOE_DEV_SCALE = 1, 2, 4
MOE_LAYER_EVENTS = 7
STAGE_NAMES = ["route", "dispatch", "ffn_setup", "ffn_gate_up", "ffn_down", "combine"]


class MoEError(RuntimeError):
    def __init__(self, fn, code, msg, cuda_err=0):
        super().__init__(f"{fn}: {msg} (code {code}" + (f", cudaError {cuda_err})" if cuda_err else ")"))
        self.code = code
        self.cuda_error = cuda_err


class Cfg(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("k", ctypes.c_int32), ("n_group", ctypes.c_int32),
                ("topk_group", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("d_ff_shared", ctypes.c_int32), ("R", ctypes.c_int32),
                ("route_scale", ctypes.c_float), ("act_dtype", ctypes.c_int32),
                ("w_dtype", ctypes.c_int32)]


class Sizes(ctypes.Structure):
    _fields_ = [("recv_rows", ctypes.c_int64), ("cap", ctypes.c_int32),
                ("recv_bytes", ctypes.c_size_t), ("recv_scale_bytes", ctypes.c_size_t),
                ("ebuf_bytes", ctypes.c_size_t), ("ws_bytes", ctypes.c_size_t)]


MOE_OPT_GATHER_X, MOE_OPT_SHARED_SIDE_STREAM, MOE_OPT_FUSED_FFN = 1, 2, 4


class PlacementC(ctypes.Structure):
    _fields_ = [("slots_per_rank", ctypes.c_int32), ("max_copies", ctypes.c_int32),
                ("slot_expert", ctypes.c_void_p), ("n_copies", ctypes.c_void_p),
                ("copy_slot", ctypes.c_void_p)]


class LayerOpts(ctypes.Structure):
    _fields_ = [("flags", ctypes.c_uint32), ("side_stream", ctypes.c_void_p),
                ("fork_event", ctypes.c_void_p), ("join_event", ctypes.c_void_p),
                ("side_ctas", ctypes.c_int32), ("placement", ctypes.POINTER(PlacementC))]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w13", "w13_scales", "w2", "w2_scales", "ws13", "ws13_scales", "ws2",
                 "ws2_scales")]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmoe.so not found at {LIB_PATH}; build it with "
                          "`python combine_grouped_gemm_gb300/build.py`")
    L = ctypes.CDLL(LIB_PATH)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
    sigs = {
        "moe_validate": [P],
        "moe_query_sizes": [P, P],
        "moe_route": [P, P, P, P, P, P, P, S],
        "moe_route_noalloc": [P, P, P, P, P, P, S],
        "moe_dispatch": [P, P, P, P, P, P, P, P, P, S],
        "moe_expert_ffn": [P, P, P, P, P, P, P, P, P, S],
        "moe_combine": [P, P, P, P, P, P, P, S],
        "moe_layer": [P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, S, P],
        "moe_layer_ex": [P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, S, P],
        "moe_dispatch_index": [P, P, P, P, P, P, S],
        "moe_place_experts": [I, I, I, P, I, P, P, P],
        "moe_query_sizes_placed": [P, I, P],
        "moe_expert_ffn_gather": [P, P, P, P, P, P, P, P, S],
        "moe_clear_status": [P, S],
        "moe_read_status": [P, P, S],
        "moe_selftest_wait": [P, ctypes.c_int64, S],
        "moe_strerror": [I],
        "moe_abi_version": [],
        "moe_last_cuda_error": [],
    }
    for name, args in sigs.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = ctypes.c_char_p if name == "moe_strerror" else ctypes.c_int
    return L


_lib = _load()

EXPORTED = ["moe_validate", "moe_query_sizes", "moe_route", "moe_route_noalloc", "moe_dispatch",
            "moe_expert_ffn", "moe_combine", "moe_layer", "moe_layer_ex", "moe_dispatch_index",
            "moe_expert_ffn_gather", "moe_place_experts", "moe_query_sizes_placed",
            "moe_clear_status", "moe_read_status", "moe_selftest_wait",
            "moe_strerror", "moe_abi_version", "moe_last_cuda_error"]


def _check(fn, rc):
    if rc != 0:
        err = _lib.moe_last_cuda_error() if rc == 4 else 0
        raise MoEError(fn, rc, _lib.moe_strerror(rc).decode(), err)


def _dtype_code(v):
    if isinstance(v, str):
        return MOE_FP8_E4M3 if v in ("fp8", "e4m3") else MOE_BF16
    return int(v)


def make_cfg(c) -> Cfg:
    """Cfg from any object with the moe_cfg fields (act / w may be "bf16" / "fp8"; an e4m3
    configuration with scales == "pow2" takes the power-of-two recipe)."""
    act = _dtype_code(getattr(c, "act_dtype", getattr(c, "act", MOE_BF16)))
    w = _dtype_code(getattr(c, "w_dtype", getattr(c, "w", act)))
    if getattr(c, "scales", "amax") == "pow2":
        act = MOE_FP8_E4M3_POW2 if act == MOE_FP8_E4M3 else act
        w = MOE_FP8_E4M3_POW2 if w == MOE_FP8_E4M3 else w
    return Cfg(c.T, c.d, c.E, c.k, c.n_group, c.topk_group, c.d_ff, c.d_ff_shared, c.R,
               float(c.route_scale), act, w)


def _p(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        return int(t)
    if not t.is_cuda:
        raise ValueError("libmoe takes CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("libmoe takes contiguous tensors")
    return t.data_ptr()


def _s(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


_WEIGHT_KEYS = ("w13", "w13_s", "w2", "w2_s", "ws13", "ws13_s", "ws2", "ws2_s")


def _weights(w: dict) -> Weights:
    """moe_weights from a dict with keys w13, w13_s, w2, w2_s, ws13, ws13_s, ws2, ws2_s."""
    return Weights(*[_p(w.get(n)) for n in _WEIGHT_KEYS])


def validate(cfg) -> int:
    return _lib.moe_validate(ctypes.byref(make_cfg(cfg)))


def query_sizes(cfg) -> dict:
    s = Sizes()
    _check("moe_query_sizes", _lib.moe_query_sizes(ctypes.byref(make_cfg(cfg)), ctypes.byref(s)))
    return {n: getattr(s, n) for n, _ in Sizes._fields_}


def query_sizes_placed(cfg, slots_per_rank) -> dict:
    s = Sizes()
    _check("moe_query_sizes_placed", _lib.moe_query_sizes_placed(
        ctypes.byref(make_cfg(cfg)), int(slots_per_rank), ctypes.byref(s)))
    return {n: getattr(s, n) for n, _ in Sizes._fields_}


def place_experts(load, R, slots_per_rank, max_copies=8):
    """moe_place_experts on the host: (slot_expert [R*S], n_copies [E], copy_slot [E][max])
    as numpy int32 arrays, from estimated loads [E]."""
    import numpy as np
    ld = np.ascontiguousarray(load, dtype=np.float64)
    E = ld.size
    se = np.empty(R * slots_per_rank, dtype=np.int32)
    nc = np.empty(E, dtype=np.int32)
    cs = np.empty((E, max_copies), dtype=np.int32)
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)   # noqa: E731
    _check("moe_place_experts", _lib.moe_place_experts(E, R, slots_per_rank, ptr(ld), max_copies,
                                                       ptr(se), ptr(nc), ptr(cs)))
    return se, nc, cs


class Placement:
    """A placement of the experts on slots (see moe_placement), held on the device."""

    def __init__(self, slot_expert, n_copies, copy_slot, slots_per_rank, device="cuda"):
        self.slots_per_rank = int(slots_per_rank)
        self.slot_expert = torch.as_tensor(slot_expert, dtype=torch.int32).to(device).contiguous()
        self.n_copies = torch.as_tensor(n_copies, dtype=torch.int32).to(device).contiguous()
        self.copy_slot = torch.as_tensor(copy_slot, dtype=torch.int32).to(device).contiguous()
        self.c = PlacementC(self.slots_per_rank, self.copy_slot.shape[1],
                            self.slot_expert.data_ptr(), self.n_copies.data_ptr(),
                            self.copy_slot.data_ptr())

    @classmethod
    def from_loads(cls, load, R, slots_per_rank, max_copies=8, device="cuda"):
        se, nc, cs = place_experts(load, R, slots_per_rank, max_copies)
        return cls(se, nc, cs, slots_per_rank, device)


def route(cfg, x, w_gate, bias, topk_idx, topk_w, ws, stream=None):
    _check("moe_route", _lib.moe_route(ctypes.byref(make_cfg(cfg)), _p(x), _p(w_gate), _p(bias),
                                       _p(topk_idx), _p(topk_w), _p(ws), _s(stream)))


def route_noalloc(cfg, x, w_gate, bias, topk_idx, topk_w, stream=None):
    """moe_route for callers that cannot supply a workspace: the library's own fixed device
    array holds the router's scratch (see moe_route_noalloc in include/moe.h)."""
    _check("moe_route_noalloc", _lib.moe_route_noalloc(ctypes.byref(make_cfg(cfg)), _p(x),
                                                       _p(w_gate), _p(bias), _p(topk_idx),
                                                       _p(topk_w), _s(stream)))


def dispatch(cfg, x, topk_idx, recv, recv_scales, counts, row_of, src_tok=None, stream=None,
             status=None):
    """status: None or a device tensor whose first 4 bytes receive MOE_DEV_* bits (e.g. ws)."""
    _check("moe_dispatch", _lib.moe_dispatch(ctypes.byref(make_cfg(cfg)), _p(x), _p(topk_idx),
                                             _p(recv), _p(recv_scales), _p(counts), _p(row_of),
                                             _p(src_tok), _p(status), _s(stream)))


def expert_ffn(cfg, recv, recv_scales, counts, x, weights: dict, ebuf, shared_out, ws,
               stream=None):
    w = _weights(weights)
    _check("moe_expert_ffn", _lib.moe_expert_ffn(ctypes.byref(make_cfg(cfg)), _p(recv),
                                                 _p(recv_scales), _p(counts), _p(x),
                                                 ctypes.byref(w), _p(ebuf), _p(shared_out),
                                                 _p(ws), _s(stream)))


def combine(cfg, ebuf, row_of, topk_w, shared_out, y, stream=None, status=None):
    _check("moe_combine", _lib.moe_combine(ctypes.byref(make_cfg(cfg)), _p(ebuf), _p(row_of),
                                           _p(topk_w), _p(shared_out), _p(y), _p(status),
                                           _s(stream)))


def layer(cfg, x, w_gate, bias, weights: dict, bufs: dict, y, stream=None, events=None):
    """The whole layer. bufs holds topk_idx, topk_w, recv, recv_scales, counts, row_of, ebuf,
    shared_out and ws (see Buffers). events: None or MOE_LAYER_EVENTS torch.cuda.Event that
    have been recorded once (so their handles exist)."""
    w = _weights(weights)
    ev = None
    if events is not None:
        arr = (ctypes.c_void_p * MOE_LAYER_EVENTS)(*[e.cuda_event for e in events])
        ev = ctypes.cast(arr, ctypes.c_void_p)
    b = bufs
    _check("moe_layer", _lib.moe_layer(ctypes.byref(make_cfg(cfg)), _p(x), _p(w_gate), _p(bias),
                                       ctypes.byref(w), _p(b["topk_idx"]), _p(b["topk_w"]),
                                       _p(b["recv"]), _p(b.get("recv_scales")), _p(b["counts"]),
                                       _p(b["row_of"]), _p(b["ebuf"]), _p(b.get("shared_out")),
                                       _p(y), _p(b["ws"]), _s(stream), ev))


def layer_ex(cfg, opts: LayerOpts | None, x, w_gate, bias, weights: dict, bufs: dict, y,
             stream=None, events=None):
    """moe_layer_ex: the layer with the variants of opts (None: moe_layer)."""
    w = _weights(weights)
    ev = None
    if events is not None:
        arr = (ctypes.c_void_p * MOE_LAYER_EVENTS)(*[e.cuda_event for e in events])
        ev = ctypes.cast(arr, ctypes.c_void_p)
    b = bufs
    _check("moe_layer_ex", _lib.moe_layer_ex(ctypes.byref(make_cfg(cfg)),
                                             ctypes.byref(opts) if opts is not None else None,
                                             _p(x), _p(w_gate), _p(bias), ctypes.byref(w),
                                             _p(b["topk_idx"]), _p(b["topk_w"]), _p(b.get("recv")),
                                             _p(b.get("recv_scales")), _p(b["counts"]),
                                             _p(b["row_of"]), _p(b["ebuf"]),
                                             _p(b.get("shared_out")), _p(y), _p(b["ws"]),
                                             _s(stream), ev))


def dispatch_index(cfg, topk_idx, counts, row_of, src_tok, stream=None, status=None):
    _check("moe_dispatch_index", _lib.moe_dispatch_index(ctypes.byref(make_cfg(cfg)), _p(topk_idx),
                                                         _p(counts), _p(row_of), _p(src_tok),
                                                         _p(status), _s(stream)))


def expert_ffn_gather(cfg, x, counts, src_tok, weights: dict, ebuf, shared_out, ws, stream=None):
    w = _weights(weights)
    _check("moe_expert_ffn_gather",
           _lib.moe_expert_ffn_gather(ctypes.byref(make_cfg(cfg)), _p(x), _p(counts), _p(src_tok),
                                      ctypes.byref(w), _p(ebuf), _p(shared_out), _p(ws),
                                      _s(stream)))


def clear_status(ws, stream=None):
    _check("moe_clear_status", _lib.moe_clear_status(_p(ws), _s(stream)))


def read_status(ws, stream=None) -> int:
    st = ctypes.c_uint32(0)
    _check("moe_read_status", _lib.moe_read_status(_p(ws), ctypes.byref(st), _s(stream)))
    return st.value


def selftest_wait(ws, limit_ns, stream=None):
    """Launches the library's wait diagnostic (see moe_selftest_wait): a kernel whose bounded
    waits run out after about limit_ns and set MOE_DEV_TIMEOUT in ws's status word."""
    _check("moe_selftest_wait", _lib.moe_selftest_wait(_p(ws), int(limit_ns), _s(stream)))


def abi_version() -> int:
    return _lib.moe_abi_version()


class Buffers(dict):
    """Device buffers of one layer configuration, allocated once with torch (the library itself
    allocates nothing)."""

    def __init__(self, cfg, device="cuda", with_recv=True, slots_per_rank=0):
        super().__init__()
        s = query_sizes_placed(cfg, slots_per_rank) if slots_per_rank else query_sizes(cfg)
        T, k, d, R, E = cfg.T, cfg.k, cfg.d, cfg.R, cfg.E
        if slots_per_rank:
            E = R * slots_per_rank     # counts are over the slots
        self.sizes = s
        fp8 = make_cfg(cfg).act_dtype != MOE_BF16
        self["topk_idx"] = torch.empty((T, k), dtype=torch.int32, device=device)
        self["topk_w"] = torch.empty((T, k), dtype=torch.float32, device=device)
        self["recv"] = (torch.empty((s["recv_rows"], d),
                                    dtype=torch.uint8 if fp8 else torch.bfloat16, device=device)
                        if with_recv else None)
        self["recv_scales"] = (torch.empty((d // 128, s["recv_rows"]), dtype=torch.float32,
                                           device=device) if fp8 and with_recv else None)
        self["counts"] = torch.empty((R, E), dtype=torch.int32, device=device)
        self["row_of"] = torch.empty((T, k), dtype=torch.int32, device=device)
        self["ebuf"] = torch.empty((s["recv_rows"], d), dtype=torch.bfloat16, device=device)
        self["shared_out"] = (torch.empty((T, d), dtype=torch.bfloat16, device=device)
                              if cfg.d_ff_shared else None)
        self["ws"] = torch.zeros(s["ws_bytes"], dtype=torch.uint8, device=device)


class MoELayer:
    """One MoE layer with resident weights: ``y = layer(x)`` runs router, dispatch, expert
    FFNs and combine on the current stream through ``moe_layer`` (``moe_layer_ex`` when a
    variant is asked for).

    gather: the expert GEMMs read routed rows from x by token (no receive-buffer copy; the
    receive buffers are not allocated). side_stream: the shared expert runs on a second stream
    of its own, limited to side_ctas CTAs per GEMM. placement: redundant experts on slots
    (Placement); the dispatch splits each expert's rows over its copies. fused: both expert
    GEMMs and the combine in one persistent launch (bf16)."""

    def __init__(self, cfg, w_gate, bias, weights: dict, device="cuda", gather=False,
                 side_stream=False, side_ctas=0, placement: Placement | None = None,
                 fused=False):
        self.cfg = cfg
        self.w_gate = w_gate
        self.bias = bias
        self.weights = weights
        self.placement = placement
        self.bufs = Buffers(cfg, device, with_recv=not gather,
                            slots_per_rank=placement.slots_per_rank if placement else 0)
        self.opts = None
        if gather or side_stream or fused or placement is not None:
            self.opts = LayerOpts(flags=(MOE_OPT_GATHER_X if gather else 0)
                                  | (MOE_OPT_SHARED_SIDE_STREAM if side_stream else 0)
                                  | (MOE_OPT_FUSED_FFN if fused else 0),
                                  side_ctas=int(side_ctas))
            if placement is not None:
                self.opts.placement = ctypes.pointer(placement.c)
            if side_stream:
                # the stream and events live as long as the layer object
                self._side = torch.cuda.Stream(device=device)
                self._fork = torch.cuda.Event()
                self._join = torch.cuda.Event()
                cur = torch.cuda.current_stream(device)
                self._fork.record(cur)      # gives the events their handles
                self._join.record(cur)
                torch.cuda.synchronize(device)
                self.opts.side_stream = self._side.cuda_stream
                self.opts.fork_event = self._fork.cuda_event
                self.opts.join_event = self._join.cuda_event

    def _run(self, x, y, stream, events):
        if self.opts is None:
            layer(self.cfg, x, self.w_gate, self.bias, self.weights, self.bufs, y, stream, events)
        else:
            layer_ex(self.cfg, self.opts, x, self.w_gate, self.bias, self.weights, self.bufs, y,
                     stream, events)

    def __call__(self, x, y=None, stream=None, events=None):
        if y is None:
            y = torch.empty((self.cfg.T, self.cfg.d), dtype=torch.bfloat16, device=x.device)
        self._run(x, y, stream, events)
        return y

    def run_host(self, x_host, y_host, stream=None):
        """Host-to-host call: copies x_host (pinned bf16 [T][d]) to the device, runs the layer
        and copies the output back into y_host (pinned), all enqueued on the stream. The caller
        synchronises before reading y_host."""
        if not hasattr(self, "_x_dev"):
            self._x_dev = torch.empty((self.cfg.T, self.cfg.d), dtype=torch.bfloat16,
                                      device=self.w_gate.device)
            self._y_dev = torch.empty_like(self._x_dev)
        s = stream or torch.cuda.current_stream()
        with torch.cuda.stream(s):
            self._x_dev.copy_(x_host, non_blocking=True)
            self._run(self._x_dev, self._y_dev, s, None)
            y_host.copy_(self._y_dev, non_blocking=True)
        return y_host
