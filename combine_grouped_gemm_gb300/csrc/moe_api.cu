// C ABI of libmoe (declared in include/moe.h): argument checks, workspace layout, and the
// launch sequence router -> dispatch -> expert FFN (schedule, gate/up GEMM, down GEMM) ->
// combine on the caller's stream. Nothing here allocates memory or waits for the device,
// except moe_read_status.
#include <math.h>
#include <stdlib.h>

#include <algorithm>

#include "moe_internal.h"

// NVTX ranges around the layer's stages, so a profiler's timeline (or `ncu --nvtx`) can tell
// them apart. NVTX is header-only: without a profiler attached a range costs a pointer check.
#if __has_include(<nvtx3/nvToolsExt.h>)
#include <nvtx3/nvToolsExt.h>
#define MOE_NVTX 1
#else
#define MOE_NVTX 0
#endif

namespace moe {

namespace {
thread_local int g_last_cuda_error = 0;
}  // namespace

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return MOE_ERR_CUDA;
}

namespace {
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t up256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// one NVTX range for the lifetime of the object (no-op without the NVTX header)
struct StageRange {
  explicit StageRange(const char* name) {
#if MOE_NVTX
    nvtxRangePushA(name);
#else
    (void)name;
#endif
  }
  ~StageRange() {
#if MOE_NVTX
    nvtxRangePop();
#endif
  }
  StageRange(const StageRange&) = delete;
  StageRange& operator=(const StageRange&) = delete;
};

}  // namespace

int validate(const moe_cfg& c) {
  if (c.T < 1 || c.d < 1 || c.E < 1 || c.k < 1 || c.n_group < 1 || c.topk_group < 1 ||
      c.d_ff < 1 || c.d_ff_shared < 0 || c.R < 1)
    return MOE_ERR_INVALID_ARG;
  if (c.T % c.R || c.E % c.R || c.E % c.n_group) return MOE_ERR_INVALID_ARG;
  if (c.topk_group > c.n_group || c.k > c.topk_group * (c.E / c.n_group))
    return MOE_ERR_INVALID_ARG;
  if (c.act_dtype < MOE_BF16 || c.act_dtype > MOE_FP8_E4M3_POW2 || c.w_dtype < MOE_BF16 ||
      c.w_dtype > MOE_FP8_E4M3_POW2)
    return MOE_ERR_INVALID_ARG;
  if (!isfinite(c.route_scale)) return MOE_ERR_INVALID_ARG;
  // limits of these kernels
  if (c.d % 128 || c.d_ff % 128 || c.d_ff_shared % 128) return MOE_ERR_UNSUPPORTED;
  if (c.E > 1024 || c.k > 32 || c.n_group > 64 || c.R > 64) return MOE_ERR_UNSUPPORTED;
  if (c.act_dtype != c.w_dtype) return MOE_ERR_UNSUPPORTED;
  if (c.d_ff_shared != 0 && c.d_ff_shared != c.d_ff) return MOE_ERR_UNSUPPORTED;
  // the block-scaled down GEMM computes two 128-column output tiles per unit
  if (c.act_dtype == MOE_FP8_E4M3_POW2 && c.d % 256) return MOE_ERR_UNSUPPORTED;
  // ... and keeps a row's scale bytes (one per 128-column block) in 64 bytes
  if (c.act_dtype == MOE_FP8_E4M3_POW2 && (c.d > 128 * kSfRowBytes || c.d_ff > 128 * kSfRowBytes))
    return MOE_ERR_UNSUPPORTED;
  const long long rows = (long long)c.R * c.R * cap_of(c);
  if (rows >= (1ll << 31) || (long long)c.T * c.k >= (1ll << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

WsLayout ws_layout(const moe_cfg& c) {
  WsLayout L{};
  const size_t tk = (size_t)c.T * c.k;
  const size_t ab = act_bytes(c);
  const bool fp8 = is_fp8(c);
  // token tile: 128 rows for e4m3 (the token rows are the M operand there) and for bf16 when
  // experts average 16 rows or more; 64 otherwise (DSV3 layer: 128 is 2-17 % faster from 512
  // tokens, 64 is 1.5 % faster at 256)
  L.bn = (fp8 || tk >= (size_t)16 * c.E) ? 128 : 64;
  L.max_tiles = c.E + (int)((tk + L.bn - 1) / L.bn);
  size_t o = 0;
  L.status = o;     o = up256(o + 16);
  L.partials = o;   o = up256(o + sizeof(float) * kRouteChunks * (size_t)c.T * c.E);
  L.grp_n = o;      o = up256(o + sizeof(int32_t) * c.E);
  L.grp_off = o;    o = up256(o + sizeof(int32_t) * c.E);
  L.n_tiles = o;    o = up256(o + 2 * sizeof(int32_t));   // tiles, of which hot (listed first)
  L.tiles = o;      o = up256(o + sizeof(Tile) * (size_t)L.max_tiles);
  L.row_list = o;   o = up256(o + sizeof(int32_t) * tk);
  L.h = o;          o = up256(o + ab * tk * c.d_ff);
  L.h_scales = o;   o = up256(o + (fp8 ? sizeof(float) * tk * (c.d_ff / 128) : 0));
  L.hs = o;         o = up256(o + ab * (size_t)c.T * c.d_ff_shared);
  L.hs_scales = o;  o = up256(o + (fp8 ? sizeof(float) * (size_t)c.T * (c.d_ff_shared / 128) : 0));
  L.xq = o;         o = up256(o + (fp8 ? (size_t)c.T * c.d : 0));
  L.xq_scales = o;  o = up256(o + (fp8 ? sizeof(float) * (size_t)c.T * (c.d / 128) : 0));
  L.run_start = o;  o = up256(o + sizeof(int32_t) * (size_t)c.R * c.E);
  L.run_pre = o;    o = up256(o + sizeof(int32_t) * (size_t)c.R * c.E);
  L.src_tok = o;    o = up256(o + sizeof(int32_t) * (size_t)c.R * c.R * cap_of(c));
  L.tok_list = o;   o = up256(o + sizeof(int32_t) * tk);
  L.grp_order = o;  o = up256(o + sizeof(int32_t) * c.E);
  L.shared_tiles = c.d_ff_shared ? (c.T + L.bn - 1) / L.bn : 0;
  L.fused_done_n = L.max_tiles + L.shared_tiles + 2;
  L.fused_done = o; o = up256(o + sizeof(int32_t) * (size_t)L.fused_done_n);
  const bool p2 = pow2_scales(c);
  L.sf_gu = o;      o = up256(o + (p2 ? (size_t)kSfRowBytes * tk : 0));
  L.sf_x = o;       o = up256(o + (p2 ? (size_t)kSfRowBytes * c.T : 0));
  L.sf_h = o;       o = up256(o + (p2 ? (size_t)kSfRowBytes * tk : 0));
  L.sf_hs = o;      o = up256(o + (p2 ? (size_t)kSfRowBytes * c.T : 0));
  L.max_tiles2 = c.E + (int)((tk + 2 * L.bn - 1) / (2 * L.bn));
  L.n_tiles2 = o;   o = up256(o + 2 * sizeof(int32_t));
  L.tiles2 = o;     o = up256(o + sizeof(Tile) * (size_t)L.max_tiles2);
  L.total = o;
  return L;
}

}  // namespace moe

using namespace moe;

#define MOE_CHECK_CFG(cfg)                      \
  do {                                          \
    if (!(cfg)) return MOE_ERR_INVALID_ARG;     \
    const int rc_ = validate(*(cfg));           \
    if (rc_ != MOE_OK) return rc_;              \
  } while (0)

#define MOE_NEED(p)                              \
  do {                                           \
    if (!(p)) return MOE_ERR_INVALID_ARG;        \
    if (!aligned16(p)) return MOE_ERR_MISALIGNED; \
  } while (0)

#define MOE_OPT(p)                                      \
  do {                                                  \
    if ((p) && !aligned16(p)) return MOE_ERR_MISALIGNED; \
  } while (0)

extern "C" {

int moe_abi_version(void) { return MOE_ABI_VERSION; }

int moe_last_cuda_error(void) { return g_last_cuda_error; }

const char* moe_strerror(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (shape constraint or NULL pointer)";
    case MOE_ERR_UNSUPPORTED: return "shape not supported by these kernels";
    case MOE_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
    case MOE_ERR_CUDA: return "CUDA call or kernel launch failed";
    default: return "unknown error code";
  }
}

int moe_validate(const moe_cfg* cfg) {
  MOE_CHECK_CFG(cfg);
  return MOE_OK;
}

namespace {
void fill_sizes(const moe_cfg& c, moe_sizes* out) {
  const int cap = cap_of(c);
  out->cap = cap;
  out->recv_rows = (int64_t)c.R * c.R * cap;
  out->recv_bytes = (size_t)out->recv_rows * c.d * act_bytes(c);
  out->recv_scale_bytes =
      is_fp8(c) ? (size_t)out->recv_rows * (c.d / 128) * sizeof(float) : 0;
  out->ebuf_bytes = (size_t)out->recv_rows * c.d * 2;
  out->ws_bytes = ws_layout(c).total;
}
}  // namespace

int moe_query_sizes(const moe_cfg* cfg, moe_sizes* out) {
  MOE_CHECK_CFG(cfg);
  if (!out) return MOE_ERR_INVALID_ARG;
  fill_sizes(*cfg, out);
  return MOE_OK;
}

int moe_query_sizes_placed(const moe_cfg* cfg, int32_t slots_per_rank, moe_sizes* out) {
  MOE_CHECK_CFG(cfg);
  if (!out || slots_per_rank < 1 || (long long)slots_per_rank * cfg->R < cfg->E)
    return MOE_ERR_INVALID_ARG;
  if ((long long)slots_per_rank * cfg->R > 1024) return MOE_ERR_UNSUPPORTED;
  moe_placement p{};
  p.slots_per_rank = slots_per_rank;
  const moe_cfg cs = slot_cfg(*cfg, &p);
  const int rc = validate(cs);
  if (rc != MOE_OK) return rc;
  fill_sizes(cs, out);
  return MOE_OK;
}

int moe_place_experts(int32_t E, int32_t R, int32_t S, const double* load, int32_t max_copies,
                      int32_t* slot_expert, int32_t* n_copies, int32_t* copy_slot) {
  if (!load || !slot_expert || !n_copies || !copy_slot) return MOE_ERR_INVALID_ARG;
  if (E < 1 || R < 1 || S < 1 || max_copies < 1) return MOE_ERR_INVALID_ARG;
  const long long G = (long long)R * S;
  if (G < E || G > (1 << 20)) return MOE_ERR_INVALID_ARG;
  for (int e = 0; e < E; ++e)
    if (!(load[e] >= 0.0) || !isfinite(load[e])) return MOE_ERR_INVALID_ARG;
  // copies: each spare slot to the largest load per copy (first maximum: lower expert)
  for (int e = 0; e < E; ++e) n_copies[e] = 1;
  for (long long spare = G - E; spare > 0; --spare) {
    int best = 0;
    double best_share = load[0] / n_copies[0];
    for (int e = 1; e < E; ++e) {
      const double share = load[e] / n_copies[e];
      if (share > best_share) {
        best = e;
        best_share = share;
      }
    }
    if (++n_copies[best] > max_copies) return MOE_ERR_INVALID_ARG;
  }
  // the copies in placement order: share descending, then expert, then copy ascending
  struct Copy {
    double share;
    int e, c, rank;
  };
  Copy* list = static_cast<Copy*>(malloc(sizeof(Copy) * (size_t)G));
  double* rank_load = static_cast<double*>(calloc((size_t)R, sizeof(double)));
  int* rank_fill = static_cast<int*>(calloc((size_t)R, sizeof(int)));
  if (!list || !rank_load || !rank_fill) {
    free(list);
    free(rank_load);
    free(rank_fill);
    return MOE_ERR_INVALID_ARG;
  }
  long long n = 0;
  for (int e = 0; e < E; ++e)
    for (int c = 0; c < n_copies[e]; ++c) list[n++] = Copy{load[e] / n_copies[e], e, c, -1};
  std::stable_sort(list, list + n, [](const Copy& a, const Copy& b) { return a.share > b.share; });
  // largest first onto the least-loaded rank with a free slot (first minimum: lower rank)
  for (long long i = 0; i < n; ++i) {
    int r_min = -1;
    for (int r = 0; r < R; ++r)
      if (rank_fill[r] < S && (r_min < 0 || rank_load[r] < rank_load[r_min])) r_min = r;
    list[i].rank = r_min;
    rank_load[r_min] += list[i].share;
    ++rank_fill[r_min];
  }
  // slots of a rank in (expert, copy) order: sort by (rank, expert, copy)
  std::sort(list, list + n, [](const Copy& a, const Copy& b) {
    if (a.rank != b.rank) return a.rank < b.rank;
    if (a.e != b.e) return a.e < b.e;
    return a.c < b.c;
  });
  for (long long p = 0; p < G; ++p) slot_expert[p] = list[p].e;
  for (long long i = 0; i < (long long)E * max_copies; ++i) copy_slot[i] = -1;
  for (int e = 0; e < E; ++e) n_copies[e] = 0;
  for (long long p = 0; p < G; ++p) {
    const int e = slot_expert[p];
    copy_slot[(long long)e * max_copies + n_copies[e]++] = static_cast<int32_t>(p);
  }
  free(list);
  free(rank_load);
  free(rank_fill);
  return MOE_OK;
}

int moe_route(const moe_cfg* cfg, const void* x, const float* w_gate, const float* bias,
              int32_t* topk_idx, float* topk_w, void* ws, cudaStream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_NEED(x);
  MOE_NEED(w_gate);
  MOE_NEED(bias);
  MOE_NEED(topk_idx);
  MOE_NEED(topk_w);
  MOE_NEED(ws);
  const WsLayout L = ws_layout(*cfg);
  char* w = static_cast<char*>(ws);
  cudaError_t e = launch_route(*cfg, x, w_gate, bias, topk_idx, topk_w,
                               reinterpret_cast<float*>(w + L.partials),
                               reinterpret_cast<uint32_t*>(w + L.status), stream);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

int moe_dispatch(const moe_cfg* cfg, const void* x, const int32_t* topk_idx, void* recv,
                 float* recv_scales, int32_t* counts, int32_t* row_of, int32_t* src_tok,
                 uint32_t* status, cudaStream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_NEED(x);
  MOE_NEED(topk_idx);
  MOE_NEED(recv);
  MOE_NEED(counts);
  MOE_NEED(row_of);
  MOE_OPT(src_tok);
  if (is_fp8(*cfg)) MOE_NEED(recv_scales);
  if (status && (reinterpret_cast<uintptr_t>(status) & 3u)) return MOE_ERR_MISALIGNED;
  cudaError_t e = launch_dispatch(*cfg, x, topk_idx, recv, recv_scales, counts, row_of, src_tok,
                                  status, stream);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

int moe_expert_ffn(const moe_cfg* cfg, const void* recv, const float* recv_scales,
                   const int32_t* counts, const void* x, const moe_weights* w, void* ebuf,
                   void* shared_out, void* ws, cudaStream_t stream) {
  MOE_CHECK_CFG(cfg);
  const moe_cfg& c = *cfg;
  MOE_NEED(recv);
  MOE_NEED(counts);
  MOE_NEED(ebuf);
  MOE_NEED(ws);
  if (!w) return MOE_ERR_INVALID_ARG;
  MOE_NEED(w->w13);
  MOE_NEED(w->w2);
  const bool fp8 = is_fp8(c);
  if (fp8) {
    MOE_NEED(recv_scales);
    MOE_NEED(w->w13_scales);
    MOE_NEED(w->w2_scales);
  }
  if (c.d_ff_shared) {
    MOE_NEED(x);
    MOE_NEED(w->ws13);
    MOE_NEED(w->ws2);
    MOE_NEED(shared_out);
    if (fp8) {
      MOE_NEED(w->ws13_scales);
      MOE_NEED(w->ws2_scales);
    }
  }
  const WsLayout L = ws_layout(c);
  char* wsp = static_cast<char*>(ws);
  // the GEMMs follow this call's own kernels: programmatic launches
  cudaError_t e = launch_ffn_setup(c, L, counts, x, wsp, stream);
  if (e == cudaSuccess)
    e = launch_ffn_gemm(c, L, 0, recv, recv_scales, x, *w, ebuf, shared_out, wsp, stream, true);
  if (e == cudaSuccess)
    e = launch_ffn_gemm(c, L, 1, recv, recv_scales, x, *w, ebuf, shared_out, wsp, stream, true);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

int moe_combine(const moe_cfg* cfg, const void* ebuf, const int32_t* row_of,
                const float* topk_w, const void* shared_out, void* y, uint32_t* status,
                cudaStream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_NEED(ebuf);
  MOE_NEED(row_of);
  MOE_NEED(topk_w);
  MOE_OPT(shared_out);
  MOE_NEED(y);
  if (status && (reinterpret_cast<uintptr_t>(status) & 3u)) return MOE_ERR_MISALIGNED;
  cudaError_t e = launch_combine(*cfg, ebuf, row_of, topk_w, shared_out, y, status, stream);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

namespace {

// The layer on `stream` with the variants of opts (see moe_layer_ex). Pointers are checked by
// the caller.
int layer_impl(const moe_cfg& c0, const moe_layer_opts& o, const void* x, const float* w_gate,
               const float* bias, const moe_weights* w, int32_t* topk_idx, float* topk_w,
               void* recv, float* recv_scales, int32_t* counts, int32_t* row_of, void* ebuf,
               void* shared_out, void* y, void* ws, cudaStream_t stream,
               const cudaEvent_t* events) {
  // with a placement every stage after the router works on the slots (c), the router on the
  // experts (c0)
  const moe_cfg c = slot_cfg(c0, o.placement);
  const WsLayout L = ws_layout(c);
  char* wsp = static_cast<char*>(ws);
  const bool fp8 = is_fp8(c);
  const bool gather = (o.flags & MOE_OPT_GATHER_X) != 0;
  const bool side = (o.flags & MOE_OPT_SHARED_SIDE_STREAM) != 0 && c.d_ff_shared > 0;
  const bool fused = (o.flags & MOE_OPT_FUSED_FFN) != 0;
  int32_t* src_tok = gather ? reinterpret_cast<int32_t*>(wsp + L.src_tok) : nullptr;
  auto rec = [&](int i) -> cudaError_t {
    return events ? cudaEventRecord(events[i], stream) : cudaSuccess;
  };
  // Without stage events every kernel after the first follows a kernel of this call directly
  // and is launched programmatically (its CTAs become resident while the previous kernel
  // runs; measured on the DSV3 layer: 20 us less per step at T = 64, 39 us at T = 4096). With
  // events, each stage starts after its event as usual, so the events time the stages
  // themselves.
  const bool pdl = events == nullptr;
  const StageRange layer_range("moe_layer");
  cudaError_t e = rec(0);
  bool quantised = false;
  if (e == cudaSuccess && side) {
    // the shared expert's input first (e4m3), then its two GEMMs on the side stream
    const StageRange r("shared_expert_side");
    if (fp8) {
      e = launch_quant_x(c, L, x, wsp, stream, false);
      quantised = true;
    }
    if (e == cudaSuccess) e = cudaEventRecord(o.fork_event, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(o.side_stream, o.fork_event, 0);
    FfnPart sp;
    sp.routed = false;
    sp.ctas = o.side_ctas > 0 ? o.side_ctas : 16;
    sp.weight_experts = c0.E;
    for (int stg = 0; stg < 2 && e == cudaSuccess; ++stg)
      e = launch_ffn_gemm(c, L, stg, recv, recv_scales, x, *w, ebuf, shared_out, wsp,
                          o.side_stream, stg == 1, sp);
    if (e == cudaSuccess) e = cudaEventRecord(o.join_event, o.side_stream);
  }
  if (e == cudaSuccess) {
    const StageRange r("route");
    e = launch_route(c0, x, w_gate, bias, topk_idx, topk_w,
                     reinterpret_cast<float*>(wsp + L.partials),
                     reinterpret_cast<uint32_t*>(wsp + L.status), stream, pdl && !side,
                     c.d_ff_shared && !side ? w->ws13 : nullptr,
                     (size_t)2 * c.d_ff_shared * c.d * act_bytes(c));
  }
  if (e == cudaSuccess) e = rec(1);
  if (e == cudaSuccess) {
    const StageRange r("dispatch");
    e = launch_dispatch(c0, x, topk_idx, gather ? nullptr : recv, recv_scales, counts, row_of,
                        src_tok, reinterpret_cast<uint32_t*>(wsp + L.status), stream, pdl, false,
                        o.placement);
  }
  if (e == cudaSuccess) e = rec(2);
  if (e == cudaSuccess) {
    const StageRange r("ffn_setup");
    e = launch_ffn_setup(c, L, counts, x, wsp, stream, pdl, src_tok, !quantised,
                         o.placement ? o.placement->slot_expert : nullptr);
  }
  if (e == cudaSuccess) e = rec(3);
  FfnPart mp;
  mp.shared = !side;
  mp.src_tok = src_tok;
  mp.group_expert = o.placement ? o.placement->slot_expert : nullptr;
  mp.weight_experts = c0.E;
  if (fused) {
    // both GEMMs and the combine in one launch; the stage events after it all mark its end
    const StageRange r("ffn_fused");
    if (e == cudaSuccess)
      e = launch_ffn_fused(c, L, recv, x, *w, ebuf, shared_out, row_of, topk_w, y, wsp, stream,
                           mp);
    for (int i = 4; i <= 6 && e == cudaSuccess; ++i) e = rec(i);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e);
  }
  if (e == cudaSuccess) {
    const StageRange r("ffn_gate_up");
    e = launch_ffn_gemm(c, L, 0, recv, recv_scales, x, *w, ebuf, shared_out, wsp, stream, pdl,
                        mp);
  }
  if (e == cudaSuccess) e = rec(4);
  if (e == cudaSuccess) {
    const StageRange r("ffn_down");
    e = launch_ffn_gemm(c, L, 1, recv, recv_scales, x, *w, ebuf, shared_out, wsp, stream, pdl,
                        mp);
  }
  if (e == cudaSuccess) e = rec(5);
  if (e == cudaSuccess && side) e = cudaStreamWaitEvent(stream, o.join_event, 0);
  if (e == cudaSuccess) {
    const StageRange r("combine");
    e = launch_combine(c, ebuf, row_of, topk_w, c.d_ff_shared ? shared_out : nullptr, y,
                       reinterpret_cast<uint32_t*>(wsp + L.status), stream, pdl && !side);
  }
  if (e == cudaSuccess) e = rec(6);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

}  // namespace

#define MOE_LAYER_CHECKS(gather)              \
  MOE_CHECK_CFG(cfg);                         \
  const moe_cfg& c = *cfg;                    \
  MOE_NEED(x);                                \
  MOE_NEED(w_gate);                           \
  MOE_NEED(bias);                             \
  MOE_NEED(topk_idx);                         \
  MOE_NEED(topk_w);                           \
  if (!(gather)) MOE_NEED(recv);              \
  MOE_NEED(counts);                           \
  MOE_NEED(row_of);                           \
  MOE_NEED(ebuf);                             \
  MOE_NEED(y);                                \
  MOE_NEED(ws);                               \
  if (!w) return MOE_ERR_INVALID_ARG;         \
  MOE_NEED(w->w13);                           \
  MOE_NEED(w->w2);                            \
  const bool fp8 = is_fp8(c); \
  if (fp8) {                                  \
    if (!(gather)) MOE_NEED(recv_scales);     \
    MOE_NEED(w->w13_scales);                  \
    MOE_NEED(w->w2_scales);                   \
  }                                           \
  if (c.d_ff_shared) {                        \
    MOE_NEED(w->ws13);                        \
    MOE_NEED(w->ws2);                         \
    MOE_NEED(shared_out);                     \
    if (fp8) {                                \
      MOE_NEED(w->ws13_scales);               \
      MOE_NEED(w->ws2_scales);                \
    }                                         \
  }

int moe_layer(const moe_cfg* cfg, const void* x, const float* w_gate, const float* bias,
              const moe_weights* w, int32_t* topk_idx, float* topk_w, void* recv,
              float* recv_scales, int32_t* counts, int32_t* row_of, void* ebuf,
              void* shared_out, void* y, void* ws, cudaStream_t stream,
              const cudaEvent_t* events) {
  MOE_LAYER_CHECKS(false);
  const moe_layer_opts o{};
  return layer_impl(c, o, x, w_gate, bias, w, topk_idx, topk_w, recv, recv_scales, counts,
                    row_of, ebuf, shared_out, y, ws, stream, events);
}

int moe_layer_ex(const moe_cfg* cfg, const moe_layer_opts* opts, const void* x,
                 const float* w_gate, const float* bias, const moe_weights* w, int32_t* topk_idx,
                 float* topk_w, void* recv, float* recv_scales, int32_t* counts, int32_t* row_of,
                 void* ebuf, void* shared_out, void* y, void* ws, cudaStream_t stream,
                 const cudaEvent_t* events) {
  const moe_layer_opts o = opts ? *opts : moe_layer_opts{};
  if (o.flags & ~(MOE_OPT_GATHER_X | MOE_OPT_SHARED_SIDE_STREAM | MOE_OPT_FUSED_FFN))
    return MOE_ERR_INVALID_ARG;
  MOE_LAYER_CHECKS((o.flags & MOE_OPT_GATHER_X) != 0);
  if (o.flags & MOE_OPT_FUSED_FFN) {
    if (c.act_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    // the combine runs inside the launch, so the shared expert cannot be on another stream
    if ((o.flags & MOE_OPT_SHARED_SIDE_STREAM) && c.d_ff_shared) return MOE_ERR_INVALID_ARG;
  }
  if (o.placement) {
    const moe_placement& p = *o.placement;
    if (p.slots_per_rank < 1 || (long long)p.slots_per_rank * c.R < c.E || p.max_copies < 1)
      return MOE_ERR_INVALID_ARG;
    if ((long long)p.slots_per_rank * c.R > 1024) return MOE_ERR_UNSUPPORTED;
    MOE_NEED(p.slot_expert);
    MOE_NEED(p.n_copies);
    MOE_NEED(p.copy_slot);
    const int rc = validate(slot_cfg(c, &p));
    if (rc != MOE_OK) return rc;
  }
  if ((o.flags & MOE_OPT_SHARED_SIDE_STREAM) && c.d_ff_shared) {
    if (!o.side_stream || !o.fork_event || !o.join_event || o.side_stream == stream)
      return MOE_ERR_INVALID_ARG;
    if (o.side_ctas < 0 || o.side_ctas > 4096) return MOE_ERR_INVALID_ARG;
  }
  return layer_impl(c, o, x, w_gate, bias, w, topk_idx, topk_w, recv, recv_scales, counts,
                    row_of, ebuf, shared_out, y, ws, stream, events);
}

int moe_dispatch_index(const moe_cfg* cfg, const int32_t* topk_idx, int32_t* counts,
                       int32_t* row_of, int32_t* src_tok, uint32_t* status,
                       cudaStream_t stream) {
  MOE_CHECK_CFG(cfg);
  MOE_NEED(topk_idx);
  MOE_NEED(counts);
  MOE_NEED(row_of);
  MOE_NEED(src_tok);
  if (status && (reinterpret_cast<uintptr_t>(status) & 3u)) return MOE_ERR_MISALIGNED;
  cudaError_t e = launch_dispatch(*cfg, nullptr, topk_idx, nullptr, nullptr, counts, row_of,
                                  src_tok, status, stream);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

int moe_expert_ffn_gather(const moe_cfg* cfg, const void* x, const int32_t* counts,
                          const int32_t* src_tok, const moe_weights* w, void* ebuf,
                          void* shared_out, void* ws, cudaStream_t stream) {
  MOE_CHECK_CFG(cfg);
  const moe_cfg& c = *cfg;
  MOE_NEED(x);
  MOE_NEED(counts);
  MOE_NEED(src_tok);
  MOE_NEED(ebuf);
  MOE_NEED(ws);
  if (!w) return MOE_ERR_INVALID_ARG;
  MOE_NEED(w->w13);
  MOE_NEED(w->w2);
  const bool fp8 = is_fp8(c);
  if (fp8) {
    MOE_NEED(w->w13_scales);
    MOE_NEED(w->w2_scales);
  }
  if (c.d_ff_shared) {
    MOE_NEED(w->ws13);
    MOE_NEED(w->ws2);
    MOE_NEED(shared_out);
    if (fp8) {
      MOE_NEED(w->ws13_scales);
      MOE_NEED(w->ws2_scales);
    }
  }
  const WsLayout L = ws_layout(c);
  char* wsp = static_cast<char*>(ws);
  FfnPart part;
  part.src_tok = src_tok;
  cudaError_t e = launch_ffn_setup(c, L, counts, x, wsp, stream, false, src_tok);
  if (e == cudaSuccess)
    e = launch_ffn_gemm(c, L, 0, nullptr, nullptr, x, *w, ebuf, shared_out, wsp, stream, true,
                        part);
  if (e == cudaSuccess)
    e = launch_ffn_gemm(c, L, 1, nullptr, nullptr, x, *w, ebuf, shared_out, wsp, stream, true,
                        part);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

int moe_clear_status(void* ws, cudaStream_t stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(uint32_t), stream);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

int moe_read_status(const void* ws, uint32_t* status, cudaStream_t stream) {
  if (!ws || !status) return MOE_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemcpy(status, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? MOE_OK : cuda_fail(e);
}

}  // extern "C"
