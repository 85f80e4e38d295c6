// Internal declarations shared by the host API (moe_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Router: d is cut into this many equal chunks, each summed as one sequential FMA chain.
constexpr int kRouteChunks = 16;

// One entry of the expert-GEMM tile schedule: rows [n0, n0+nlen) of group g, which has ntiles
// token tiles in all (its entries are consecutive, n0 = j * bn for the j-th). With placed
// experts a group's tiles cover the compact rows of all the expert's copies, and g is its first
// copy.
struct Tile {
  int32_t group;
  int32_t n0;
  int32_t nlen;
  int32_t ntiles;
};

// Byte offsets of the pieces of the workspace (all 256-byte aligned).
struct WsLayout {
  size_t status;      // uint32 status word
  size_t partials;    // router partial dot products: fp32 [16][T][E]
  size_t grp_n;       // int32 [E]: rows received by each routed expert
  size_t grp_off;     // int32 [E]: first compact row of each routed expert
  size_t n_tiles;     // int32 [2]: routed tiles in the schedule; of those, tiles of groups with
                      // two or more (listed first)
  size_t tiles;       // Tile [max_tiles]
  size_t row_list;    // int32 [T*k]: receive row of each compact row
  size_t h;           // SwiGLU intermediate of routed rows: [T*k][d_ff] (bf16 or e4m3)
  size_t h_scales;    // e4m3: fp32, block-major [d_ff/128][T*k]
  size_t hs;          // shared expert intermediate: [T][d_ff_shared]
  size_t hs_scales;   // e4m3: fp32, block-major [d_ff_shared/128][T]
  size_t xq;          // e4m3: x quantised once per token [T][d] (shared-expert input; the
                      // routed rows' source in gather mode)
  size_t xq_scales;   // e4m3: fp32, block-major [d/128][T]
  size_t run_start;   // int32 [R][E]: receive row of the first row source s sent expert e
  size_t run_pre;     // int32 [R][E]: rows of expert e from sources before s
  size_t src_tok;     // int32 [R*R*cap]: token of each filled receive row (gather mode)
  size_t tok_list;    // int32 [T*k]: token of each compact row (gather mode)
  size_t grp_order;   // int32 [E]: group at each schedule position (placed experts)
  size_t fused_done;  // int32 [fused_done_n]: dependency counters of the fused expert launch
  // power-of-two e4m3 only: the UE8M0 scale bytes of each GEMM input row, row-major with
  // kSfRowBytes bytes a row (byte b: the row's 128-column block b), for the block-scaled MMA
  size_t sf_gu;       // [T*k]: routed gate/up input rows (compact order)
  size_t sf_x;        // [T]: the shared expert's gate/up input rows (x quantised)
  size_t sf_h;        // [T*k]: routed down input rows (h)
  size_t sf_hs;       // [T]: the shared expert's down input rows (hs)
  // the same schedule in tiles of 2 * bn rows (the bf16 down GEMM when experts average a full
  // bn-row tile or more)
  size_t n_tiles2;    // int32 [2], as n_tiles
  size_t tiles2;      // Tile [max_tiles2]
  int max_tiles2;
  int shared_tiles;   // token tiles of the shared expert (0: none)
  int fused_done_n;   // max_tiles + shared_tiles + 2
  size_t total;
  int bn;             // token-tile width of the expert GEMMs
  int max_tiles;      // bound on routed tiles: E + T*k/bn
};

int validate(const moe_cfg& c);
// Records e as this host thread's last CUDA error (moe_last_cuda_error) and returns
// MOE_ERR_CUDA: every entry point reports a failed CUDA call through it.
int cuda_fail(cudaError_t e);
WsLayout ws_layout(const moe_cfg& c);
inline int cap_of(const moe_cfg& c) {
  int Er = c.E / c.R, Ts = c.T / c.R;
  return Ts * (c.k < Er ? c.k : Er);
}
inline bool is_fp8(const moe_cfg& c) { return c.act_dtype != MOE_BF16; }
// Scale bytes per row of the power-of-two recipe's byte tables: one per 128-column block of
// K <= 8192.
constexpr int kSfRowBytes = 64;
// e4m3 with power-of-two block scales (the block-scaled MMA's recipe)
inline bool pow2_scales(const moe_cfg& c) { return c.act_dtype == MOE_FP8_E4M3_POW2; }
inline size_t act_bytes(const moe_cfg& c) { return is_fp8(c) ? 1 : 2; }

// The configuration seen by the stages after the router when the experts are placed on slots:
// E becomes the slot count R * slots_per_rank (one group of the grouped GEMMs per slot). The
// group fields are not used after the router; they are set to one group so the copy validates.
inline moe_cfg slot_cfg(const moe_cfg& c, const moe_placement* p) {
  if (!p) return c;
  moe_cfg s = c;
  s.E = c.R * p->slots_per_rank;
  s.n_group = 1;
  s.topk_group = 1;
  return s;
}

// launch_route's selection kernel also starts pulling [warm, warm + warm_bytes) into L2 (the
// shared expert's gate/up weights, which the gate/up GEMM reads first) while the rest of the
// routing runs with the memory system mostly idle.
// Kernel launchers. Each returns the launch error (cudaSuccess when enqueued). With pdl the
// launcher's kernels are launched programmatically: each may become resident while the
// previous kernel in the stream is still running, and waits for it before touching memory
// (launch_route's first kernel, which follows the caller's own work, is always launched as
// usual).
cudaError_t launch_route(const moe_cfg& c, const void* x, const float* w_gate, const float* bias,
                         int32_t* topk_idx, float* topk_w, float* partials, uint32_t* status,
                         cudaStream_t st, bool pdl = false, const void* warm = nullptr,
                         size_t warm_bytes = 0);

// With recv == nullptr only the index pass runs (counts, row_of, src_tok): the gather mode,
// whose expert GEMMs read token rows straight from x. clear_src_tok: fill src_tok with -1
// first (the stage call's contract for rows that receive nothing).
// status: nullable device word that index errors are OR-ed into (MOE_DEV_BOUNDS).
// placement: NULL, or the experts' slots; counts and the receive rows are then over the slots.
cudaError_t launch_dispatch(const moe_cfg& c, const void* x, const int32_t* topk_idx, void* recv,
                            float* recv_scales, int32_t* counts, int32_t* row_of,
                            int32_t* src_tok, uint32_t* status, cudaStream_t st,
                            bool pdl = false, bool clear_src_tok = true,
                            const moe_placement* placement = nullptr);

// Entries of row_of outside [0, recv_rows) are skipped and reported in status (nullable).
cudaError_t launch_combine(const moe_cfg& c, const void* ebuf, const int32_t* row_of,
                           const float* topk_w, const void* shared_out, void* y,
                           uint32_t* status, cudaStream_t st, bool pdl = false);

// Which parts of the expert stage a GEMM launch covers, and where its routed token rows come
// from.
struct FfnPart {
  bool routed = true;        // the routed experts' units
  bool shared = true;        // the shared expert's units (when it exists)
  const int32_t* src_tok = nullptr;  // gather mode: token of each receive row; the routed rows
                                     // are read from x (e4m3: x quantised per token) instead of
                                     // from the receive buffer
  int ctas = 0;              // grid size (0: one CTA per SM)
  const int32_t* group_expert = nullptr;  // the expert whose weights each group uses (slots of
                                          // a placement); nullptr: group g is expert g
  int weight_experts = 0;    // experts in the weight tensors (0: the cfg's E)
};

// Expert FFN set-up: tile schedule from counts (+ e4m3 quantisation of x for the shared expert
// and, in gather mode, the routed rows). src_tok != nullptr: gather mode (the schedule also
// lists each compact row's token).
// quantise == false: the e4m3 quantisation of x was enqueued already (launch_quant_x).
// group_expert: the slot->expert map of a placement (the schedule orders the groups by expert).
cudaError_t launch_ffn_setup(const moe_cfg& c, const WsLayout& L, const int32_t* counts,
                             const void* x, char* ws, cudaStream_t st, bool pdl = false,
                             const int32_t* src_tok = nullptr, bool quantise = true,
                             const int32_t* group_expert = nullptr);

// e4m3: x quantised once per token into the workspace (xq, xq_scales).
cudaError_t launch_quant_x(const moe_cfg& c, const WsLayout& L, const void* x, char* ws,
                           cudaStream_t st, bool pdl = false);

// The two grouped GEMMs. stage: 0 = gate/up with the SwiGLU epilogue, 1 = down projection.
cudaError_t launch_ffn_gemm(const moe_cfg& c, const WsLayout& L, int stage, const void* recv,
                            const float* recv_scales, const void* x, const moe_weights& w,
                            void* ebuf, void* shared_out, char* ws, cudaStream_t st,
                            bool pdl = false, const FfnPart& part = FfnPart());

// bf16: both GEMMs and the combine in one persistent (cooperative) launch with device-side
// dependency counters (csrc/moe_fused.cu). The combine's arguments are those of
// launch_combine; part as for launch_ffn_gemm (the shared expert must be part of it).
cudaError_t launch_ffn_fused(const moe_cfg& c, const WsLayout& L, const void* recv, const void* x,
                             const moe_weights& w, void* ebuf, void* shared_out,
                             const int32_t* row_of, const float* topk_w, void* y, char* ws,
                             cudaStream_t st, const FfnPart& part);

// e4m3 grouped GEMMs (non-swapped, per-128-K-block scale promotion), same stages.
cudaError_t launch_ffn_gemm_e4m3(const moe_cfg& c, const WsLayout& L, int stage, const void* recv,
                                 const float* recv_scales, const moe_weights& w, void* ebuf,
                                 void* shared_out, char* ws, cudaStream_t st, bool pdl,
                                 const FfnPart& part);

// e4m3 grouped GEMMs with power-of-two block scales applied by the tensor core (block-scaled
// MMA, csrc/moe_ffn_mx8.cu), same stages.
cudaError_t launch_ffn_gemm_mx8(const moe_cfg& c, const WsLayout& L, int stage, const void* recv,
                                const float* recv_scales, const moe_weights& w, void* ebuf,
                                void* shared_out, char* ws, cudaStream_t st, bool pdl,
                                const FfnPart& part);

// 1x128 e4m3 quantisation of T rows of width d (the dispatch's rule), row t -> row t; pow2:
// power-of-two scales.
cudaError_t launch_quant_rows_e4m3(const void* x, int T, int d, void* out, float* scales,
                                   cudaStream_t st, bool pdl = false, bool pow2 = false);

// 2-D row-major tensor map [rows][cols] with a box of box_rows x 128 bytes, 128-byte swizzle.
bool make_tensor_map_2d(CUtensorMap* m, const void* base, int elem_bytes, uint64_t cols,
                        uint64_t rows, uint32_t box_rows);

// Streaming multiprocessors of the current device.
int sm_count();

// Raises kern's dynamic shared-memory limit on the current device to at least `bytes` (no-op up
// to 48 KB). The runtime is called only the first time a kernel needs a larger size on a
// device, so steady-state calls enqueue launches and nothing else.
cudaError_t ensure_smem_limit(const void* kern, size_t bytes);

}  // namespace moe
