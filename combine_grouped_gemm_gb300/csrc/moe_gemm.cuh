// Definitions shared by the bf16 grouped-GEMM kernels (moe_ffn.cu: one launch per stage;
// moe_fused.cu: both stages and the combine in one persistent launch): the launch arguments,
// the unit list (shared-expert tiles first, then every (token tile, weight tile) of every
// routed group), the warp roles and the shared-memory stage shapes. The GEMMs themselves are
// described in moe_ffn.cu.
#pragma once

#include "moe_device.cuh"

namespace moe {

// ---------------------------------------------------------------------------------------
// Grouped GEMM
// ---------------------------------------------------------------------------------------
struct GemmArgs {
  const Tile* tiles;
  const int32_t* n_tiles;  // [0]: tiles in the list; [1]: of those, the first ones, whose groups
                           // have two or more token tiles
  const int32_t* grp_off;
  const int32_t* row_list;
  int tk;                 // compact rows (T*k)
  long long recv_rows;    // receive rows (bound of gathered / scattered row indices)
  int T;                  // shared-expert rows
  int mt_routed;          // 128-row weight tiles per routed expert
  int mt_shared;          // 128-row weight tiles of the shared expert (0: none)
  int n_shared_tiles;     // token tiles of the shared expert
  int k_steps;            // K / 64
  int a_rows_routed;      // weight rows per routed expert
  int a_up_routed;        // offset of the up rows (gate/up stage)
  int a_up_shared;
  void* out_routed;       // gate/up: h [tk][F] (compact rows); down: ebuf [recv_rows][d]
  void* out_shared;       // gate/up: hs [T][Fs]; down: shared_out [T][d]
  int ld_routed;          // output row length (elements)
  int ld_shared;
  int box_routed;         // rows per box of the contiguous token-row maps (routed / shared)
  int box_shared;
  const uint8_t* gather_base;  // gate/up: receive buffer (routed token rows are gathered)
  long long gather_ld;         // bytes per receive row
  uint32_t* status;
  const int32_t* group_expert; // expert whose weights group g uses (nullptr: expert g)
  int n_experts;               // experts in the weight tensors
};

// The expert whose weight rows a routed group reads: itself, or the expert its slot holds
// (redundant experts). An entry outside [0, n_experts) is reported and replaced by expert 0, so
// no weight read leaves the tensors.
__device__ __forceinline__ int weight_expert(const int32_t* group_expert, int g, int n_experts,
                                             uint32_t* status) {
  if (!group_expert) return g;
  const int e = group_expert[g];
  if (e >= 0 && e < n_experts) return e;
  raise_status(status, MOE_DEV_BOUNDS);
  return 0;
}

struct Unit {
  int g;       // routed expert, or -1 for the shared expert
  int n0, nlen, m;
  int nt;      // token tiles of the group (units that read this unit's weight tiles)
  int ti;      // the unit's token tile: its index in the tile list, or the shared tile number
};

// Unit u -> (group, token tile, weight tile). Shared-expert units come first, token-tile-major.
// A routed expert with nt token tiles owns units [mt*b, mt*(b+nt)), b = its first tile, taken
// either token-tile-major (unit mt*b + j*mt + m: a token tile's rows serve consecutive units)
// or weight-tile-major (unit mt*b + m*nt + j: the nt units that read weight tile m run on
// adjacent CTAs at about the same time). The separate GEMM launches take both stages
// weight-tile-major: on the skew workload this cut the down GEMM's DRAM reads from 10.56 to
// 8.50 GB, and, once the multi-tile groups' weight tiles were kept evict-last and their units
// interleaved with the one-tile groups', the gate/up GEMM's time by 3 % (2932 -> 2837 us). The
// fused launch takes gate/up token-tile-major. n_tiles: entries in the tile list.
template <int BN, bool kWeightMajor>
__device__ __forceinline__ Unit decode_unit(const GemmArgs& a, int u, int n_tiles) {
  Unit r;
  const int us = a.n_shared_tiles * a.mt_shared;
  if (u < us) {
    const int tt = u / a.mt_shared;
    r.g = -1;
    r.m = u - tt * a.mt_shared;
    r.n0 = tt * BN;
    r.nlen = min(BN, a.T - r.n0);
    r.nt = a.n_shared_tiles;
    r.ti = tt;
  } else {
    const int v = u - us;
    const int tt0 = v / a.mt_routed;   // a tile of the unit's expert (the ranges coincide)
    const Tile t0 = a.tiles[tt0];
    Tile t = t0;
    int ti = tt0;
    if (!kWeightMajor) {
      r.m = v - tt0 * a.mt_routed;
    } else {
      const int base = tt0 - t0.n0 / BN;
      // (a list cut short at its bound, already reported, keeps every index inside it)
      const int nt = max(1, min(t0.ntiles, n_tiles - base));
      const int local = v - base * a.mt_routed;
      r.m = local / nt;
      const int j = local - r.m * nt;
      ti = base + j;
      if (ti != tt0) t = a.tiles[ti];
    }
    r.nt = t0.ntiles;
    r.g = t.group;
    r.n0 = t.n0;
    r.nlen = t.nlen;
    r.ti = ti;
  }
  return r;
}

// Schedule slot s -> unit. Units [0, hot) (the shared expert's and those of groups with two or
// more token tiles: each weight tile is read once per token tile, from L2 after the first, so
// they keep the tensor pipe busy) and units [hot, units) (one-tile groups: every weight tile is
// read once, from HBM) are merged evenly, each in its own order, so that at any time about the
// same share of the CTAs streams weights from HBM. Taken in list order, the two kinds ran one
// after the other: on the skewed prefill each GEMM took about its HBM time plus its tensor time.
__device__ __forceinline__ int interleave_unit(int s, int units, int hot) {
  const int cold = units - hot;
  if (hot <= 0 || cold <= 0) return s;
  const long long c0 = static_cast<long long>(s) * cold / units;   // cold slots before s
  const long long c1 = static_cast<long long>(s + 1) * cold / units;
  return c1 > c0 ? hot + static_cast<int>(c0) : s - static_cast<int>(c0);
}

// Units of the tensor-bound part of a launch's list (see interleave_unit): the shared expert's
// units, then those of the routed tiles listed first. 0 (the list order) unless the routed
// groups are of both kinds: with one-tile routed groups only, spreading the shared expert's
// units over the launch made the gate/up GEMM 2-3 % slower at 512 and 1024 tokens.
__device__ __forceinline__ int hot_units(const GemmArgs& a, int n_tiles) {
  const int hot_tiles = min(max(a.n_tiles[1], 0), n_tiles);
  if (hot_tiles == 0 || hot_tiles == n_tiles) return 0;
  return a.n_shared_tiles * a.mt_shared + hot_tiles * a.mt_routed;
}

// L2 policy of a unit's weight tiles. A group with one token tile reads each weight tile once:
// evict-first, so the stream does not push out what is reused. A group with several token
// tiles (a hot expert, or the shared expert at prefill) reads each weight tile once per token
// tile, in units that run close together: evict-last keeps the tile for the next one. On the
// skewed prefill (hottest expert about 10x the mean load) this took the gate/up GEMM from 3358
// to 2858 us and the down GEMM from 1822 to 1761 us; the decode layer, one tile per expert,
// is unchanged.
__device__ __forceinline__ uint64_t weight_policy(const Unit& t, uint64_t once, uint64_t reused) {
  return t.nt > 1 ? reused : once;
}

// Gate/up only: warps that gather the routed token rows with 16-byte cp.async copies (tiles of
// more than kSmallTile rows; smaller ones are four-row TMA gathers).
constexpr int kGatherWarps = 2;
constexpr int kSmallTile = 32;
constexpr int kGatherThreads = kGatherWarps * 32;
template <int STAGE>
struct GemmThreads {
  static constexpr int kGather = STAGE == 0 ? kGatherThreads : 0;
  static constexpr int kAll = 192 + kGather;
};

template <int STAGE, int BN, int STAGES>
struct GemmShape {
  static constexpr int NA = STAGE == 0 ? 2 : 1;    // weight tiles per stage (gate, up)
  static constexpr int A_BYTES = 128 * 128;        // 128 rows x 64 bf16
  static constexpr int B_BYTES = BN * 128;         // BN rows x 64 bf16
  static constexpr int STAGE_BYTES = NA * A_BYTES + B_BYTES;
  static constexpr int ACC_COLS = NA * BN;         // fp32 accumulator columns per buffer
  static constexpr int TMEM_COLS = 2 * ACC_COLS <= 32 ? 32 : 2 * ACC_COLS;
  static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 + 256;
  static_assert(STAGE_BYTES % 1024 == 0, "stages stay 1024-byte aligned");
  static_assert((TMEM_COLS & (TMEM_COLS - 1)) == 0 && TMEM_COLS <= 512, "tensor memory");
};


// Host side: the arguments and TMA tensor maps of one bf16 GEMM stage (0 = gate/up with the
// SwiGLU epilogue, 1 = down projection) for configuration c, as launch_ffn_gemm builds them.
// maps: A (routed weights), A shared, B (routed token rows), B shared. wide: the down stage on
// the schedule's 2 * bn-row tiles (launch_ffn_gemm's 256-row kernel).
cudaError_t prepare_bf16_gemm(const moe_cfg& c, const WsLayout& L, int stage, const void* recv,
                              const void* x, const moe_weights& w, void* ebuf, void* shared_out,
                              char* ws, const FfnPart& part, GemmArgs* args, CUtensorMap maps[4],
                              bool wide = false);

}  // namespace moe
