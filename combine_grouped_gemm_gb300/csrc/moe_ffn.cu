// Expert FFN: device-side tile schedule from the dispatch counts, then two grouped GEMMs on
// the 5th-generation tensor cores (tcgen05, accumulators in tensor memory, operands staged in
// shared memory by TMA):
//   gate/up : for the rows of each expert, g = X Wg^T and u = X Wu^T into two tensor-memory
//             accumulators; epilogue h = bf16(silu(g) * u)
//   down    : o = h Wd^T; epilogue bf16 rows written back at the receive-row index.
// The shared expert is one more group whose rows are the T tokens of x.
//
// Method: "7.13 Serving Mixture-of-Experts" (llm-stack-book), Expert Parallelism Mechanics,
// expert compute (one grouped GEMM over the rows each expert received, ragged groups padded
// or masked); "One-Sided Expert-Parallel All-to-All for Mixture-of-Experts Inference over
// NVLink", abstract (the grouped GEMMs read the rank-major receive buffers in place rather
// than a per-expert copy); "Mixture-of-experts serving" (learn-kernels), paragraph 1 (one
// always-active shared expert).
//
// GEMM shape: the weights are the M operand (128 rows of W per tile: "swap AB"), the
// expert's rows are the N operand (a token tile of up to BN rows, N padded to a multiple of
// 16), K is the model width (gate/up) or d_ff (down). An expert's rows lie in up to R runs of
// the receive buffer (one per source rank); the producer gathers them row by row with 1-row
// TMA boxes, which land in the same 128-byte-swizzled layout an 8-row box would produce.
// Columns of a tile past its real rows hold stale shared memory; they only feed accumulator
// columns the epilogue never stores.
//
// Roles in a CTA (192 threads, one CTA per SM, persistent over the unit list):
//   warp 0      TMA producer (lane 0: weight tiles; all lanes: gathered token rows)
//   warp 1      tensor-memory allocation; lane 0 issues tcgen05.mma and commits
//   warps 2..5  epilogue: tcgen05.ld of the accumulator rows, SwiGLU, bf16 stores
// Shared-memory stages hand over through full/empty mbarriers; the two tensor-memory
// accumulator buffers hand over through tmem_full/tmem_empty mbarriers, so the epilogue of a
// unit overlaps the main loop of the next. Every wait is bounded (see moe_device.cuh).
#include <mutex>

#include "moe_gemm.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------------------------------
// Tile schedule (one CTA)
// ---------------------------------------------------------------------------------------
constexpr int kPlanThreads = 1024;             // upper bound; launched with E rounded up to 32
// counts table staged in shared memory up to this: the 48 KB a kernel gets without an opt-in,
// less the kernel's static shared memory (warp sums and rank bases, 388 bytes; two tables by
// schedule position, 8 KB)
constexpr size_t kPlanStageBytes = 39 * 1024;
constexpr int kPlanFusedRows = 1024;            // fill the row list in the plan CTA up to this T*k

// Block-wide exclusive scan of one int per thread (blockDim.x a multiple of 32, <= 1024).
__device__ int block_exclusive_scan(int v, int* total, int* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  __syncthreads();
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < static_cast<int>(blockDim.x >> 5) ? warp_sums[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    warp_sums[lane] = wi - w;  // exclusive prefix of warp totals
    if (lane == 31) warp_sums[32] = wi;
  }
  __syncthreads();
  const int ex = warp_sums[warp] + incl - v;
  *total = warp_sums[32];
  __syncthreads();
  return ex;
}

// row_list[c] for every compact row c: its expert by binary search on the compact offsets,
// its source run by a scan of the run prefixes, then the run's receive row plus the position.
// In gather mode (src_tok != nullptr) tok_list[c] also receives the compact row's token.
// grp_order (nullable): the group at each position of the schedule order (compact offsets
// ascend along it); nullptr: the groups in index order.
__device__ __forceinline__ void fill_rows(const int32_t* grp_n, const int32_t* grp_off,
                                          const int32_t* run_start, const int32_t* run_pre,
                                          int32_t* row_list, uint32_t* status, int E, int R,
                                          int tk, int first, int stride,
                                          const int32_t* src_tok, int32_t* tok_list,
                                          long long recv_rows, int T,
                                          const int32_t* grp_order) {
  auto at = [&](int i) -> int {
    const int g = grp_order ? grp_order[i] : i;
    return g >= 0 && g < E ? g : 0;
  };
  for (int c = first; c < tk; c += stride) {
    int lo = 0, hi = E - 1;  // last position whose compact offset is <= c
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (grp_off[at(mid)] <= c) lo = mid;
      else hi = mid - 1;
    }
    int i = lo;
    while (i > 0 && grp_n[at(i)] == 0) --i;  // an empty group shares its offset with the next
    while (i < E - 1 && c >= grp_off[at(i)] + grp_n[at(i)]) ++i;
    const int e = at(i);
    const int p = c - grp_off[e];
    if (p < 0 || p >= grp_n[e]) {
      raise_status(status, MOE_DEV_BOUNDS);
      row_list[c] = -1;
      if (tok_list) tok_list[c] = -1;
      continue;
    }
    int s = 0;
    while (s + 1 < R && run_pre[(s + 1) * E + e] <= p) ++s;
    const int row = run_start[s * E + e] + (p - run_pre[s * E + e]);
    row_list[c] = row;
    if (tok_list) {
      int t = (row >= 0 && row < recv_rows) ? src_tok[row] : -1;
      if (t < 0 || t >= T) {
        raise_status(status, MOE_DEV_BOUNDS);
        t = -1;
      }
      tok_list[c] = t;
    }
  }
}

// From counts[R][E]: rows per expert and their compact offsets, the list of token tiles, and
// for every (source, expert) run the receive row of its first row and the number of the
// expert's rows from earlier sources (compact rows are expert-major, then source, then
// position). The row list itself is filled here for up to kPlanFusedRows rows, else by
// ffn_rows_kernel.
__global__ void __launch_bounds__(kPlanThreads) ffn_plan_kernel(
    const int32_t* __restrict__ counts, int32_t* __restrict__ grp_n, int32_t* __restrict__ grp_off,
    int32_t* __restrict__ n_tiles, Tile* __restrict__ tiles, int32_t* __restrict__ run_start,
    int32_t* __restrict__ run_pre, int32_t* __restrict__ row_list, uint32_t* status, int E, int R,
    int cap, int bn, int max_tiles, int tk, const int32_t* __restrict__ src_tok,
    int32_t* __restrict__ tok_list, int T, const int32_t* __restrict__ group_expert,
    int32_t* __restrict__ grp_order, int32_t* __restrict__ n_tiles2, Tile* __restrict__ tiles2,
    int max_tiles2) {
  __shared__ int warp_sums[33];
  __shared__ int rank_base[64];
  __shared__ int ord_g[kPlanThreads];   // group at each schedule position (then its expert)
  __shared__ int ord_n[kPlanThreads];   // its rows
  extern __shared__ int32_t cnt_s[];   // counts staged once: [R][E] when it fits, else unused
  pdl_wait();
  pdl_trigger();
  const int e = threadIdx.x;
  const bool act = e < E;
  const int Er = E / R;
  const bool staged = (size_t)R * E * sizeof(int32_t) <= kPlanStageBytes;
  if (staged)
    for (int i = threadIdx.x; i < R * E; i += blockDim.x) cnt_s[i] = max(0, counts[i]);
  __syncthreads();
  auto cnt = [&](int s_) -> int {
    return staged ? cnt_s[s_ * E + e] : max(0, counts[(size_t)s_ * E + e]);
  };

  int n = 0;
  if (act)
    for (int s = 0; s < R; ++s) n += cnt(s);
  // Schedule order of the groups (compact rows): by index, or, when the groups are slots
  // holding copies of experts, by (expert, slot), so the compact rows of an expert's copies are
  // contiguous. Thread i then handles the group at position i.
  int g_i = e, n_i = n;
  if (group_expert) {
    if (act) {
      const int eg = group_expert[e];
      int pos = 0;
      for (int h = 0; h < E; ++h) {
        const int eh = group_expert[h];
        pos += (eh < eg || (eh == eg && h < e)) ? 1 : 0;
      }
      ord_g[pos] = e;
      ord_n[pos] = n;
      grp_order[pos] = e;
    }
    __syncthreads();
    g_i = act ? ord_g[threadIdx.x] : 0;
    n_i = act ? ord_n[threadIdx.x] : 0;
  }
  int total;
  const int off = block_exclusive_scan(act ? n_i : 0, &total, warp_sums);
  if (threadIdx.x == 0 && total != tk) raise_status(status, MOE_DEV_BOUNDS);
  // GEMM tiles: over each group's rows, or, for the copies of a placed expert, over all of the
  // expert's rows at once (contiguous in the order above), named by its first copy. The copies'
  // rows then go through the expert's weights in the same units, as without a placement: on
  // one GPU the copies share one set of weights, and reading it once per copy would only add
  // weight traffic. The receive layout and the counts stay per slot.
  int tile_rows = act ? n_i : 0;   // rows this position's tiles cover
  if (group_expert) {
    __syncthreads();   // (ord_g was read above)
    if (act) ord_g[threadIdx.x] = group_expert[g_i];
    __syncthreads();
    if (act) {
      const int eg = ord_g[threadIdx.x];
      const bool head = threadIdx.x == 0 || ord_g[threadIdx.x - 1] != eg;
      tile_rows = 0;
      if (head)
        for (int q = threadIdx.x; q < E && ord_g[q] == eg; ++q) tile_rows += ord_n[q];
    }
  }
  // The tile list holds the groups with two or more token tiles first (each of their weight
  // tiles is read once per token tile, from L2 after the first: tensor-bound units), then the
  // one-tile groups (every weight tile read once: HBM-bound units), each part in schedule
  // order; n_tiles[1] counts the first part. The GEMMs interleave the two (interleave_unit).
  const int nt = (tile_rows + bn - 1) / bn;
  int tiles_hot, tiles_cold;
  const int toff_h = block_exclusive_scan(nt >= 2 ? nt : 0, &tiles_hot, warp_sums);
  const int toff_c = block_exclusive_scan(nt >= 2 ? 0 : nt, &tiles_cold, warp_sums);
  const int toff = nt >= 2 ? toff_h : tiles_hot + toff_c;
  const int tiles_total = tiles_hot + tiles_cold;
  if (act) {
    grp_n[g_i] = n_i;
    grp_off[g_i] = off;
    for (int j = 0; j < nt; ++j) {
      const int ti = toff + j;
      if (ti < max_tiles) tiles[ti] = Tile{g_i, j * bn, min(bn, tile_rows - j * bn), nt};
    }
  }
  if (threadIdx.x == 0) {
    if (tiles_total > max_tiles) raise_status(status, MOE_DEV_BOUNDS);
    n_tiles[0] = min(tiles_total, max_tiles);
    n_tiles[1] = min(tiles_hot, max_tiles);
  }
  // the same rows in tiles of 2 * bn (max_tiles2 == 0: not needed by this layer's GEMMs)
  if (max_tiles2 > 0) {
    const int nt2 = (tile_rows + 2 * bn - 1) / (2 * bn);
    int hot2, cold2;
    const int toff2_h = block_exclusive_scan(nt2 >= 2 ? nt2 : 0, &hot2, warp_sums);
    const int toff2_c = block_exclusive_scan(nt2 >= 2 ? 0 : nt2, &cold2, warp_sums);
    const int toff2 = nt2 >= 2 ? toff2_h : hot2 + toff2_c;
    const int tiles_total2 = hot2 + cold2;
    if (act)
      for (int j = 0; j < nt2; ++j) {
        const int ti = toff2 + j;
        if (ti < max_tiles2)
          tiles2[ti] = Tile{g_i, j * 2 * bn, min(2 * bn, tile_rows - j * 2 * bn), nt2};
      }
    if (threadIdx.x == 0) {
      if (tiles_total2 > max_tiles2) raise_status(status, MOE_DEV_BOUNDS);
      n_tiles2[0] = min(tiles_total2, max_tiles2);
      n_tiles2[1] = min(hot2, max_tiles2);
    }
  }

  // per (source, expert) run: first receive row, rows from earlier sources
  int pre = 0;
  if (32 % Er == 0) {
    // each destination rank's experts lie in one warp: a segmented warp scan per source
    const int seg_lane = (threadIdx.x & 31) % Er;
    for (int s = 0; s < R; ++s) {
      const int c = act ? cnt(s) : 0;
      int incl = c;
      for (int o = 1; o < Er; o <<= 1) {
        const int nb = __shfl_up_sync(0xffffffffu, incl, o);
        if (seg_lane >= o) incl += nb;
      }
      if (act) {
        const int r = e / Er;
        const int in_seg = incl - c;
        if (in_seg + c > cap) raise_status(status, MOE_DEV_BOUNDS);
        run_start[s * E + e] = (r * R + s) * cap + in_seg;
        run_pre[s * E + e] = pre;
        pre += c;
      }
    }
  } else {
    for (int s = 0; s < R; ++s) {
      const int c = act ? cnt(s) : 0;
      int dummy;
      const int ex = block_exclusive_scan(c, &dummy, warp_sums);
      if (act && e % Er == 0) rank_base[e / Er] = ex;
      __syncthreads();
      if (act) {
        const int r = e / Er;
        const int in_seg = ex - rank_base[r];
        if (in_seg + c > cap) raise_status(status, MOE_DEV_BOUNDS);
        run_start[s * E + e] = (r * R + s) * cap + in_seg;
        run_pre[s * E + e] = pre;
        pre += c;
      }
      __syncthreads();
    }
  }
  // few rows: fill the row list here (the tables above are this CTA's own writes)
  if (tk <= kPlanFusedRows) {
    __syncthreads();
    fill_rows(grp_n, grp_off, run_start, run_pre, row_list, status, E, R, tk, threadIdx.x,
              blockDim.x, src_tok, tok_list, (long long)R * R * cap, T,
              group_expert ? grp_order : nullptr);
  }
}

// The row list (see fill_rows), filled by a grid when there are many rows.
__global__ void __launch_bounds__(256) ffn_rows_kernel(const int32_t* __restrict__ grp_n,
                                                       const int32_t* __restrict__ grp_off,
                                                       const int32_t* __restrict__ run_start,
                                                       const int32_t* __restrict__ run_pre,
                                                       int32_t* __restrict__ row_list,
                                                       uint32_t* status, int E, int R, int tk,
                                                       const int32_t* __restrict__ src_tok,
                                                       int32_t* __restrict__ tok_list,
                                                       long long recv_rows, int T,
                                                       const int32_t* __restrict__ grp_order) {
  pdl_wait();
  pdl_trigger();
  fill_rows(grp_n, grp_off, run_start, run_pre, row_list, status, E, R, tk,
            blockIdx.x * blockDim.x + threadIdx.x, gridDim.x * blockDim.x, src_tok, tok_list,
            recv_rows, T, grp_order);
}

template <int STAGE, int BN, int STAGES>
__global__ void __launch_bounds__(GemmThreads<STAGE>::kAll, 1)
    ffn_gemm_bf16_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap mapA,
                         const __grid_constant__ CUtensorMap mapAs,
                         const __grid_constant__ CUtensorMap mapB,
                         const __grid_constant__ CUtensorMap mapBs) {
  using S = GemmShape<STAGE, BN, STAGES>;
  // 256-row token tiles (down stage): the token rows come as two boxes of at most 128 rows
  static_assert(BN <= 128 || STAGE == 1, "256-row token tiles: down stage only");
  constexpr int kBoxRows = BN > 128 ? 128 : BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * S::STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      // the TMA lane's expect_tx arrival, plus one per gather thread (gate/up)
      mbar_init(&full[i], 1 + GemmThreads<STAGE>::kGather);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4);   // one arrival per epilogue warp
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&mapA);
    tma_prefetch_map(&mapB);
    if (a.mt_shared) {
      tma_prefetch_map(&mapAs);
      tma_prefetch_map(&mapBs);
    }
  }
  // the previous kernel's outputs (schedule, activations) and its tensor memory are free from here
  pdl_wait();
  if (warp == 1) {
    tmem_alloc(tmem_slot, S::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int n_tiles = *a.n_tiles;
  const int units = a.n_shared_tiles * a.mt_shared + n_tiles * a.mt_routed;
  const int hot = hot_units(a, n_tiles);

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    const uint64_t pol_w1 = l2_policy_evict_first();   // weights read once
    const uint64_t pol_wk = l2_policy_evict_last();    // weights read again (weight_policy)
    const uint64_t pol_x = l2_policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int sl = blockIdx.x; sl < units && ok; sl += gridDim.x) {
      const int u = interleave_unit(sl, units, hot);
      const Unit t = decode_unit<BN, true>(a, u, n_tiles);
      const bool sh = t.g < 0;
      const uint64_t pol_w = weight_policy(t, pol_w1, pol_wk);
      const CUtensorMap* amap = sh ? &mapAs : &mapA;
      const CUtensorMap* bmap = sh ? &mapBs : &mapB;
      const int we = sh ? 0 : weight_expert(a.group_expert, t.g, a.n_experts,
                                             lane == 0 ? a.status : nullptr);
      const int arow0 = (sh ? 0 : we * a.a_rows_routed) + t.m * 128;
      const int arow1 = arow0 + (sh ? a.a_up_shared : a.a_up_routed);
      // Token rows of the unit. Routed gate/up rows are gathered: a small tile (decode) by
      // this warp with tile::gather4 (lane j loads rows 4j..4j+3; a missing row repeats a valid
      // one of its group, filling a column the epilogue never stores), a larger one by the
      // gather warps with cp.async. The shared expert's rows (x) and the down projection's
      // rows (h) are contiguous: one box per k-step.
      int box_row = -1;
      uint32_t b_bytes = 0;
      int g4[4] = {-1, -1, -1, -1};
      bool g4_on = false;
      if (STAGE == 0 && !sh && t.nlen <= kSmallTile) {
        int nbad = 0;
        if (lane < kSmallTile / 4) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int p = 4 * lane + i;
            int row = -1;
            if (p < t.nlen) {
              const int ci = a.grp_off[t.g] + t.n0 + p;
              row = (ci >= 0 && ci < a.tk) ? a.row_list[ci] : -1;
              if (row >= a.recv_rows) row = -1;
              if (row < 0) ++nbad;
            }
            g4[i] = row;
          }
          int first = -1;
#pragma unroll
          for (int i = 3; i >= 0; --i) first = g4[i] >= 0 ? g4[i] : first;
#pragma unroll
          for (int i = 0; i < 4; ++i) g4[i] = g4[i] >= 0 ? g4[i] : first;
          g4_on = first >= 0;
        }
        const uint32_t on = __ballot_sync(0xffffffffu, g4_on);
        if (__any_sync(0xffffffffu, nbad > 0) && lane == 0) raise_status(a.status, MOE_DEV_BOUNDS);
        b_bytes = 512u * __popc(on);
      }
      int nbox = 1;   // 256-row tiles: a second box when the tile has more than 128 rows
      if (STAGE == 1 || sh) {
        const int row0 = sh ? t.n0 : a.grp_off[t.g] + t.n0;
        const bool in = row0 >= 0 && row0 < (sh ? a.T : a.tk);
        if (!in && lane == 0) raise_status(a.status, MOE_DEV_BOUNDS);
        box_row = in ? row0 : -1;
        if (BN > kBoxRows && t.nlen > kBoxRows) nbox = 2;
        b_bytes = in ? 128u * static_cast<uint32_t>(nbox * (sh ? a.box_shared : a.box_routed)) : 0u;
      }
      const uint32_t tx = S::NA * S::A_BYTES + b_bytes;
      for (int ks = 0; ks < a.k_steps; ++ks) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.status)) {
          ok = false;
          break;
        }
        uint8_t* sa = smem + stage * S::STAGE_BYTES;
        uint8_t* sb = sa + S::NA * S::A_BYTES;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[stage], tx);
          tma_load_2d(sa, amap, &full[stage], ks * 64, arow0, pol_w);
          if (S::NA == 2) tma_load_2d(sa + S::A_BYTES, amap, &full[stage], ks * 64, arow1, pol_w);
          if (box_row >= 0) {
            tma_load_2d(sb, bmap, &full[stage], ks * 64, box_row, pol_x);
            if (BN > kBoxRows && nbox == 2)
              tma_load_2d(sb + kBoxRows * 128, bmap, &full[stage], ks * 64, box_row + kBoxRows,
                          pol_x);
          }
        }
        __syncwarp();
        if (g4_on)
          tma_gather4(sb + lane * 512, bmap, &full[stage], ks * 64, g4[0], g4[1], g4[2], g4[3],
                      pol_x);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // Every load of this CTA is issued: the next kernel may start launching. (Not earlier: its
    // CTAs would sit on the SMs, waiting, for the whole GEMM.)
    pdl_trigger();
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int sl = blockIdx.x; sl < units && ok; sl += gridDim.x) {
        const int u = interleave_unit(sl, units, hot);
        const Unit t = decode_unit<BN, true>(a, u, n_tiles);
        const uint32_t n_pad = static_cast<uint32_t>(max(16, (t.nlen + 15) & ~15));
        const uint32_t idesc = idesc_bf16(128, n_pad);
        const int b = it & 1;
        if (!mbar_wait(&tempty[b], ((it >> 1) & 1) ^ 1u, abort_flag, a.status)) break;
        tc_fence_after();
        const uint32_t d0 = tmem + b * S::ACC_COLS;
        const uint32_t d1 = d0 + BN;
        for (int ks = 0; ks < a.k_steps; ++ks) {
          if (!mbar_wait(&full[stage], phase, abort_flag, a.status)) {
            ok = false;
            break;
          }
          // gate/up: token rows gathered by cp.async (generic proxy) are ordered, observed
          // through the barrier, before the MMA's reads
          if (STAGE == 0) fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t sa = smem_addr(smem + stage * S::STAGE_BYTES);
          const uint32_t sb = sa + S::NA * S::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t db = smem_desc_sw128(sb + kk * 32);
            const uint32_t acc = (ks | kk) != 0;
            mma_f16(d0, smem_desc_sw128(sa + kk * 32), db, idesc, acc);
            if (S::NA == 2) mma_f16(d1, smem_desc_sw128(sa + S::A_BYTES + kk * 32), db, idesc, acc);
          }
          mma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) mma_commit(&tfull[b]);
        ++it;
      }
    }
    __syncwarp();
  } else if (warp >= 6) {
    // ------------------------------ token-row gather (gate/up) ------------------------------
    // Thread gt copies 16-byte chunk j = gt % 8 of rows p = gt/8 + 8i of the token tile into
    // the 128-byte-swizzled layout (chunk j of row p at chunk j ^ (p % 8) = j ^ gt/8), then arms
    // an arrival on the stage's full barrier that the hardware performs once every copy the
    // thread has issued so far has landed (a thread with nothing to copy arrives at once). The
    // MMA thread puts a proxy fence between its wait and its tensor-core reads.
    constexpr int kRowsPer = BN / 8;
    const int gt = threadIdx.x - 192;
    const int j = gt & 7, rg = gt >> 3;
    const uint32_t dst_off = static_cast<uint32_t>(rg * 128 + ((j ^ rg) << 4));
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int sl = blockIdx.x; sl < units && ok; sl += gridDim.x) {
      const int u = interleave_unit(sl, units, hot);
      const Unit t = decode_unit<BN, true>(a, u, n_tiles);
      const bool gather = STAGE == 0 && t.g >= 0 && t.nlen > kSmallTile;
      const uint8_t* src[kRowsPer];
#pragma unroll
      for (int i = 0; i < kRowsPer; ++i) {
        const int p = rg + 8 * i;
        src[i] = nullptr;
        if (gather && p < t.nlen) {
          const int ci = a.grp_off[t.g] + t.n0 + p;
          const long long row = (ci >= 0 && ci < a.tk) ? a.row_list[ci] : -1;
          if (row >= 0 && row < a.recv_rows) src[i] = a.gather_base + row * a.gather_ld + j * 16;
          else raise_status(a.status, MOE_DEV_BOUNDS);
        }
      }
      for (int ks = 0; ks < a.k_steps; ++ks) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.status)) {
          ok = false;
          break;
        }
        const uint32_t sb =
            smem_addr(smem + stage * S::STAGE_BYTES + S::NA * S::A_BYTES) + dst_off;
#pragma unroll
        for (int i = 0; i < kRowsPer; ++i)
          if (src[i])
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sb + i * 1024),
                         "l"(src[i] + ks * 128)
                         : "memory");
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(
                         smem_addr(&full[stage]))
                     : "memory");
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // after an abort: copies still in flight land before the CTA exits
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else {
    // ------------------------------ epilogue ------------------------------
    const int quarter = warp & 3;  // tensor-memory lanes 32*quarter .. +31
    const int rrow = quarter * 32 + lane;
    int it = 0;
    for (int sl = blockIdx.x; sl < units; sl += gridDim.x) {
      const int u = interleave_unit(sl, units, hot);
      const Unit t = decode_unit<BN, true>(a, u, n_tiles);
      const bool sh = t.g < 0;
      const int b = it & 1;
      if (!mbar_wait(&tfull[b], (it >> 1) & 1, abort_flag, a.status)) break;
      tc_fence_after();
      const uint32_t tb = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + b * S::ACC_COLS;
      const int f = t.m * 128 + rrow;  // output column
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(sh ? a.out_shared : a.out_routed);
      const int ld = sh ? a.ld_shared : a.ld_routed;
      // output row of tile column lane + 32*i, looked up once per unit (-1: not stored)
      long long orows[BN / 32];
      const int base = sh ? 0 : a.grp_off[t.g];
#pragma unroll
      for (int i = 0; i < BN / 32; ++i) {
        const int p = lane + 32 * i;
        long long o = -1;
        if (p < t.nlen) {
          if (sh) {
            o = t.n0 + p;
          } else if (STAGE == 0) {
            o = base + t.n0 + p;
            if (o < 0 || o >= a.tk) o = -1;
          } else {
            const int ci = base + t.n0 + p;
            o = (ci >= 0 && ci < a.tk) ? a.row_list[ci] : -1;
            if (o >= a.recv_rows) o = -1;
          }
        }
        orows[i] = o;
      }
      for (int c0 = 0; c0 < t.nlen; c0 += 16) {
        uint32_t ra[16], rb[16];
        tmem_ld16(tb + c0, ra);
        if (S::NA == 2) tmem_ld16(tb + BN + c0, rb);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int p = c0 + j;   // c0 is a multiple of 16: column p is lane p % 32 of group p / 32
          const long long orow = __shfl_sync(0xffffffffu, orows[(c0 >> 5) & (BN / 32 - 1)], p & 31);
          if (p >= t.nlen || orow < 0) continue;
          float val;
          if (S::NA == 2) val = silu(__uint_as_float(ra[j])) * __uint_as_float(rb[j]);
          else val = __uint_as_float(ra[j]);
          out[orow * ld + f] = __float2bfloat16_rn(val);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[b]);
      ++it;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, S::TMEM_COLS);
  }
}

template <int STAGE, int BN, int STAGES>
cudaError_t run_gemm(const GemmArgs& a, const CUtensorMap& mA, const CUtensorMap& mAs,
                     const CUtensorMap& mB, const CUtensorMap& mBs, cudaStream_t st, bool pdl,
                     int ctas) {
  using S = GemmShape<STAGE, BN, STAGES>;
  auto kern = ffn_gemm_bf16_kernel<STAGE, BN, STAGES>;
  const cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(kern), S::SMEM);
  if (err != cudaSuccess) return err;
  return launch_kernel(kern, dim3(ctas > 0 ? ctas : sm_count()), dim3(GemmThreads<STAGE>::kAll),
                       S::SMEM, st, pdl, a, mA, mAs, mB, mBs);
}

}  // namespace

// ---------------------------------------------------------------------------------------
// Host side: tensor maps
// ---------------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D row-major tensor [rows][cols] of 16-bit (elem_bytes 2) or 8-bit elements, box of
// box_rows rows x 128 bytes, 128-byte swizzle.
bool make_tensor_map_2d(CUtensorMap* m, const void* base, int elem_bytes, uint64_t cols, uint64_t rows,
              uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * elem_bytes};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elem_bytes), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r =
      fn(m, elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t ensure_smem_limit(const void* kern, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  // a fixed table, so that no call allocates host memory either (when it is full the runtime
  // is simply called every time)
  struct Entry {
    const void* kern;
    int dev;
    size_t bytes;
  };
  constexpr int kEntries = 256;
  static std::mutex mu;
  static Entry set_so_far[kEntries];
  static int used = 0;
  std::lock_guard<std::mutex> lock(mu);
  Entry* hit = nullptr;
  for (int i = 0; i < used; ++i)
    if (set_so_far[i].kern == kern && set_so_far[i].dev == dev) hit = &set_so_far[i];
  if (hit && hit->bytes >= bytes) return cudaSuccess;
  err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(bytes));
  if (err != cudaSuccess) return err;
  if (hit)
    hit->bytes = bytes;
  else if (used < kEntries)
    set_so_far[used++] = Entry{kern, dev, bytes};
  return cudaSuccess;
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}


cudaError_t launch_quant_x(const moe_cfg& c, const WsLayout& L, const void* x, char* ws,
                           cudaStream_t st, bool pdl) {
  return launch_quant_rows_e4m3(x, c.T, c.d, ws + L.xq, reinterpret_cast<float*>(ws + L.xq_scales),
                                st, pdl, pow2_scales(c));
}

cudaError_t launch_ffn_setup(const moe_cfg& c, const WsLayout& L, const int32_t* counts,
                             const void* x, char* ws, cudaStream_t st, bool pdl,
                             const int32_t* src_tok, bool quantise,
                             const int32_t* group_expert) {
  if (quantise && is_fp8(c) && (c.d_ff_shared || src_tok)) {
    const cudaError_t err = launch_quant_x(c, L, x, ws, st, pdl);
    if (err != cudaSuccess) return err;
  }
  uint32_t* status = reinterpret_cast<uint32_t*>(ws + L.status);
  const size_t stage = (size_t)c.R * c.E * sizeof(int32_t);
  const int32_t* grp_n = reinterpret_cast<const int32_t*>(ws + L.grp_n);
  const int32_t* grp_off = reinterpret_cast<const int32_t*>(ws + L.grp_off);
  const int tk = c.T * c.k;
  const int plan_threads = c.E <= 32 ? 32 : (c.E + 31) / 32 * 32;   // one thread per expert
  cudaError_t err = launch_kernel(
      ffn_plan_kernel, dim3(1), dim3(plan_threads), stage <= kPlanStageBytes ? stage : 0, st, pdl,
      counts, reinterpret_cast<int32_t*>(ws + L.grp_n), reinterpret_cast<int32_t*>(ws + L.grp_off),
      reinterpret_cast<int32_t*>(ws + L.n_tiles), reinterpret_cast<Tile*>(ws + L.tiles),
      reinterpret_cast<int32_t*>(ws + L.run_start), reinterpret_cast<int32_t*>(ws + L.run_pre),
      reinterpret_cast<int32_t*>(ws + L.row_list), status, c.E, c.R, cap_of(c), L.bn,
      L.max_tiles, tk, src_tok, src_tok ? reinterpret_cast<int32_t*>(ws + L.tok_list) : nullptr,
      c.T, group_expert, reinterpret_cast<int32_t*>(ws + L.grp_order),
      reinterpret_cast<int32_t*>(ws + L.n_tiles2), reinterpret_cast<Tile*>(ws + L.tiles2),
      L.bn == 128 && !is_fp8(c) ? L.max_tiles2 : 0);   // the bf16 GEMMs' 256-row schedule
  if (err != cudaSuccess) return err;
  if (tk <= kPlanFusedRows) return cudaSuccess;   // the plan CTA filled the row list
  const int blocks = (tk + 255) / 256 < 4 * 152 ? (tk + 255) / 256 : 4 * 152;
  return launch_kernel(
      ffn_rows_kernel, dim3(blocks), dim3(256), 0, st, pdl, grp_n, grp_off,
      reinterpret_cast<const int32_t*>(ws + L.run_start),
      reinterpret_cast<const int32_t*>(ws + L.run_pre), reinterpret_cast<int32_t*>(ws + L.row_list),
      status, c.E, c.R, tk, src_tok,
      src_tok ? reinterpret_cast<int32_t*>(ws + L.tok_list) : nullptr,
      (long long)c.R * c.R * cap_of(c), c.T,
      group_expert ? reinterpret_cast<const int32_t*>(ws + L.grp_order) : nullptr);
}

cudaError_t prepare_bf16_gemm(const moe_cfg& c, const WsLayout& L, int stage, const void* recv,
                              const void* x, const moe_weights& w, void* ebuf, void* shared_out,
                              char* ws, const FfnPart& part, GemmArgs* args,
                              CUtensorMap maps[4], bool wide) {
  const int cap = cap_of(c);
  const long long recv_rows = (long long)c.R * c.R * cap;
  const int F = c.d_ff, Fs = c.d_ff_shared, d = c.d, tk = c.T * c.k;
  const bool has_shared = Fs > 0;
  // gather mode: the gate/up stage reads routed token rows from x, by token, through the
  // schedule's token list (the down stage still writes ebuf at the receive rows)
  const bool gather = part.src_tok != nullptr && stage == 0;

  GemmArgs a{};
  wide = wide && stage == 1;
  const int tbn = wide ? 2 * L.bn : L.bn;   // token-tile rows of this launch's schedule
  a.tiles = reinterpret_cast<const Tile*>(ws + (wide ? L.tiles2 : L.tiles));
  a.n_tiles = reinterpret_cast<const int32_t*>(ws + (wide ? L.n_tiles2 : L.n_tiles));
  a.grp_off = reinterpret_cast<const int32_t*>(ws + L.grp_off);
  a.row_list = reinterpret_cast<const int32_t*>(ws + L.row_list);
  a.tk = tk;
  a.recv_rows = recv_rows;
  a.T = c.T;
  a.status = reinterpret_cast<uint32_t*>(ws + L.status);
  a.n_shared_tiles = has_shared ? (c.T + tbn - 1) / tbn : 0;
  a.group_expert = part.group_expert;
  const int n_w = part.weight_experts > 0 ? part.weight_experts : c.E;
  a.n_experts = n_w;

  CUtensorMap& mA = maps[0];
  CUtensorMap& mAs = maps[1];
  CUtensorMap& mB = maps[2];
  CUtensorMap& mBs = maps[3];
  bool ok = true;
  if (stage == 0) {
    a.mt_routed = F / 128;
    a.mt_shared = has_shared ? Fs / 128 : 0;
    a.k_steps = d / 64;
    a.a_rows_routed = 2 * F;
    a.a_up_routed = F;
    a.a_up_shared = Fs;
    a.out_routed = ws + L.h;
    a.out_shared = has_shared ? static_cast<void*>(ws + L.hs) : nullptr;
    a.ld_routed = F;
    a.ld_shared = Fs;
    a.gather_base = static_cast<const uint8_t*>(gather ? x : recv);
    a.gather_ld = 2ll * d;
    a.box_routed = 1;
    a.box_shared = c.T < L.bn ? c.T : L.bn;
    if (gather) {
      a.row_list = reinterpret_cast<const int32_t*>(ws + L.tok_list);
      a.recv_rows = c.T;
    }
    ok &= make_tensor_map_2d(&mA, w.w13, 2, d, (uint64_t)n_w * 2 * F, 128);
    ok &= make_tensor_map_2d(&mB, gather ? x : recv, 2, d, gather ? c.T : recv_rows, 1);
    if (has_shared) {
      ok &= make_tensor_map_2d(&mAs, w.ws13, 2, d, 2ull * Fs, 128);
      ok &= make_tensor_map_2d(&mBs, x, 2, d, c.T, a.box_shared);
    }
  } else {
    a.mt_routed = d / 128;
    a.mt_shared = has_shared ? d / 128 : 0;
    a.k_steps = F / 64;
    a.a_rows_routed = d;
    a.a_up_routed = 0;
    a.a_up_shared = 0;
    a.out_routed = ebuf;
    a.out_shared = shared_out;
    a.ld_routed = d;
    a.ld_shared = d;
    // the down projection's input rows are contiguous: one box of up to bn rows per k-step
    a.box_routed = tk < L.bn ? tk : L.bn;
    a.box_shared = c.T < L.bn ? c.T : L.bn;
    ok &= make_tensor_map_2d(&mA, w.w2, 2, F, (uint64_t)n_w * d, 128);
    ok &= make_tensor_map_2d(&mB, ws + L.h, 2, F, tk, a.box_routed);
    if (has_shared) {
      if (Fs != F) return cudaErrorNotSupported;  // one K loop length per launch
      ok &= make_tensor_map_2d(&mAs, w.ws2, 2, Fs, d, 128);
      ok &= make_tensor_map_2d(&mBs, ws + L.hs, 2, Fs, c.T, a.box_shared);
    }
  }
  if (stage == 0 && has_shared && Fs % 128) return cudaErrorInvalidValue;
  if (!has_shared) {
    mAs = mA;
    mBs = mB;
  }
  if (!ok) return cudaErrorInvalidValue;
  if (!part.routed) a.mt_routed = 0;   // this launch runs the shared expert's units only
  if (!part.shared) {                  // ... or the routed experts' units only
    a.mt_shared = 0;
    a.n_shared_tiles = 0;
  }
  *args = a;
  return cudaSuccess;
}

cudaError_t launch_ffn_gemm(const moe_cfg& c, const WsLayout& L, int stage, const void* recv,
                            const float* recv_scales, const void* x, const moe_weights& w,
                            void* ebuf, void* shared_out, char* ws, cudaStream_t st, bool pdl,
                            const FfnPart& part) {
  if (pow2_scales(c))
    return launch_ffn_gemm_mx8(c, L, stage, recv, recv_scales, w, ebuf, shared_out, ws, st, pdl,
                               part);
  if (is_fp8(c))
    return launch_ffn_gemm_e4m3(c, L, stage, recv, recv_scales, w, ebuf, shared_out, ws, st, pdl,
                                part);
  // down, with a full 128-row token tile per expert on average: 256-row token tiles (M = 128
  // weight rows, N up to 256), so each weight tile is read from L2 once per 256 rows
  const int n_experts = part.weight_experts > 0 ? part.weight_experts : c.E;   // not slots
  const bool wide = stage == 1 && L.bn == 128 && (long long)c.T * c.k >= 128ll * n_experts;
  GemmArgs a{};
  CUtensorMap m[4];
  const cudaError_t err =
      prepare_bf16_gemm(c, L, stage, recv, x, w, ebuf, shared_out, ws, part, &a, m, wide);
  if (err != cudaSuccess) return err;
  if (L.bn == 64) {
    if (stage == 0) return run_gemm<0, 64, 5>(a, m[0], m[1], m[2], m[3], st, pdl, part.ctas);
    return run_gemm<1, 64, 8>(a, m[0], m[1], m[2], m[3], st, pdl, part.ctas);
  }
  if (stage == 0) return run_gemm<0, 128, 4>(a, m[0], m[1], m[2], m[3], st, pdl, part.ctas);
  if (wide) return run_gemm<1, 256, 4>(a, m[0], m[1], m[2], m[3], st, pdl, part.ctas);
  return run_gemm<1, 128, 6>(a, m[0], m[1], m[2], m[3], st, pdl, part.ctas);
}

}  // namespace moe
