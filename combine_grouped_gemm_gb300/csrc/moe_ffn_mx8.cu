// e4m3 expert GEMMs with power-of-two block scales applied by the tensor core (the second FP8
// recipe, MOE_FP8_E4M3_POW2).
//
// Method: as in moe_ffn.cu ("7.13 Serving Mixture-of-Experts", Expert Parallelism Mechanics,
// expert compute; "One-Sided Expert-Parallel All-to-All ...", abstract, grouped GEMMs reading
// the receive buffers in place) with e4m3 activations and weights in 1x128 / 128x128 blocks
// ("Serving Mixture-of-Experts", DeepEP section, FP8 dispatch). With power-of-two scales each
// block's scale is a UE8M0 byte (its exponent), and the block-scaled MMA
// (tcgen05.mma kind::mxf8f6f4.block_scale) multiplies every 32-wide K slice of A and B by its
// scale bytes before accumulating. The whole K loop then accumulates in one tensor-memory
// accumulator, with no per-block promotion on the CUDA cores (the amax/448 recipe's kernel,
// moe_ffn_fp8.cu, is bound by that promotion chain).
//
// Scale bytes in tensor memory, for an M = 128, N = 256 MMA (scale_vec::1X, one byte per row
// per 32-wide K slice; a 32-bit cell holds the bytes of four slices, chosen by the instruction
// descriptor's scale-factor ids): the A scales of row i sit in lane i, column base + i / 32;
// the B scales of column n in lanes 32q + n % 32 of every lane quarter q, column base + n / 32.
// Here one 128-K block has one scale, so a cell holds the same byte four times.
//
// The input rows' scale bytes come from row-major byte tables in the workspace (64 bytes a
// row, byte b for the row's 128-column block b): a scale warp loads its row's bytes once per
// unit, as four 16-byte vectors, one unit ahead, instead of one scattered fp32 scale per
// k-step. mx8_scale_bytes_kernel fills the gate/up tables from the dispatch's fp32 scales;
// the gate/up epilogue writes h's bytes itself.
//
// Roles (768 threads, one CTA per SM, persistent over the unit list):
//   warps 0..3    scale warps: warp q writes its lane quarter's A scale cell and B scale cells
//                 of each k-step into the stage's tensor-memory scale slot (tcgen05.st)
//   warps 4..19   epilogue: warp w drains lanes 32*(w%4).. and columns 32*((w-4)/4).. of the
//                 accumulator (gate and up, or the two output tiles) into registers, releases
//                 it, then finishes the unit (SwiGLU + e4m3 re-quantisation, or bf16 rows)
//   warp 20       TMA producer: weight tiles, and contiguous token rows (the shared expert's
//                 x, the down projection's h) as one box
//   warp 21       tensor-memory allocation; lane 0 issues the MMAs
//   warps 22, 23  copy warps (gate/up): the routed token rows, gathered by row with cp.async
//                 into the 128-byte-swizzled tile (a TMA tile::gather4 per four rows measured
//                 about four times slower on 128-row tiles)
// Units are weight-tile-major (the token tiles that read one weight tile run on adjacent CTAs
// and fetch each 32 KB weight tile of a k-step together). Each CTA decodes its units once,
// into a table in shared memory, before the roles start.
#include "moe_device.cuh"
#include "moe_scale.cuh"

namespace moe {
namespace {

struct Mx8Args {
  const Tile* tiles;
  const int32_t* n_tiles;
  const int32_t* grp_off;
  const int32_t* row_list;      // compact row -> receive row (or token, gather mode)
  int tk;
  long long a_rows_routed;      // bound of routed A row indices
  int T;
  int mt_routed, mt_shared;     // weight tiles (units along N) per group
  int n_shared_tiles;
  int k_steps;                  // K / 128
  int b_rows_routed;            // weight rows per routed expert (2F or d)
  int b_up_routed, b_up_shared; // offset of a unit's second weight tile (up rows, or the next
                                // 128 output columns)
  const uint8_t* sf_routed;     // scale bytes of the routed input rows, by compact row
  const uint8_t* sf_shared;     // scale bytes of the shared expert's input rows, by token
  const float* w_sc_routed;     // [E][b_rows_routed/128][K/128]
  const float* w_sc_shared;     // [b_rows_shared/128][K/128]
  void* out_routed;             // gate/up: e4m3 h [tk][F]; down: bf16 ebuf [recv rows][d]
  uint8_t* out_sf_routed;       // gate/up: h's scale bytes, by compact row
  void* out_shared;             // gate/up: e4m3 hs [T][Fs]; down: bf16 shared_out [T][d]
  uint8_t* out_sf_shared;       // gate/up: hs's scale bytes, by token
  int ld_routed, ld_shared;     // output row length (elements)
  long long out_rows_routed;    // bound of routed output row indices
  int box_routed, box_shared;   // rows per box of the contiguous token-row maps
  const void* gather_base;      // gate/up: the routed token rows' array (receive buffer or xq)
  long long gather_ld;          // bytes per row of it
  uint32_t* status;
  const int32_t* group_expert;  // expert whose weights group g uses (nullptr: expert g)
  int n_experts;
};

// One unit of a CTA: group g (-1: the shared expert), token tile [n0, n0 + nlen), weight tile
// m, the group's first compact row goff and the expert whose weights it reads.
struct UnitInfo {
  int g, n0, nlen, m, goff, we;
};

__device__ __forceinline__ int weight_expert_mx(const int32_t* group_expert, int g, int n_experts,
                                                uint32_t* status) {
  if (!group_expert) return g;
  const int e = group_expert[g];
  if (e >= 0 && e < n_experts) return e;
  if (status) raise_status(status, MOE_DEV_BOUNDS);
  return 0;
}

// Unit u -> its UnitInfo, weight-tile-major; shared-expert units first. n_tiles: entries in
// the tile list. status (nullable) receives MOE_DEV_BOUNDS for a slot outside the weights.
__device__ __forceinline__ UnitInfo decode_unit_mx(const Mx8Args& a, int u, int n_tiles,
                                                   uint32_t* status) {
  UnitInfo r;
  const int us = a.n_shared_tiles * a.mt_shared;
  if (u < us) {
    r.g = -1;
    r.m = u / a.n_shared_tiles;
    r.n0 = (u - r.m * a.n_shared_tiles) * 128;
    r.nlen = min(128, a.T - r.n0);
    r.goff = 0;
    r.we = 0;
  } else {
    const int v = u - us;
    const int tt0 = v / a.mt_routed;   // a tile of the unit's expert (the ranges coincide)
    const Tile t0 = a.tiles[tt0];
    const int base = tt0 - t0.n0 / 128;
    // (a list cut short at its bound, already reported, keeps every index inside it)
    const int nt = max(1, min(t0.ntiles, n_tiles - base));
    const int local = v - base * a.mt_routed;
    r.m = local / nt;
    const int j = local - r.m * nt;
    const Tile t = base + j == tt0 ? t0 : a.tiles[base + j];
    r.g = t.group;
    r.n0 = t.n0;
    r.nlen = t.nlen;
    r.goff = a.grp_off[t.group];
    r.we = weight_expert_mx(a.group_expert, t.group, a.n_experts, status);
  }
  return r;
}

constexpr int kStages = 4;
constexpr int kSfWarps = 4;
constexpr int kEpiWarps = 16;
constexpr int kProducerWarp = kSfWarps + kEpiWarps;   // 20
constexpr int kMmaWarp = kProducerWarp + 1;           // 21
constexpr int kCopyWarp0 = kMmaWarp + 1;              // 22, 23
constexpr int kCopyThreads = 64;
constexpr int kThreads = kCopyWarp0 * 32 + kCopyThreads;   // 768
constexpr int kABytes = 128 * 128;                    // 128 token rows x 128 e4m3
constexpr int kBBytes = 128 * 128;                    // one 128-row weight tile
constexpr int kStageBytes = kABytes + 2 * kBBytes;
constexpr int kTmemCols = 512;
constexpr int kSfCol0 = 256;        // scale slots after the 256-column accumulator
constexpr int kSfSlotCols = 32;     // per stage: A scales at +0..3, B scales at +16..23
constexpr int kMaxUnitTable = 256;  // units of a CTA decoded into shared memory (more: on the fly)
constexpr int kBarOff = kStages * kStageBytes;
constexpr int kAmaxOff = kBarOff + 512;                          // [2][4][32][4] floats
constexpr int kUnitOff = kAmaxOff + 2 * 4 * 32 * 4 * 4;          // UnitInfo [kMaxUnitTable]
constexpr int kWsfOff = kUnitOff + kMaxUnitTable * (int)sizeof(UnitInfo);   // [4 warps][128] B
constexpr int kSmem = kWsfOff + kSfWarps * 2 * kSfRowBytes + 1024;

// Instruction descriptor of the block-scaled e4m3 MMA, M = 128, N = 256, K-major operands:
// B scale-factor id in bits 4-5, formats e4m3 (0) in bits 7-9 and 10-12, N >> 3 in bits 17-22,
// UE8M0 scales (bit 23), M >> 4 in bits 24-28, A scale-factor id in bits 29-30.
__device__ __forceinline__ uint32_t idesc_mx8(uint32_t sf_id) {
  return (sf_id << 4) | ((256u >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24) | (sf_id << 29);
}

__device__ __forceinline__ void mma_mx8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, "
      "[%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v)
               : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, uint32_t v0, uint32_t v1) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %1, %1, %1, %2, %2, %2, %2};" ::"r"(taddr),
      "r"(v0), "r"(v1)
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t rep4(uint32_t byte) { return byte * 0x01010101u; }

// The hardware arrives on bar once every cp.async this thread has issued so far has landed;
// the arrival counts as one of the barrier's expected arrivals.
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

template <int STAGE>
__global__ void __launch_bounds__(kThreads, 1)
    ffn_gemm_mx8_kernel(const Mx8Args a, const __grid_constant__ CUtensorMap mapA,
                        const __grid_constant__ CUtensorMap mapAs,
                        const __grid_constant__ CUtensorMap mapB,
                        const __grid_constant__ CUtensorMap mapBs) {
  // weight rows between consecutive units' first tiles: gate/up 128 (the second tile is the up
  // projection, F rows further); down 256 (two adjacent 128-column output tiles)
  constexpr int kStep = STAGE == 0 ? 128 : 256;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* xbar = acc_empty + 1;   // [4] amax exchange of the warps on one lane quarter
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xbar + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* amax_x = reinterpret_cast<float*>(smem + kAmaxOff);
  UnitInfo* unit_tab = reinterpret_cast<UnitInfo*>(smem + kUnitOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      // the producer's expect_tx arrival, the scale warps, (gate/up) every copy thread
      mbar_init(&full[i], 1 + kSfWarps + (STAGE == 0 ? kCopyThreads : 0));
      mbar_init(&empty[i], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kEpiWarps);
    for (int i = 0; i < 4; ++i) mbar_init(&xbar[i], 4);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_map(&mapA);
    tma_prefetch_map(&mapB);
    if (a.mt_shared) {
      tma_prefetch_map(&mapAs);
      tma_prefetch_map(&mapBs);
    }
  }
  // the previous kernel's outputs (schedule, activations) and its tensor memory are free from here
  pdl_wait();
  const int n_tiles = *a.n_tiles;
  const int units = a.n_shared_tiles * a.mt_shared + n_tiles * a.mt_routed;
  // units of this CTA: blockIdx.x, blockIdx.x + gridDim.x, ...
  const int n_my = blockIdx.x < units ? (units - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  for (int i = threadIdx.x; i < min(n_my, kMaxUnitTable); i += blockDim.x)
    unit_tab[i] = decode_unit_mx(a, blockIdx.x + i * gridDim.x, n_tiles, a.status);
  auto unit_at = [&](int i) -> UnitInfo {
    return i < kMaxUnitTable ? unit_tab[i]
                             : decode_unit_mx(a, blockIdx.x + i * gridDim.x, n_tiles, nullptr);
  };
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------ TMA producer ------------------------------
    const uint64_t pol_w = l2_policy_evict_last();
    const uint64_t pol_x = l2_policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int i = 0; i < n_my && ok; ++i) {
      const UnitInfo t = unit_at(i);
      const bool sh = t.g < 0;
      const CUtensorMap* amap = sh ? &mapAs : &mapA;
      const CUtensorMap* bmap = sh ? &mapBs : &mapB;
      const int brow0 = (sh ? 0 : t.we * a.b_rows_routed) + t.m * kStep;
      const int brow1 = brow0 + (sh ? a.b_up_shared : a.b_up_routed);
      // Token rows: the shared expert's rows (x) and the down projection's rows (h) are one box
      // per k-step; routed gate/up rows are gathered by the copy warps.
      int box_row = -1;
      uint32_t a_bytes = 0;
      if (STAGE == 1 || sh) {
        const int row0 = sh ? t.n0 : t.goff + t.n0;
        const bool in = row0 >= 0 && row0 < (sh ? a.T : a.tk);
        if (!in && lane == 0) raise_status(a.status, MOE_DEV_BOUNDS);
        box_row = in ? row0 : -1;
        a_bytes = in ? 128u * static_cast<uint32_t>(sh ? a.box_shared : a.box_routed) : 0u;
      }
      const uint32_t tx = 2 * kBBytes + a_bytes;
      for (int ks = 0; ks < a.k_steps; ++ks) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.status)) {
          ok = false;
          break;
        }
        uint8_t* sa = smem + stage * kStageBytes;
        uint8_t* sb = sa + kABytes;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[stage], tx);
          tma_load_2d(sb, bmap, &full[stage], ks * 128, brow0, pol_w);
          tma_load_2d(sb + kBBytes, bmap, &full[stage], ks * 128, brow1, pol_w);
          if (box_row >= 0) tma_load_2d(sa, amap, &full[stage], ks * 128, box_row, pol_x);
        }
        __syncwarp();
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // Every load of this CTA is issued: the next kernel may start launching.
    pdl_trigger();
  } else if (warp == kMmaWarp) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int i = 0; i < n_my && ok; ++i) {
        // the epilogue has drained the previous unit's accumulator
        if (!mbar_wait(acc_empty, (static_cast<uint32_t>(i) & 1u) ^ 1u, abort_flag, a.status))
          break;
        tc_fence_after();
        for (int ks = 0; ks < a.k_steps; ++ks) {
          if (!mbar_wait(&full[stage], phase, abort_flag, a.status)) {
            ok = false;
            break;
          }
          // gate/up: the gathered token rows were written by cp.async (generic proxy); the
          // fence orders them, observed through the barrier, before the MMA's reads
          if (STAGE == 0) fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t sa = smem_addr(smem + stage * kStageBytes);
          const uint32_t sb = sa + kABytes;
          const uint32_t sf = tmem + kSfCol0 + stage * kSfSlotCols;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_mx8(tmem, smem_desc_sw128(sa + kk * 32), smem_desc_sw128(sb + kk * 32),
                    idesc_mx8(static_cast<uint32_t>(kk)), sf, sf + 16, (ks | kk) != 0);
          mma_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) mma_commit(acc_full);
      }
    }
    __syncwarp();
  } else if (warp >= kCopyWarp0) {
    // ------------------------------ copy warps ------------------------------
    // Gate/up only. Thread gt copies 16-byte chunk j = gt % 8 of tile rows p = gt/8 + 8i
    // (i < 16) into the 128-byte-swizzled layout the MMA descriptor expects (chunk j of row p at
    // chunk j ^ (p % 8) = j ^ gt/8), then arms an arrival on the stage's full barrier that the
    // hardware performs once its copies have landed (a thread with nothing to copy arrives at
    // once). The MMA thread puts a proxy fence between its wait and its tensor-core reads.
    if (STAGE == 0) {
      const int gt = threadIdx.x - kCopyWarp0 * 32;
      const int j = gt & 7, rg = gt >> 3;
      const uint32_t dst_off = static_cast<uint32_t>(rg * 128 + ((j ^ rg) << 4));
      const uint8_t* gbase = reinterpret_cast<const uint8_t*>(a.gather_base) + j * 16;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int i = 0; i < n_my && ok; ++i) {
        const UnitInfo t = unit_at(i);
        const bool gather = t.g >= 0;
        int src[16];   // row of each of the thread's 16 tile rows (-1: none)
#pragma unroll
        for (int i2 = 0; i2 < 16; ++i2) {
          const int p = rg + 8 * i2;
          src[i2] = -1;
          if (gather && p < t.nlen) {
            const int ci = t.goff + t.n0 + p;
            const long long row = (ci >= 0 && ci < a.tk) ? a.row_list[ci] : -1;
            if (row >= 0 && row < a.a_rows_routed) src[i2] = static_cast<int>(row);
            else raise_status(a.status, MOE_DEV_BOUNDS);
          }
        }
        for (int ks = 0; ks < a.k_steps; ++ks) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.status)) {
            ok = false;
            break;
          }
          if (gather) {
            const uint32_t sa = smem_addr(smem + stage * kStageBytes) + dst_off;
            const uint8_t* gk = gbase + ks * 128;
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2)
              if (src[i2] >= 0)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa + i2 * 1024),
                             "l"(gk + (long long)src[i2] * a.gather_ld)
                             : "memory");
          }
          cp_async_arrive(&full[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // after an abort: copies still in flight land before the CTA exits
      asm volatile("cp.async.wait_all;" ::: "memory");
    }
  } else if (warp < kSfWarps) {
    // ------------------------------ scale warps ------------------------------
    // Warp q, lane l: tile row r = 32q + l. Per unit: the row's scale bytes (four 16-byte loads
    // of its table row) and the unit's two weight-block scales of every k-step (lane l loads
    // k-steps l and l + 32, converted to bytes in the warp's shared-memory rows), both issued
    // one unit ahead. Per k-step: the A cell (lane r, column q of the stage's slot) and the B
    // cells (columns 16..23, gate bytes then up bytes) once the MMAs that read the slot's
    // previous k-step have completed (the stage's empty barrier); the stage's full barrier
    // then counts this warp's arrival.
    const int q = warp;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const int r = q * 32 + lane;
    uint8_t* wsf = smem + kWsfOff + q * 2 * kSfRowBytes;   // [gate 64][up 64] bytes
    const int kb_n = a.k_steps;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    bool scale_ok = true;
    uint4 na[4];
    float nw[4];   // weight scales of k-steps l, l + 32 (gate), l, l + 32 (up)
    auto issue = [&](int i) {
      const UnitInfo t = unit_at(i);
      const bool sh = t.g < 0;
      const long long row = sh ? (long long)t.n0 + r : (long long)t.goff + t.n0 + r;
      const bool in = r < t.nlen && row >= 0 && row < (sh ? a.T : a.tk);
      const uint4* src = reinterpret_cast<const uint4*>((sh ? a.sf_shared : a.sf_routed) +
                                                        (in ? row : 0) * kSfRowBytes);
      // (defaults first, then loads under a predicate, so nothing waits for them before their
      // use one unit later)
#pragma unroll
      for (int j = 0; j < 4; ++j) na[j] = make_uint4(0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu, 0x7f7f7f7fu);
      if (in) {
#pragma unroll
        for (int j = 0; j < 4; ++j) na[j] = __ldg(src + j);
      }
      const float* wsc = (sh ? a.w_sc_shared
                             : a.w_sc_routed + (size_t)t.we * (a.b_rows_routed / 128) * kb_n) +
                         (size_t)t.m * (kStep / 128) * kb_n;
      const int w_up = (sh ? a.b_up_shared : a.b_up_routed) / 128 * kb_n;
      nw[0] = nw[1] = nw[2] = nw[3] = 1.0f;
      if (lane < kb_n) {
        nw[0] = __ldg(wsc + lane);
        nw[2] = __ldg(wsc + w_up + lane);
      }
      if (lane + 32 < kb_n) {
        nw[1] = __ldg(wsc + lane + 32);
        nw[3] = __ldg(wsc + w_up + lane + 32);
      }
    };
    if (n_my > 0) issue(0);
    for (int i = 0; i < n_my && ok; ++i) {
      uint32_t aw[16] = {na[0].x, na[0].y, na[0].z, na[0].w, na[1].x, na[1].y, na[1].z, na[1].w,
                         na[2].x, na[2].y, na[2].z, na[2].w, na[3].x, na[3].y, na[3].z, na[3].w};
      __syncwarp();   // every lane is done with the previous unit's weight bytes
      wsf[lane] = static_cast<uint8_t>(ue8m0_of(nw[0], scale_ok));
      wsf[lane + 32] = static_cast<uint8_t>(ue8m0_of(nw[1], scale_ok));
      wsf[64 + lane] = static_cast<uint8_t>(ue8m0_of(nw[2], scale_ok));
      wsf[96 + lane] = static_cast<uint8_t>(ue8m0_of(nw[3], scale_ok));
      __syncwarp();
      if (i + 1 < n_my) issue(i + 1);
      uint32_t cur = aw[0];
      for (int ks = 0; ks < kb_n; ++ks) {
        const uint32_t ab = cur & 0xFFu;
        cur >>= 8;
        if ((ks & 3) == 3) {   // the next four k-steps' bytes
#pragma unroll
          for (int j = 0; j < 15; ++j) aw[j] = aw[j + 1];
          cur = aw[0];
        }
        const uint32_t gb = wsf[ks], ub = wsf[64 + ks];
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t slot = tmem + lane_base + kSfCol0 + stage * kSfSlotCols;
        tmem_st1(slot + q, rep4(ab));
        tmem_st8(slot + 16, rep4(gb), rep4(ub));
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[stage]);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!__all_sync(0xffffffffu, scale_ok) && lane == 0) raise_status(a.status, MOE_DEV_SCALE);
  } else {
    // ------------------------------ epilogue ------------------------------
    const int quarter = warp & 3;
    const int part = (warp - kSfWarps) >> 2;   // columns 32*part .. 32*part+31 of each tile
    const int r = quarter * 32 + lane;         // token row of the tile (tensor-memory lane)
    const uint32_t tb = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + part * 32;
    for (int i = 0; i < n_my; ++i) {
      const uint32_t it = static_cast<uint32_t>(i);
      const UnitInfo t = unit_at(i);
      const bool sh = t.g < 0;
      const bool live = r < t.nlen;
      const int goff = t.goff;
      // down: this lane's output row (the receive row), looked up before the accumulator wait
      long long orow_down = -1;
      if (STAGE == 1 && live) {
        if (sh) {
          orow_down = t.n0 + r;
        } else {
          const int ci = goff + t.n0 + r;
          const long long row = (ci >= 0 && ci < a.tk) ? a.row_list[ci] : -1;
          orow_down = (row >= 0 && row < a.out_rows_routed) ? row : -1;
        }
      }
      if (!mbar_wait(acc_full, it & 1u, abort_flag, a.status)) break;
      tc_fence_after();
      if (STAGE == 0) {
        // h = silu(gate) * up for the warp's 32 columns, drained in two halves
        float h[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t g[16], v[16];
          tmem_ld16(tb + half * 16, g);
          tmem_ld16(tb + 128 + half * 16, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            h[half * 16 + j] = silu_fast(__uint_as_float(g[j])) * __uint_as_float(v[j]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty);
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(h[j]));
        // the 128-column block of h is split over the four warps of this lane quarter:
        // exchange their amax (slots alternate by unit parity)
        float* slot = amax_x + (((it & 1u) * 4 + quarter) * 32 + lane) * 4;
        slot[part] = amax;
        __syncwarp();
        if (lane == 0) mbar_arrive(&xbar[quarter]);
        if (!mbar_wait(&xbar[quarter], it & 1u, abort_flag, a.status)) break;
        amax = fmaxf(fmaxf(slot[0], slot[1]), fmaxf(slot[2], slot[3]));
        const float scale = pow2_block_scale(amax);
        if (live) {
          const long long orow = sh ? (long long)t.n0 + r : (long long)goff + t.n0 + r;
          const bool in = sh || (orow >= 0 && orow < a.tk);
          if (in) {
            uint8_t* out = static_cast<uint8_t*>(sh ? a.out_shared : a.out_routed) +
                           orow * (sh ? a.ld_shared : a.ld_routed) + t.m * 128 + part * 32;
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
              uint32_t w[4];
#pragma unroll
              for (int b = 0; b < 4; ++b) {
                const int j = qq * 16 + b * 4;
                const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
                    make_float2(__fdiv_rn(h[j], scale), __fdiv_rn(h[j + 1], scale)),
                    __NV_SATFINITE, __NV_E4M3);
                const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
                    make_float2(__fdiv_rn(h[j + 2], scale), __fdiv_rn(h[j + 3], scale)),
                    __NV_SATFINITE, __NV_E4M3);
                w[b] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
              }
              reinterpret_cast<uint4*>(out)[qq] = make_uint4(w[0], w[1], w[2], w[3]);
            }
            if (part == 0) {   // the row's scale byte for block m (its exponent field)
              uint8_t* osf = sh ? a.out_sf_shared : a.out_sf_routed;
              osf[orow * kSfRowBytes + t.m] =
                  static_cast<uint8_t>((__float_as_uint(scale) >> 23) & 0xFFu);
            }
          }
        }
      } else {
        // the unit's two 128-column output tiles: columns 32*part.. of each, packed to bf16 as
        // they are drained; the accumulator is released before any store is issued
        uint32_t pk[2][16];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t v0[16], v1[16];
          tmem_ld16(tb + h2 * 128, v0);
          tmem_ld16(tb + h2 * 128 + 16, v1);
          tmem_ld_wait();
          if (h2 == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            pk[h2][j] = pack_bf16x2(__uint_as_float(v0[2 * j]), __uint_as_float(v0[2 * j + 1]));
            pk[h2][8 + j] =
                pack_bf16x2(__uint_as_float(v1[2 * j]), __uint_as_float(v1[2 * j + 1]));
          }
        }
        if (live && orow_down >= 0) {
          __nv_bfloat16* orow_p = static_cast<__nv_bfloat16*>(sh ? a.out_shared : a.out_routed) +
                                  orow_down * (sh ? a.ld_shared : a.ld_routed) + t.m * 256 +
                                  part * 32;
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            uint4* out = reinterpret_cast<uint4*>(orow_p + h2 * 128);
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
              out[qq] = make_uint4(pk[h2][4 * qq], pk[h2][4 * qq + 1], pk[h2][4 * qq + 2],
                                   pk[h2][4 * qq + 3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

namespace {

// The gate/up GEMM's input scale bytes. Compact row c < n_routed takes the scales of its
// source row row_list[c] (a receive row, or a token in gather mode; -1 or out of range: none)
// from the block-major fp32 table xs [K/128][xs_ld]; token t < n_shared (the shared expert's
// input) those of x quantised, xq_sc [K/128][T]. A byte is the scale's exponent field; a scale
// that is not a positive normal power of two is reported (MOE_DEV_SCALE). Bytes past K/128,
// and the bytes of a row without a source, are 127 (scale 1).
__global__ void __launch_bounds__(256) mx8_scale_bytes_kernel(
    const int32_t* __restrict__ row_list, long long row_bound, const float* __restrict__ xs,
    long long xs_ld, const float* __restrict__ xq_sc, int T, int n_routed, int n_shared, int kb_n,
    uint8_t* __restrict__ sf_gu, uint8_t* __restrict__ sf_x, uint32_t* __restrict__ status) {
  pdl_wait();
  pdl_trigger();
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)n_routed + n_shared) return;
  const float* src;
  long long ld, row;
  uint8_t* dst;
  if (i < n_routed) {
    const long long r = row_list[i];
    row = (r >= 0 && r < row_bound) ? r : -1;
    src = xs;
    ld = xs_ld;
    dst = sf_gu + i * kSfRowBytes;
  } else {
    row = i - n_routed;
    src = xq_sc;
    ld = T;
    dst = sf_x + row * kSfRowBytes;
  }
  bool ok = true;
  uint32_t w[kSfRowBytes / 4];
#pragma unroll
  for (int j = 0; j < kSfRowBytes / 4; ++j) {
    uint32_t v = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int kb = 4 * j + b;
      const uint32_t byte = (row >= 0 && kb < kb_n) ? ue8m0_of(src[kb * ld + row], ok) : 127u;
      v |= byte << (8 * b);
    }
    w[j] = v;
  }
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int j = 0; j < kSfRowBytes / 16; ++j)
    d4[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  if (!ok) raise_status(status, MOE_DEV_SCALE);
}

}  // namespace

cudaError_t launch_ffn_gemm_mx8(const moe_cfg& c, const WsLayout& L, int stage, const void* recv,
                                const float* recv_scales, const moe_weights& w, void* ebuf,
                                void* shared_out, char* ws, cudaStream_t st, bool pdl,
                                const FfnPart& part) {
  const int cap = cap_of(c);
  const long long recv_rows = (long long)c.R * c.R * cap;
  const int F = c.d_ff, Fs = c.d_ff_shared, d = c.d, tk = c.T * c.k;
  const bool has_shared = Fs > 0;
  // gather mode: the gate/up stage reads routed token rows (and their scales) from x quantised
  // once per token, by token, through the schedule's token list
  const bool gather = part.src_tok != nullptr && stage == 0;
  if (d % 256) return cudaErrorNotSupported;
  if (recv_rows > 0x7fffffffLL) return cudaErrorNotSupported;   // 32-bit scale-row strides
  Mx8Args a{};
  a.tiles = reinterpret_cast<const Tile*>(ws + L.tiles);
  a.n_tiles = reinterpret_cast<const int32_t*>(ws + L.n_tiles);
  a.grp_off = reinterpret_cast<const int32_t*>(ws + L.grp_off);
  a.row_list = reinterpret_cast<const int32_t*>(ws + L.row_list);
  a.tk = tk;
  a.T = c.T;
  a.status = reinterpret_cast<uint32_t*>(ws + L.status);
  a.n_shared_tiles = has_shared ? (c.T + 127) / 128 : 0;
  a.out_rows_routed = recv_rows;
  a.group_expert = part.group_expert;
  const int n_w = part.weight_experts > 0 ? part.weight_experts : c.E;
  a.n_experts = n_w;
  CUtensorMap mA, mAs, mB, mBs;
  bool ok = true;
  if (stage == 0) {
    a.a_rows_routed = recv_rows;
    a.mt_routed = F / 128;
    a.mt_shared = has_shared ? Fs / 128 : 0;
    a.k_steps = d / 128;
    a.b_rows_routed = 2 * F;
    a.b_up_routed = F;
    a.b_up_shared = Fs;
    a.sf_routed = reinterpret_cast<const uint8_t*>(ws + L.sf_gu);
    a.sf_shared = reinterpret_cast<const uint8_t*>(ws + L.sf_x);
    a.w_sc_routed = w.w13_scales;
    a.w_sc_shared = w.ws13_scales;
    a.out_routed = ws + L.h;
    a.out_sf_routed = reinterpret_cast<uint8_t*>(ws + L.sf_h);
    a.out_shared = ws + L.hs;
    a.out_sf_shared = reinterpret_cast<uint8_t*>(ws + L.sf_hs);
    a.ld_routed = F;
    a.ld_shared = Fs;
    a.box_routed = 1;
    a.box_shared = c.T < 128 ? c.T : 128;
    a.gather_base = recv;
    a.gather_ld = d;
    if (gather) {
      a.row_list = reinterpret_cast<const int32_t*>(ws + L.tok_list);
      a.a_rows_routed = c.T;
      a.gather_base = ws + L.xq;
    }
    // (routed gate/up rows are gathered with cp.async; the map is a placeholder)
    ok &= make_tensor_map_2d(&mA, ws + L.xq, 1, d, c.T, 1);
    ok &= make_tensor_map_2d(&mB, w.w13, 1, d, (uint64_t)n_w * 2 * F, 128);
    if (has_shared) {
      ok &= make_tensor_map_2d(&mAs, ws + L.xq, 1, d, c.T, a.box_shared);
      ok &= make_tensor_map_2d(&mBs, w.ws13, 1, d, 2ull * Fs, 128);
    }
  } else {
    if (has_shared && Fs != F) return cudaErrorNotSupported;
    a.a_rows_routed = tk;
    a.mt_routed = d / 256;
    a.mt_shared = has_shared ? d / 256 : 0;
    a.k_steps = F / 128;
    a.b_rows_routed = d;
    a.b_up_routed = 128;
    a.b_up_shared = 128;
    a.sf_routed = reinterpret_cast<const uint8_t*>(ws + L.sf_h);
    a.sf_shared = reinterpret_cast<const uint8_t*>(ws + L.sf_hs);
    a.w_sc_routed = w.w2_scales;
    a.w_sc_shared = w.ws2_scales;
    a.out_routed = ebuf;
    a.out_shared = shared_out;
    a.ld_routed = d;
    a.ld_shared = d;
    a.box_routed = tk < 128 ? tk : 128;
    a.box_shared = c.T < 128 ? c.T : 128;
    ok &= make_tensor_map_2d(&mA, ws + L.h, 1, F, tk, a.box_routed);
    ok &= make_tensor_map_2d(&mB, w.w2, 1, F, (uint64_t)n_w * d, 128);
    if (has_shared) {
      ok &= make_tensor_map_2d(&mAs, ws + L.hs, 1, Fs, c.T, a.box_shared);
      ok &= make_tensor_map_2d(&mBs, w.ws2, 1, Fs, d, 128);
    }
  }
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
  const dim3 grid(part.ctas > 0 ? part.ctas : sm_count());
  if (stage == 0) {
    // the input rows' scale bytes first (routed rows of this launch, and the shared expert's)
    const int n_routed = a.mt_routed ? tk : 0;
    const int n_shared = a.mt_shared ? c.T : 0;
    if (n_routed + n_shared > 0) {
      const cudaError_t e = launch_kernel(
          mx8_scale_bytes_kernel, dim3((n_routed + n_shared + 255) / 256), dim3(256), 0, st, pdl,
          a.row_list, a.a_rows_routed, gather ? reinterpret_cast<const float*>(ws + L.xq_scales)
                                              : recv_scales,
          gather ? (long long)c.T : recv_rows,
          reinterpret_cast<const float*>(ws + L.xq_scales), c.T, n_routed, n_shared, d / 128,
          reinterpret_cast<uint8_t*>(ws + L.sf_gu), reinterpret_cast<uint8_t*>(ws + L.sf_x),
          a.status);
      if (e != cudaSuccess) return e;
      pdl = true;   // the GEMM follows the pre-pass
    }
    auto kern = ffn_gemm_mx8_kernel<0>;
    const cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(kern), kSmem);
    if (err != cudaSuccess) return err;
    return launch_kernel(kern, grid, dim3(kThreads), kSmem, st, pdl, a, mA, mAs, mB, mBs);
  }
  auto kern = ffn_gemm_mx8_kernel<1>;
  const cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(kern), kSmem);
  if (err != cudaSuccess) return err;
  return launch_kernel(kern, grid, dim3(kThreads), kSmem, st, pdl, a, mA, mAs, mB, mBs);
}

}  // namespace moe
