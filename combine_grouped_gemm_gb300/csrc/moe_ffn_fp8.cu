// e4m3 expert GEMMs with fp32 block scales (the FP8 prefill path).
//
// Method: as in moe_ffn.cu ("7.13 Serving Mixture-of-Experts", Expert Parallelism Mechanics,
// expert compute; "One-Sided Expert-Parallel All-to-All ...", abstract, grouped GEMMs reading
// the receive buffers in place), with DeepEP-style FP8 activations ("Serving
// Mixture-of-Experts", DeepEP section): activations carry one fp32 scale per token per 128
// columns, weights one fp32 scale per 128x128 block, and the SwiGLU intermediate is
// re-quantised the same way before the down projection.
//
// Because every 128-wide block of K carries its own pair of scales, the product of one block
// is accumulated alone in tensor memory (tcgen05.mma kind::f8f6f4, fp32 accumulate) and then
// "promoted": added into fp32 registers times (token scale x weight scale). To make that a
// single scalar per thread, this kernel is NOT swapped: the token rows are the M operand (128
// rows per tile, one tensor-memory lane each) and the weight rows the N operand (128 per
// tile), so the thread that owns lane j multiplies a whole partial row by one number.
// Two partial buffers in tensor memory alternate so the tensor core computes block kb+1 while
// the promoter warps read block kb.
//
// Roles (640 threads, one CTA per SM, persistent over the unit list):
//   warp 0       TMA producer (weight tiles; contiguous token rows as one box)
//   warp 1       tensor-memory allocation; lane 0 issues the MMAs
//   warps 2..17  promoters / epilogue: warp w owns lanes 32*(w%4).. and the column quarter
//                (w-2)/4 of each accumulator (32 columns of gate and of up)
//   warps 18,19  copy warps: per k-step the tile's 128 token scales and its weight scales into
//                a shared-memory scale ring, and (gate/up, routed units) the token rows
// Every global load of the k-step loop is issued by the producer or the copy warps, so the
// promoters' loop holds only barrier waits, shared-memory reads, tensor-memory loads and FMAs.
#include "moe_device.cuh"

namespace moe {
namespace {

struct Fp8Args {
  const Tile* tiles;
  const int32_t* n_tiles;
  const int32_t* grp_off;
  const int32_t* row_list;
  int tk;
  long long a_rows_routed;      // bound of routed A row indices
  int T;
  int mt_routed, mt_shared;     // weight tiles (units along N) per group
  int n_shared_tiles;
  int k_steps;                  // K / 128
  int b_rows_routed;            // weight rows per routed expert (2F or d)
  int b_up_routed, b_up_shared; // offset of a unit's second weight tile (gate/up: the up rows)
  // Token scales are block-major, [K/128][rows]: the scales of one K block for consecutive
  // rows are consecutive, so a warp's 32 rows read one or two cache lines per k-step.
  const float* a_sc_routed;     // token scales of routed A rows [K/128][a_sc_ld_routed]
  const float* a_sc_shared;     // token scales of shared A rows [K/128][T]
  int a_sc_ld_routed;           // rows per K block of a_sc_routed
  const float* w_sc_routed;     // [E][b_rows_routed/128][K/128]
  const float* w_sc_shared;     // [b_rows_shared/128][K/128]
  void* out_routed;             // gate/up: e4m3 h [tk][F]; down: bf16 ebuf [recv rows][d]
  float* out_sc_routed;         // gate/up: h scales, block-major [F/128][tk]
  void* out_shared;             // gate/up: e4m3 hs [T][Fs]; down: bf16 shared_out [T][d]
  float* out_sc_shared;         // gate/up: hs scales, block-major [Fs/128][T]
  int ld_routed, ld_shared;     // output row length (elements)
  long long out_rows_routed;    // bound of routed output row indices
  int box_routed, box_shared;   // rows per box of the contiguous token-row maps
  const uint8_t* gather_base;   // gate/up: receive buffer (routed token rows are gathered)
  long long gather_ld;          // bytes per receive row
  uint32_t* status;
  const int32_t* group_expert;  // expert whose weights group g uses (nullptr: expert g)
  int n_experts;                // experts in the weight tensors
};

// The expert whose weights a routed group reads (see the bf16 kernels): itself, or the expert
// its slot holds; an entry outside [0, n_experts) is reported and replaced by expert 0.
__device__ __forceinline__ int weight_expert8(const int32_t* group_expert, int g, int n_experts,
                                              uint32_t* status) {
  if (!group_expert) return g;
  const int e = group_expert[g];
  if (e >= 0 && e < n_experts) return e;
  raise_status(status, MOE_DEV_BOUNDS);
  return 0;
}

struct Unit8 {
  int g, n0, nlen, m;
};

__device__ __forceinline__ Unit8 decode_unit8(const Fp8Args& a, int u) {
  Unit8 r;
  const int us = a.n_shared_tiles * a.mt_shared;
  if (u < us) {
    const int tt = u / a.mt_shared;
    r.g = -1;
    r.m = u - tt * a.mt_shared;
    r.n0 = tt * 128;
    r.nlen = min(128, a.T - r.n0);
  } else {
    const int v = u - us;
    const int tt = v / a.mt_routed;
    r.m = v - tt * a.mt_routed;
    const Tile t = a.tiles[tt];
    r.g = t.group;
    r.n0 = t.n0;
    r.nlen = t.nlen;
  }
  return r;
}

constexpr int kPromoWarps = 16;                  // 4 per tensor-memory lane quarter
constexpr int kPromoThreads = kPromoWarps * 32;
// Copy warps: token scales and weight scales of every k-step, and (gate/up) the routed token
// rows, with cp.async.
constexpr int kGatherWarps = 2;
constexpr int kGatherThreads = kGatherWarps * 32;
template <int STAGE>
struct Fp8Threads {
  static constexpr int kGather = kGatherThreads;
  static constexpr int kAll = 64 + kPromoThreads + kGather;
};
// Scale ring: slot q % SLOTS holds k-step q's 128 token scales and its two weight scales (gate,
// up). It needs no barriers of its own:
//  - filled: the copy warps' cp.async arrivals on the stage's full barrier fire only after their
//    scale copies have landed; the MMA waits on that barrier before it commits the partial
//    buffer the promoters wait for;
//  - released: with SLOTS = STAGES + NBUF, a copy warp overwrites the slot of k-step q only
//    after the stage of k-step q + NBUF has been consumed by the MMA, which waited for the
//    promoters to release the partial buffer of k-step q (and so to finish reading its slot).
constexpr int kSlotFloats = 132;   // 128 token scales + 2 weight scales, padded to 16 bytes

// (a0, a1) += (x0, x1) * s as one packed fp32x2 fused multiply-add (two IEEE fmas).
__device__ __forceinline__ void ffma2(float& a0, float& a1, uint32_t x0, uint32_t x1, float s) {
  asm("{\n\t.reg .b64 d, x, w;\n\t"
      "mov.b64 d, {%0, %1};\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 w, {%4, %4};\n\t"
      "fma.rn.f32x2 d, x, w, d;\n\t"
      "mov.b64 {%0, %1}, d;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "r"(x0), "r"(x1), "f"(s));
}

__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
// The hardware arrives on bar once every cp.async this thread has issued so far has landed;
// the arrival counts as one of the barrier's expected arrivals.
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

template <int NB_, int STAGES>
struct Fp8Shape {
  // weight tiles per stage: gate/up 2 (gate, up); down 2 (two adjacent 128-column tiles of the
  // output) when d is a multiple of 256, else 1
  static constexpr int NB = NB_;
  static constexpr int A_BYTES = 128 * 128;          // 128 token rows x 128 e4m3
  static constexpr int B_BYTES = 128 * 128;          // 128 weight rows x 128 e4m3
  static constexpr int STAGE_BYTES = A_BYTES + NB * B_BYTES;
  static constexpr int ACC_COLS = NB * 128;          // partial accumulator columns per buffer
  // partial buffers: as many as tensor memory holds (2 for N = 256, 4 for N = 128), so the
  // tensor core can run that many K blocks ahead of the promoters
  static constexpr int NBUF = 512 / ACC_COLS;
  static constexpr int TMEM_COLS = NBUF * ACC_COLS;
  static constexpr int SLOTS = STAGES + NBUF;        // scale ring slots
  // stages + barriers (512 B) + amax exchange [2][4][32][4] floats (4 KB)
  // + scale ring [SLOTS][kSlotFloats] floats + alignment slack
  static constexpr int RING_OFF = STAGES * STAGE_BYTES + 512 + 4096;
  static constexpr int SMEM = RING_OFF + SLOTS * kSlotFloats * 4 + 1024;
  static_assert(TMEM_COLS <= 512, "tensor memory");
};

template <int STAGE, int NB, int STAGES>
__global__ void __launch_bounds__(Fp8Threads<STAGE>::kAll, 1)
    ffn_gemm_e4m3_kernel(const Fp8Args a, const __grid_constant__ CUtensorMap mapA,
                         const __grid_constant__ CUtensorMap mapAs,
                         const __grid_constant__ CUtensorMap mapB,
                         const __grid_constant__ CUtensorMap mapBs) {
  using S = Fp8Shape<NB, STAGES>;
  // weight rows between consecutive units' first tiles: gate/up 128 (a unit's second tile is
  // the up projection, F rows further); down NB x 128 (adjacent output tiles)
  constexpr int kStep = STAGE == 0 ? 128 : NB * 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * S::STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* pfull = empty + STAGES;    // [NBUF] partial buffer written
  uint64_t* pempty = pfull + S::NBUF;  // [NBUF] partial buffer read
  uint64_t* xbar = pempty + S::NBUF;   // [4] amax exchange of the warps on one lane quarter
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xbar + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* amax_x = reinterpret_cast<float*>(smem + STAGES * S::STAGE_BYTES + 512);  // [2][4][32][4]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      // the TMA lane's expect_tx arrival, plus one per copy thread
      mbar_init(&full[i], 1 + Fp8Threads<STAGE>::kGather);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < S::NBUF; ++i) {
      mbar_init(&pfull[i], 1);
      mbar_init(&pempty[i], kPromoWarps);   // one arrival per promoter warp
    }
    for (int i = 0; i < 4; ++i) mbar_init(&xbar[i], 4);   // the four warps of a lane quarter
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
  const int units = a.n_shared_tiles * a.mt_shared + (*a.n_tiles) * a.mt_routed;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    const uint64_t pol_w = l2_policy_evict_last();   // weight tiles are reused by token tiles
    const uint64_t pol_x = l2_policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const Unit8 t = decode_unit8(a, u);
      const bool sh = t.g < 0;
      const CUtensorMap* amap = sh ? &mapAs : &mapA;
      const CUtensorMap* bmap = sh ? &mapBs : &mapB;
      const int we = sh ? 0 : weight_expert8(a.group_expert, t.g, a.n_experts,
                                              lane == 0 ? a.status : nullptr);
      const int brow0 = (sh ? 0 : we * a.b_rows_routed) + t.m * kStep;
      const int brow1 = brow0 + (sh ? a.b_up_shared : a.b_up_routed);
      // Token rows: routed gate/up rows are gathered by the gather warps (cp.async); the shared
      // expert's rows (x, contiguous) and the down projection's rows (h, contiguous) are one
      // box per k-step.
      int box_row = -1;
      uint32_t a_bytes = 0;
      if (STAGE == 1 || sh) {
        const int row0 = sh ? t.n0 : a.grp_off[t.g] + t.n0;
        const bool in = row0 >= 0 && row0 < (sh ? a.T : a.tk);
        if (!in && lane == 0) raise_status(a.status, MOE_DEV_BOUNDS);
        box_row = in ? row0 : -1;
        a_bytes = in ? 128u * static_cast<uint32_t>(sh ? a.box_shared : a.box_routed) : 0u;
      }
      const uint32_t tx = S::NB * S::B_BYTES + a_bytes;
      for (int ks = 0; ks < a.k_steps; ++ks) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.status)) {
          ok = false;
          break;
        }
        uint8_t* sa = smem + stage * S::STAGE_BYTES;
        uint8_t* sb = sa + S::A_BYTES;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[stage], tx);
          tma_load_2d(sb, bmap, &full[stage], ks * 128, brow0, pol_w);
          if (S::NB == 2) tma_load_2d(sb + S::B_BYTES, bmap, &full[stage], ks * 128, brow1, pol_w);
          if (box_row >= 0) tma_load_2d(sa, amap, &full[stage], ks * 128, box_row, pol_x);
        }
        __syncwarp();
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
      // gate/up: the gate and up weight tiles sit back to back in shared memory, so one MMA
      // with N = 256 computes both (columns 0..127 gate, 128..255 up)
      const uint32_t idesc = idesc_e4m3(128, S::NB * 128);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t pk = 0;  // partial-buffer use counter
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        for (int ks = 0; ks < a.k_steps; ++ks, ++pk) {
          const uint32_t pb = pk % S::NBUF;
          if (!mbar_wait(&pempty[pb], ((pk / S::NBUF) & 1u) ^ 1u, abort_flag, a.status) ||
              !mbar_wait(&full[stage], phase, abort_flag, a.status)) {
            ok = false;
            break;
          }
          // gate/up: the gathered token rows were written by cp.async (generic proxy); the
          // fence orders them, observed through the barrier, before the MMA's reads
          if (STAGE == 0) fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t sa = smem_addr(smem + stage * S::STAGE_BYTES);
          const uint32_t sb = sa + S::A_BYTES;
          const uint32_t d0 = tmem + pb * S::ACC_COLS;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            mma_f8(d0, smem_desc_sw128(sa + kk * 32), smem_desc_sw128(sb + kk * 32), idesc, kk != 0);
          }
          mma_commit(&empty[stage]);
          mma_commit(&pfull[pb]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp >= 2 + kPromoWarps) {
    // ------------------------------ copy warps ------------------------------
    // Per k-step: the tile's 128 token scales (thread gt: rows gt and gt + 64) and the two
    // weight block scales (thread 0) into the scale ring, and, for routed gate/up units, the
    // token rows: thread gt copies 16-byte chunk j = gt % 8 of rows p = gt/8 + 8i (i < 16) into
    // the 128-byte-swizzled layout the MMA descriptor expects (chunk j of row p at chunk
    // j ^ (p % 8) = j ^ gt/8). Each thread then arms an arrival on the stage's full barrier,
    // which the hardware performs once its copies have landed. The MMA thread puts a proxy
    // fence between its wait and its tensor-core reads.
    const int gt = threadIdx.x - (64 + kPromoThreads);
    const int j = gt & 7, rg = gt >> 3;
    const uint32_t dst_off = static_cast<uint32_t>(rg * 128 + ((j ^ rg) << 4));
    float* sring = reinterpret_cast<float*>(smem + S::RING_OFF);
    const int kb_n = a.k_steps;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t q = 0;   // k-steps issued (scale ring position)
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const Unit8 t = decode_unit8(a, u);
      const bool sh = t.g < 0;
      const bool gather = STAGE == 0 && !sh;
      // receive row of each of the thread's 16 tile rows (-1: none), 32-bit to save registers
      int src[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int p = rg + 8 * i;
        src[i] = -1;
        if (gather && p < t.nlen) {
          const int ci = a.grp_off[t.g] + t.n0 + p;
          const long long row = (ci >= 0 && ci < a.tk) ? a.row_list[ci] : -1;
          if (row >= 0 && row < a.a_rows_routed) src[i] = static_cast<int>(row);
          else raise_status(a.status, MOE_DEV_BOUNDS);
        }
      }
      // scale rows of tile rows gt and gt + 64 (-1: past the tile's rows)
      long long srow[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int p = gt + 64 * h;
        srow[h] = -1;
        if (p < t.nlen) {
          long long row;
          if (sh) {
            row = t.n0 + p;
          } else {
            const int ci = a.grp_off[t.g] + t.n0 + p;
            row = ci;   // down: compact row of h
            if (STAGE == 0) row = (ci >= 0 && ci < a.tk) ? a.row_list[ci] : -1;
          }
          const long long bound = sh ? a.T : (STAGE == 0 ? a.a_rows_routed : a.tk);
          if (row >= 0 && row < bound) srow[h] = row;
          else raise_status(a.status, MOE_DEV_BOUNDS);
        }
      }
      const float* xs = sh ? a.a_sc_shared : a.a_sc_routed;
      const long long xs_ld = sh ? a.T : a.a_sc_ld_routed;
      const int we = sh ? 0 : weight_expert8(a.group_expert, t.g, a.n_experts, nullptr);
      const float* wsc = (sh ? a.w_sc_shared
                             : a.w_sc_routed + (size_t)we * (a.b_rows_routed / 128) * kb_n) +
                         (size_t)t.m * (kStep / 128) * kb_n;
      const int w_up = (sh ? a.b_up_shared : a.b_up_routed) / 128 * kb_n;
      const uint8_t* gsrc = a.gather_base + j * 16;
      for (int ks = 0; ks < kb_n; ++ks, ++q) {
        const uint32_t slot = q % S::SLOTS;
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.status)) {
          ok = false;
          break;
        }
        if (gather) {
          const uint32_t sa = smem_addr(smem + stage * S::STAGE_BYTES) + dst_off;
          const uint8_t* gk = gsrc + ks * 128;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if (src[i] >= 0)
              asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa + i * 1024),
                           "l"(gk + (long long)src[i] * a.gather_ld)
                           : "memory");
        }
        float* sl = sring + slot * kSlotFloats;
#pragma unroll
        for (int h = 0; h < 2; ++h)
          if (srow[h] >= 0) cp_async4(sl + gt + 64 * h, xs + ks * xs_ld + srow[h]);
        if (gt == 0) {
          cp_async4(sl + 128, wsc + ks);
          if (S::NB == 2) cp_async4(sl + 129, wsc + w_up + ks);
        }
        // counts as one of the barrier's expected arrivals (a thread with nothing to copy
        // arrives as soon as its earlier copies have landed)
        cp_async_arrive(&full[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // after an abort: copies still in flight land before the CTA exits
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else {
    // ------------------------------ promoters / epilogue ------------------------------
    const int quarter = warp & 3;
    const int part = (warp - 2) >> 2;      // columns 32*part .. 32*part+31 of each accumulator
    const int r = quarter * 32 + lane;     // token row of the tile (tensor-memory lane)
    const int kb_n = a.k_steps;
    const float* sring = reinterpret_cast<const float*>(smem + S::RING_OFF);
    uint32_t pk = 0;   // k-steps consumed (partial-buffer and scale-ring position)
    uint32_t it = 0;
    // The schedule entry of the next unit and its group's row offset are loaded one unit ahead,
    // so these dependent global loads overlap a unit's k-steps instead of starting the next.
    Unit8 tn{0, 0, 0, 0};
    int goff_n = 0;
    if (blockIdx.x < units) {
      tn = decode_unit8(a, blockIdx.x);
      goff_n = tn.g >= 0 ? a.grp_off[tn.g] : 0;
    }
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++it) {
      const Unit8 t = tn;
      const int goff = goff_n;
      const int un = u + gridDim.x;
      if (un < units) tn = decode_unit8(a, un);
      const bool sh = t.g < 0;
      const bool live = r < t.nlen;
      // down: this lane's output row (the receive row), loaded now and used in the epilogue
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
      float acc0[32], acc1[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) acc0[j] = acc1[j] = 0.0f;
      bool ok = true;
      for (int ks = 0; ks < kb_n; ++ks, ++pk) {
        const uint32_t pb = pk % S::NBUF;
        if (!mbar_wait(&pfull[pb], (pk / S::NBUF) & 1u, abort_flag, a.status)) {
          ok = false;
          break;
        }
        // the k-step's scales (filled before the stage's full barrier fired; see the ring)
        const float* sl = sring + (pk % S::SLOTS) * kSlotFloats;
        const float xsv = sl[r];
        const float s0 = xsv * sl[128];
        const float s1 = S::NB == 2 ? xsv * sl[129] : 0.0f;
        tc_fence_after();
        const uint32_t tb = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + pb * S::ACC_COLS +
                            part * 32;
        // two tensor-memory loads in flight per wait: the gate columns, then the up columns;
        // packed fp32x2 FMAs
        {
          uint32_t v0[16], v1[16];
          tmem_ld16(tb, v0);
          tmem_ld16(tb + 16, v1);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            ffma2(acc0[j], acc0[j + 1], v0[j], v0[j + 1], s0);
            ffma2(acc0[16 + j], acc0[17 + j], v1[j], v1[j + 1], s0);
          }
        }
        if (S::NB == 2) {
          uint32_t v0[16], v1[16];
          tmem_ld16(tb + 128, v0);
          tmem_ld16(tb + 144, v1);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            ffma2(acc1[j], acc1[j + 1], v0[j], v0[j + 1], s1);
            ffma2(acc1[16 + j], acc1[17 + j], v1[j], v1[j + 1], s1);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pempty[pb]);
      }
      if (!ok) break;
      if (un < units) goff_n = tn.g >= 0 ? a.grp_off[tn.g] : 0;   // used at the next unit

      // ---- epilogue of the unit ----
      if (STAGE == 0) {
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          acc0[j] = silu_fast(acc0[j]) * acc1[j];
          amax = fmaxf(amax, fabsf(acc0[j]));
        }
        // the 128-column block of h is split over the four warps of this lane quarter:
        // exchange their amax (slots alternate by unit parity so a fast warp's next write never
        // meets a partner's pending read)
        float* slot = amax_x + (((it & 1u) * 4 + quarter) * 32 + lane) * 4;
        slot[part] = amax;
        __syncwarp();
        if (lane == 0) mbar_arrive(&xbar[quarter]);
        if (!mbar_wait(&xbar[quarter], it & 1u, abort_flag, a.status)) break;
        amax = fmaxf(fmaxf(slot[0], slot[1]), fmaxf(slot[2], slot[3]));
        const float scale = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
        if (live) {
          long long orow = sh ? (long long)t.n0 + r : (long long)goff + t.n0 + r;
          const bool in = sh || (orow >= 0 && orow < a.tk);
          if (in) {
            uint8_t* out = static_cast<uint8_t*>(sh ? a.out_shared : a.out_routed) +
                           orow * (sh ? a.ld_shared : a.ld_routed) + t.m * 128 + part * 32;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              uint32_t w[4];
#pragma unroll
              for (int b = 0; b < 4; ++b) {
                const int j = q * 16 + b * 4;
                const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
                    make_float2(__fdiv_rn(acc0[j], scale), __fdiv_rn(acc0[j + 1], scale)),
                    __NV_SATFINITE, __NV_E4M3);
                const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
                    make_float2(__fdiv_rn(acc0[j + 2], scale), __fdiv_rn(acc0[j + 3], scale)),
                    __NV_SATFINITE, __NV_E4M3);
                w[b] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
              }
              reinterpret_cast<uint4*>(out)[q] = make_uint4(w[0], w[1], w[2], w[3]);
            }
            if (part == 0) {   // block-major: consecutive lanes write consecutive rows
              float* osc = sh ? a.out_sc_shared : a.out_sc_routed;
              osc[(long long)t.m * (sh ? a.T : a.tk) + orow] = scale;
            }
          }
        }
      } else if (live) {
        const long long orow = orow_down;
        if (orow >= 0) {
          __nv_bfloat16* orow_p = static_cast<__nv_bfloat16*>(sh ? a.out_shared : a.out_routed) +
                                  orow * (sh ? a.ld_shared : a.ld_routed) + t.m * (NB * 128) +
                                  part * 32;
#pragma unroll
          for (int h = 0; h < NB; ++h) {   // the unit's first and (NB = 2) second 128 columns
            const float* acc = h ? acc1 : acc0;
            uint4* out = reinterpret_cast<uint4*>(orow_p + h * 128);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int j = q * 8;
              out[q] = make_uint4(pack_bf16x2(acc[j], acc[j + 1]), pack_bf16x2(acc[j + 2], acc[j + 3]),
                                  pack_bf16x2(acc[j + 4], acc[j + 5]), pack_bf16x2(acc[j + 6], acc[j + 7]));
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, S::TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_ffn_gemm_e4m3(const moe_cfg& c, const WsLayout& L, int stage, const void* recv,
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
  Fp8Args a{};
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
  if (recv_rows > 0x7fffffffLL) return cudaErrorNotSupported;   // 32-bit scale-row strides
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
    a.a_sc_routed = recv_scales;
    a.a_sc_ld_routed = static_cast<int>(recv_rows);
    a.a_sc_shared = reinterpret_cast<const float*>(ws + L.xq_scales);
    a.w_sc_routed = w.w13_scales;
    a.w_sc_shared = w.ws13_scales;
    a.out_routed = ws + L.h;
    a.out_sc_routed = reinterpret_cast<float*>(ws + L.h_scales);
    a.out_shared = ws + L.hs;
    a.out_sc_shared = reinterpret_cast<float*>(ws + L.hs_scales);
    a.ld_routed = F;
    a.ld_shared = Fs;
    a.gather_base = static_cast<const uint8_t*>(recv);
    a.gather_ld = d;
    a.box_routed = 1;
    a.box_shared = c.T < 128 ? c.T : 128;
    if (gather) {
      a.row_list = reinterpret_cast<const int32_t*>(ws + L.tok_list);
      a.a_rows_routed = c.T;
      a.a_sc_routed = reinterpret_cast<const float*>(ws + L.xq_scales);
      a.a_sc_ld_routed = c.T;
      a.gather_base = reinterpret_cast<const uint8_t*>(ws + L.xq);
    }
    ok &= make_tensor_map_2d(&mA, gather ? static_cast<const void*>(ws + L.xq) : recv, 1, d,
                             gather ? c.T : recv_rows, 1);
    ok &= make_tensor_map_2d(&mB, w.w13, 1, d, (uint64_t)n_w * 2 * F, 128);
    if (has_shared) {
      ok &= make_tensor_map_2d(&mAs, ws + L.xq, 1, d, c.T, a.box_shared);
      ok &= make_tensor_map_2d(&mBs, w.ws13, 1, d, 2ull * Fs, 128);
    }
  } else {
    if (has_shared && Fs != F) return cudaErrorNotSupported;
    const int nb = d % 256 == 0 ? 2 : 1;   // output columns per unit: nb x 128
    a.a_rows_routed = tk;
    a.mt_routed = d / (nb * 128);
    a.mt_shared = has_shared ? d / (nb * 128) : 0;
    a.k_steps = F / 128;
    a.b_rows_routed = d;
    a.b_up_routed = nb == 2 ? 128 : 0;
    a.b_up_shared = nb == 2 ? 128 : 0;
    a.a_sc_routed = reinterpret_cast<const float*>(ws + L.h_scales);
    a.a_sc_ld_routed = tk;
    a.a_sc_shared = reinterpret_cast<const float*>(ws + L.hs_scales);
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
  cudaError_t err;
  if (stage == 0) {
    using S = Fp8Shape<2, 4>;
    auto kern = ffn_gemm_e4m3_kernel<0, 2, 4>;
    err = ensure_smem_limit(reinterpret_cast<const void*>(kern), S::SMEM);
    if (err != cudaSuccess) return err;
    return launch_kernel(kern, grid, dim3(Fp8Threads<0>::kAll), S::SMEM, st, pdl, a, mA, mAs,
                         mB, mBs);
  } else if (d % 256 == 0) {
    using S = Fp8Shape<2, 4>;
    auto kern = ffn_gemm_e4m3_kernel<1, 2, 4>;
    err = ensure_smem_limit(reinterpret_cast<const void*>(kern), S::SMEM);
    if (err != cudaSuccess) return err;
    return launch_kernel(kern, grid, dim3(Fp8Threads<1>::kAll), S::SMEM, st, pdl, a, mA, mAs,
                         mB, mBs);
  } else {
    using S = Fp8Shape<1, 6>;
    auto kern = ffn_gemm_e4m3_kernel<1, 1, 6>;
    err = ensure_smem_limit(reinterpret_cast<const void*>(kern), S::SMEM);
    if (err != cudaSuccess) return err;
    return launch_kernel(kern, grid, dim3(Fp8Threads<1>::kAll), S::SMEM, st, pdl, a, mA, mAs,
                         mB, mBs);
  }
}

}  // namespace moe
