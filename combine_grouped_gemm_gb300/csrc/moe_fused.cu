// The expert stage and the combine in one persistent launch (bf16): gate/up GEMM -> down GEMM
// -> weighted combine, with device-side dependency counters instead of kernel boundaries.
//
// Method: "DeepSeek MoE Serving: Where Expert-Parallel All-to-All Time Goes" (groundy), the
// table of regimes and the paragraph after it: a fused MoE kernel (DeepGEMM's MegaMoE) runs
// dispatch, both grouped GEMMs and combine in one launch and wins from a few hundred tokens
// per rank; "One-Sided Expert-Parallel All-to-All ..." (abstract) weighs it against separate
// kernels at decode. Here, on one GPU, the dispatch copy is already gone in gather mode (the
// gate/up GEMM reads x in place), so the launch covers the rest of the layer after the router,
// the dispatch index and the schedule.
//
// Why it pays on one GPU: the unit lists of the two GEMMs do not divide evenly over the SMs
// (the decode layer's gate/up stage is about 14.3 waves of units at 64 tokens, 6.1 at 8), so
// with one launch per stage most SMs idle through the last wave before the down stage can
// start. Here a CTA that runs out of gate/up units takes down units at once; each down unit
// waits only for the gate/up units of its own token tile.
//
// Unit list: the gate/up units (shared-expert tiles first, token-tile-major),
// then the down units (weight-tile-major within a group); CTA c takes units c, c + grid, ...
// so every CTA finishes its gate/up units before its down units. A down unit's producer waits
// until the four epilogue warps of every gate/up unit of that token tile have published their
// rows of h (a release add per warp, an acquire load in a bounded loop), then fences the
// generic proxy before its TMA loads of h. After the GEMM loops every thread of the CTA joins
// the combine, once every down unit has published its rows.
//
// Deadlock freedom: the launch is cooperative (every CTA resident at once); gate/up units wait
// on nothing but their own pipeline; a down unit depends only on gate/up units, all of which
// come earlier in every CTA's order, and a producer waiting on its own CTA's last gate/up unit
// does not block that unit (its loads are already issued). Every wait is bounded by the global
// timer (MOE_DEV_TIMEOUT, then the CTA leaves).
#include "moe_gemm.cuh"

namespace moe {
namespace {

struct CombineArgs {
  const int32_t* row_of;
  const float* topk_w;
  const uint4* ebuf;
  const uint4* shared_out;   // nullptr: no shared expert
  uint4* y;
  int d, k, T, nslice, slice_vecs;
  long long recv_rows;
};

struct FusedArgs {
  GemmArgs gu;               // gate/up stage
  GemmArgs dn;               // down stage
  int32_t* done_tile;        // [max_tiles]: gate/up epilogue warps finished per routed tile
  int32_t* done_shared;      // [shared tiles]: the same for the shared expert's token tiles
  int32_t* done_down;        // [1]: down epilogue warps finished
  int32_t* done_up;          // [1]: gate/up epilogue warps finished, all tiles together
  CombineArgs cb;
};

struct FUnit {
  int stage;   // 0 gate/up, 1 down
  Unit t;
  int tile;    // routed: index in the tile list; shared: the shared expert's token tile
};

template <int BN>
__device__ __forceinline__ FUnit decode_fused(const FusedArgs& f, int u, int n_tiles, int U0) {
  FUnit r;
  if (u < U0) {
    r.stage = 0;
    r.t = decode_unit<BN, false>(f.gu, u, n_tiles);
  } else {
    r.stage = 1;
    r.t = decode_unit<BN, true>(f.dn, u - U0, n_tiles);
  }
  r.tile = r.t.ti;
  return r;
}

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(int32_t* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Waits until *p >= target. Bounded like every wait here: false (after setting *abort and the
// status bit) when it outlives kWaitLimitNs, or at once when the CTA is aborting.
__device__ __forceinline__ bool wait_count(const int32_t* p, int target, volatile int* abort,
                                           uint32_t* status) {
  if (ld_acquire(p) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    __nanosleep(64);
    if (ld_acquire(p) >= target) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      raise_status(status, MOE_DEV_TIMEOUT);
      return false;
    }
  }
}

// Shared memory: the gate/up stages (two weight tiles and a token tile each) and, over the same
// bytes, the down stages (one weight tile and a token tile: more of them, so the down phase
// keeps as many bytes in flight as the down kernel does). A CTA's producer moves to the down
// ring once, after its last gate/up stage has been consumed.
template <int BN, int STAGES, int STAGES2>
struct FusedShape {
  using G = GemmShape<0, BN, STAGES>;
  static constexpr int STAGE2_BYTES = G::A_BYTES + G::B_BYTES;
  static_assert(STAGE2_BYTES % 1024 == 0, "down stages stay 1024-byte aligned");
  static_assert(STAGES2 * STAGE2_BYTES <= STAGES * G::STAGE_BYTES, "down ring inside the ring");
  static_assert((2 * STAGES + 2 * STAGES2 + 4) * 8 + 8 <= 256, "barriers in the reserved bytes");
};

template <int BN, int STAGES, int STAGES2>
__global__ void __launch_bounds__(GemmThreads<0>::kAll, 1)
    ffn_fused_bf16_kernel(const __grid_constant__ FusedArgs f, const __grid_constant__ CUtensorMap gA,
                          const __grid_constant__ CUtensorMap gAs,
                          const __grid_constant__ CUtensorMap gB,
                          const __grid_constant__ CUtensorMap gBs,
                          const __grid_constant__ CUtensorMap dA,
                          const __grid_constant__ CUtensorMap dAs,
                          const __grid_constant__ CUtensorMap dB,
                          const __grid_constant__ CUtensorMap dBs) {
  // stages laid out for gate/up (two weight tiles); a down unit uses the first weight slot
  using S = GemmShape<0, BN, STAGES>;
  constexpr int S2B = FusedShape<BN, STAGES, STAGES2>::STAGE2_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * S::STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* full2 = empty + STAGES;     // the down ring
  uint64_t* empty2 = full2 + STAGES2;
  uint64_t* tfull = empty2 + STAGES2;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint32_t* status = f.gu.status;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1 + GemmThreads<0>::kGather);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < STAGES2; ++i) {
      mbar_init(&full2[i], 1);   // the producer's arrival only: nothing is gathered for down
      mbar_init(&empty2[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 4);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&gA);
    tma_prefetch_map(&gB);
    tma_prefetch_map(&dA);
    tma_prefetch_map(&dB);
    if (f.gu.mt_shared) {
      tma_prefetch_map(&gAs);
      tma_prefetch_map(&gBs);
      tma_prefetch_map(&dAs);
      tma_prefetch_map(&dBs);
    }
  }
  pdl_wait();
  if (warp == 1) {
    tmem_alloc(tmem_slot, S::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int n_tiles = *f.gu.n_tiles;
  const int U0 = f.gu.n_shared_tiles * f.gu.mt_shared + n_tiles * f.gu.mt_routed;
  const int U1 = f.dn.n_shared_tiles * f.dn.mt_shared + n_tiles * f.dn.mt_routed;
  const int units = U0 + U1;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    const uint64_t pol_w1 = l2_policy_evict_first();
    const uint64_t pol_wk = l2_policy_evict_last();
    const uint64_t pol_x = l2_policy_evict_last();
    int stage = 0, stage2 = 0;
    uint32_t phase = 0, phase2 = 0;
    bool ok = true, on_ring2 = false;
    bool all_up = false;   // seen every gate/up unit finish: no more waits or fences needed
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const FUnit fu = decode_fused<BN>(f, u, n_tiles, U0);
      const bool up = fu.stage == 0;
      if (!up && !on_ring2) {
        // the down ring overlays the gate/up stages: wait until every one of them has been
        // consumed (the waits this warp would make before refilling each)
        for (int i = 0; i < STAGES && ok; ++i) {
          const int sl = (stage + i) % STAGES;
          const uint32_t ph = stage + i >= STAGES ? phase ^ 1u : phase;
          ok = mbar_wait(&empty[sl], ph ^ 1u, abort_flag, status);
        }
        on_ring2 = true;
        if (!ok) break;
      }
      const GemmArgs& a = up ? f.gu : f.dn;
      const Unit& t = fu.t;
      const bool sh = t.g < 0;
      const uint64_t pol_w = weight_policy(t, pol_w1, pol_wk);
      const CUtensorMap* amap = up ? (sh ? &gAs : &gA) : (sh ? &dAs : &dA);
      const CUtensorMap* bmap = up ? (sh ? &gBs : &gB) : (sh ? &dBs : &dB);
      const int we = sh ? 0 : weight_expert(a.group_expert, t.g, a.n_experts,
                                             lane == 0 ? a.status : nullptr);
      const int arow0 = (sh ? 0 : we * a.a_rows_routed) + t.m * 128;
      const int arow1 = arow0 + (sh ? a.a_up_shared : a.a_up_routed);
      int box_row = -1;
      uint32_t b_bytes = 0;
      int g4[4] = {-1, -1, -1, -1};
      bool g4_on = false;
      if (up && !sh && t.nlen <= kSmallTile) {
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
      if (!up || sh) {
        const int row0 = sh ? t.n0 : a.grp_off[t.g] + t.n0;
        const bool in = row0 >= 0 && row0 < (sh ? a.T : a.tk);
        if (!in && lane == 0) raise_status(a.status, MOE_DEV_BOUNDS);
        box_row = in ? row0 : -1;
        b_bytes = in ? 128u * static_cast<uint32_t>(sh ? a.box_shared : a.box_routed) : 0u;
      }
      if (!up && !all_up) {
        // this token tile's intermediate h must be complete: every gate/up unit of the tile
        // (mt of them, four epilogue warps each) has published its rows. Once every gate/up
        // unit of the launch has (one counter), all of h is there and the remaining down units
        // go without a check.
        int done = 1;
        if (lane == 0) {
          if (ld_acquire(f.done_up) >= 4 * U0) {
            all_up = true;
          } else {
            const int32_t* cnt = sh ? f.done_shared + fu.tile : f.done_tile + fu.tile;
            const int target = 4 * (sh ? f.gu.mt_shared : f.gu.mt_routed);
            done = wait_count(cnt, target, abort_flag, status) ? 1 : 0;
          }
          // the rows were written through the generic proxy; the TMA reads them through the
          // async proxy
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        all_up = __shfl_sync(0xffffffffu, all_up ? 1 : 0, 0) != 0;
        if (!__shfl_sync(0xffffffffu, done, 0)) {
          ok = false;
          break;
        }
      }
      const uint32_t tx = (up ? 2 : 1) * S::A_BYTES + b_bytes;
      for (int ks = 0; ks < a.k_steps; ++ks) {
        uint64_t* fb = up ? &full[stage] : &full2[stage2];
        if (!mbar_wait(up ? &empty[stage] : &empty2[stage2], (up ? phase : phase2) ^ 1u,
                       abort_flag, status)) {
          ok = false;
          break;
        }
        uint8_t* sa = up ? smem + stage * S::STAGE_BYTES : smem + stage2 * S2B;
        uint8_t* sb = sa + (up ? 2 : 1) * S::A_BYTES;
        if (lane == 0) {
          mbar_arrive_expect_tx(fb, tx);
          tma_load_2d(sa, amap, fb, ks * 64, arow0, pol_w);
          if (up) tma_load_2d(sa + S::A_BYTES, amap, fb, ks * 64, arow1, pol_w);
          if (box_row >= 0) tma_load_2d(sb, bmap, fb, ks * 64, box_row, pol_x);
        }
        __syncwarp();
        if (g4_on)
          tma_gather4(sb + lane * 512, bmap, fb, ks * 64, g4[0], g4[1], g4[2], g4[3], pol_x);
        if (up) {
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        } else if (++stage2 == STAGES2) {
          stage2 = 0;
          phase2 ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      int stage = 0, stage2 = 0;
      uint32_t phase = 0, phase2 = 0;
      bool ok = true;
      int it = 0;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++it) {
        const FUnit fu = decode_fused<BN>(f, u, n_tiles, U0);
        const bool up = fu.stage == 0;
        const int k_steps = up ? f.gu.k_steps : f.dn.k_steps;
        const uint32_t n_pad = static_cast<uint32_t>(max(16, (fu.t.nlen + 15) & ~15));
        const uint32_t idesc = idesc_bf16(128, n_pad);
        const int b = it & 1;
        if (!mbar_wait(&tempty[b], ((it >> 1) & 1) ^ 1u, abort_flag, status)) break;
        tc_fence_after();
        const uint32_t d0 = tmem + b * S::ACC_COLS;
        const uint32_t d1 = d0 + BN;
        for (int ks = 0; ks < k_steps; ++ks) {
          if (!mbar_wait(up ? &full[stage] : &full2[stage2], up ? phase : phase2, abort_flag,
                         status)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();   // gathered rows written by cp.async (gate/up)
          tc_fence_after();
          const uint32_t sa = smem_addr(up ? smem + stage * S::STAGE_BYTES : smem + stage2 * S2B);
          const uint32_t sb = sa + (up ? 2 : 1) * S::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t db = smem_desc_sw128(sb + kk * 32);
            const uint32_t acc = (ks | kk) != 0;
            mma_f16(d0, smem_desc_sw128(sa + kk * 32), db, idesc, acc);
            if (up) mma_f16(d1, smem_desc_sw128(sa + S::A_BYTES + kk * 32), db, idesc, acc);
          }
          if (up) {
            mma_commit(&empty[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          } else {
            mma_commit(&empty2[stage2]);
            if (++stage2 == STAGES2) {
              stage2 = 0;
              phase2 ^= 1u;
            }
          }
        }
        if (ok) mma_commit(&tfull[b]);
      }
    }
    __syncwarp();
  } else if (warp >= 6) {
    // ------------------------------ token-row gather (gate/up) ------------------------------
    // as in the gate/up kernel; on the gate/up units with nothing to gather these threads only
    // arrive once per k-step
    constexpr int kRowsPer = BN / 8;
    const int gt = threadIdx.x - 192;
    const int j = gt & 7, rg = gt >> 3;
    const uint32_t dst_off = static_cast<uint32_t>(rg * 128 + ((j ^ rg) << 4));
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    // gate/up units only: every down unit comes after them, and the down ring's barriers
    // expect no arrival from these warps
    for (int u = blockIdx.x; u < U0 && ok; u += gridDim.x) {
      const FUnit fu = decode_fused<BN>(f, u, n_tiles, U0);
      const bool up = true;
      const GemmArgs& a = f.gu;
      const Unit& t = fu.t;
      const bool gather = t.g >= 0 && t.nlen > kSmallTile;
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
      (void)up;
      for (int ks = 0; ks < a.k_steps; ++ks) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, status)) {
          ok = false;
          break;
        }
        const uint32_t sb = smem_addr(smem + stage * S::STAGE_BYTES + 2 * S::A_BYTES) + dst_off;
        if (gather) {
#pragma unroll
          for (int i = 0; i < kRowsPer; ++i)
            if (src[i])
              asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sb + i * 1024),
                           "l"(src[i] + ks * 128)
                           : "memory");
        }
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(
                         smem_addr(&full[stage]))
                     : "memory");
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else {
    // ------------------------------ epilogue ------------------------------
    const int quarter = warp & 3;
    const int rrow = quarter * 32 + lane;
    int it = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++it) {
      const FUnit fu = decode_fused<BN>(f, u, n_tiles, U0);
      const bool up = fu.stage == 0;
      const GemmArgs& a = up ? f.gu : f.dn;
      const Unit& t = fu.t;
      const bool sh = t.g < 0;
      const int b = it & 1;
      if (!mbar_wait(&tfull[b], (it >> 1) & 1, abort_flag, status)) break;
      tc_fence_after();
      const uint32_t tb = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + b * S::ACC_COLS;
      const int fcol = t.m * 128 + rrow;
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(sh ? a.out_shared : a.out_routed);
      const int ld = sh ? a.ld_shared : a.ld_routed;
      long long orows[BN / 32];
      const int base = sh ? 0 : a.grp_off[t.g];
#pragma unroll
      for (int i = 0; i < BN / 32; ++i) {
        const int p = lane + 32 * i;
        long long o = -1;
        if (p < t.nlen) {
          if (sh) {
            o = t.n0 + p;
          } else if (up) {
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
        if (up) tmem_ld16(tb + BN + c0, rb);
        tmem_ld_wait();
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int p = c0 + jj;
          const long long orow = __shfl_sync(0xffffffffu, orows[(c0 >> 5) & (BN / 32 - 1)], p & 31);
          if (p >= t.nlen || orow < 0) continue;
          const float val = up ? silu(__uint_as_float(ra[jj])) * __uint_as_float(rb[jj])
                               : __uint_as_float(ra[jj]);
          out[orow * ld + fcol] = __float2bfloat16_rn(val);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&tempty[b]);
        // publish this warp's rows: the token tile's h (gate/up) or the output rows (down)
        int32_t* cnt = !up ? f.done_down : (sh ? f.done_shared + fu.tile : f.done_tile + fu.tile);
        red_release_add(cnt, 1);
        if (up) red_release_add(f.done_up, 1);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, S::TMEM_COLS);
  }

  // ------------------------------ combine ------------------------------
  // y[t] = bf16(sum_i w_i * ebuf[row_of[t][i]] + shared_out[t]) in fp32 in selection order,
  // the combine kernel's arithmetic, once every down unit has published its rows. The expert
  // outputs were written by other SMs during this launch, so they are read through L2 (.cg).
  __shared__ int go;
  if (threadIdx.x == 0)
    go = (!*abort_flag && wait_count(f.done_down, 4 * U1, abort_flag, status)) ? 1 : 0;
  __syncthreads();
  if (!go) return;
  const CombineArgs& cb = f.cb;
  __shared__ int32_t rows[32];
  __shared__ float wts[32];
  const int vpr = cb.d / 8;
  for (int cu = blockIdx.x; cu < cb.T * cb.nslice; cu += gridDim.x) {
    const int t = cu / cb.nslice, sl = cu - t * cb.nslice;
    __syncthreads();
    if (threadIdx.x < cb.k) {
      int row = cb.row_of[(size_t)t * cb.k + threadIdx.x];
      if (row >= cb.recv_rows) {
        if (sl == 0) raise_status(status, MOE_DEV_BOUNDS);
        row = -1;
      }
      rows[threadIdx.x] = row;
      wts[threadIdx.x] = cb.topk_w[(size_t)t * cb.k + threadIdx.x];
    }
    __syncthreads();
    const int v0 = sl * cb.slice_vecs, v1 = min(vpr, v0 + cb.slice_vecs);
    for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
      float acc[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) acc[jj] = 0.0f;
      for (int i0 = 0; i0 < cb.k; i0 += 8) {
        uint4 e[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int row = (i0 + q < cb.k) ? rows[i0 + q] : -1;
          e[q] = row >= 0 ? __ldcg(cb.ebuf + (size_t)row * vpr + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (i0 + q >= cb.k || rows[i0 + q] < 0) continue;
          const float w = wts[i0 + q];
          acc[0] = __fmaf_rn(w, bf16_lo(e[q].x), acc[0]);
          acc[1] = __fmaf_rn(w, bf16_hi(e[q].x), acc[1]);
          acc[2] = __fmaf_rn(w, bf16_lo(e[q].y), acc[2]);
          acc[3] = __fmaf_rn(w, bf16_hi(e[q].y), acc[3]);
          acc[4] = __fmaf_rn(w, bf16_lo(e[q].z), acc[4]);
          acc[5] = __fmaf_rn(w, bf16_hi(e[q].z), acc[5]);
          acc[6] = __fmaf_rn(w, bf16_lo(e[q].w), acc[6]);
          acc[7] = __fmaf_rn(w, bf16_hi(e[q].w), acc[7]);
        }
      }
      if (cb.shared_out) {
        const uint4 s = __ldcg(cb.shared_out + (size_t)t * vpr + v);
        acc[0] += bf16_lo(s.x);
        acc[1] += bf16_hi(s.x);
        acc[2] += bf16_lo(s.y);
        acc[3] += bf16_hi(s.y);
        acc[4] += bf16_lo(s.z);
        acc[5] += bf16_hi(s.z);
        acc[6] += bf16_lo(s.w);
        acc[7] += bf16_hi(s.w);
      }
      uint4 o;
      o.x = pack_bf16x2(acc[0], acc[1]);
      o.y = pack_bf16x2(acc[2], acc[3]);
      o.z = pack_bf16x2(acc[4], acc[5]);
      o.w = pack_bf16x2(acc[6], acc[7]);
      cb.y[(size_t)t * vpr + v] = o;
    }
  }
}

template <int BN, int STAGES, int STAGES2>
cudaError_t run_fused(const FusedArgs& f, const CUtensorMap* g, const CUtensorMap* dm,
                      cudaStream_t st) {
  using S = GemmShape<0, BN, STAGES>;
  auto kern = ffn_fused_bf16_kernel<BN, STAGES, STAGES2>;
  cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(kern), S::SMEM);
  if (err != cudaSuccess) return err;
  // cooperative: every CTA is resident at once, so a unit that waits for another CTA's units
  // never waits for a CTA that cannot start
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sm_count());
  cfg.blockDim = dim3(GemmThreads<0>::kAll);
  cfg.dynamicSmemBytes = S::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, kern, f, g[0], g[1], g[2], g[3], dm[0], dm[1], dm[2], dm[3]);
  if (err != cudaSuccess) (void)cudaGetLastError();
  return err;
}

}  // namespace

cudaError_t launch_ffn_fused(const moe_cfg& c, const WsLayout& L, const void* recv, const void* x,
                             const moe_weights& w, void* ebuf, void* shared_out,
                             const int32_t* row_of, const float* topk_w, void* y, char* ws,
                             cudaStream_t st, const FfnPart& part) {
  if (c.act_dtype != MOE_BF16) return cudaErrorNotSupported;
  FusedArgs f{};
  CUtensorMap g[4], dm[4];
  cudaError_t err = prepare_bf16_gemm(c, L, 0, recv, x, w, ebuf, shared_out, ws, part, &f.gu, g);
  if (err == cudaSuccess)
    err = prepare_bf16_gemm(c, L, 1, recv, x, w, ebuf, shared_out, ws, part, &f.dn, dm);
  if (err != cudaSuccess) return err;
  f.done_tile = reinterpret_cast<int32_t*>(ws + L.fused_done);
  f.done_shared = f.done_tile + L.max_tiles;
  f.done_down = f.done_shared + L.shared_tiles;
  f.done_up = f.done_down + 1;
  err = cudaMemsetAsync(f.done_tile, 0, sizeof(int32_t) * (size_t)L.fused_done_n, st);
  if (err != cudaSuccess) return err;
  CombineArgs& cb = f.cb;
  cb.row_of = row_of;
  cb.topk_w = topk_w;
  cb.ebuf = static_cast<const uint4*>(ebuf);
  cb.shared_out = c.d_ff_shared ? static_cast<const uint4*>(shared_out) : nullptr;
  cb.y = static_cast<uint4*>(y);
  cb.d = c.d;
  cb.k = c.k;
  cb.T = c.T;
  cb.recv_rows = (long long)c.R * c.R * cap_of(c);
  // column slices of the combine as in the combine kernel
  const int vpr = c.d / 8;
  int nslice = 1;
  while (c.T * nslice < 2 * 152 && vpr / (nslice * 2) >= 128) nslice *= 2;
  cb.slice_vecs = (vpr + nslice - 1) / nslice;
  cb.nslice = (vpr + cb.slice_vecs - 1) / cb.slice_vecs;
  // the stage counts of the separate kernels: gate/up 5 x 40 KB and down 8 x 24 KB (64-token
  // tiles), 4 x 48 KB and 6 x 32 KB (128-token tiles)
  if (L.bn == 64) return run_fused<64, 5, 8>(f, g, dm, st);
  return run_fused<128, 4, 6>(f, g, dm, st);
}

}  // namespace moe
