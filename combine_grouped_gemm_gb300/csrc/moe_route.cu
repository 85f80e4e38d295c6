// Router kernels: fp32 gate GEMM in a fixed summation order, sigmoid affinity, per-expert bias,
// group-limited top-k and renormalised weights.
//
// Method: "Mixture-of-experts serving" (learn-kernels), paragraph 1 (sigmoid affinity per expert
// plus a per-expert bias that steers selection), paragraph 3 (group-limited routing);
// "7.13 Serving Mixture-of-Experts" (llm-stack-book), Expert Parallelism Mechanics, router
// step (top-k, then the chosen weights renormalised).
//
// Bit-exact agreement with a CPU implementation needs one fixed sequence of fp32 operations:
//  * z = x . w: d is cut into 16 equal chunks; each chunk is a sequential fused multiply-add
//    chain starting from 0 at the chunk's first index; the 16 partials are added by a balanced
//    pairwise tree ((p0+p1)+(p2+p3))+... No tensor cores (their accumulation order is not
//    specified), no split of a chunk.
//  * e^-z: Cody-Waite range reduction n = rint(z log2 e), r = z - n ln2 (ln2 in a 9-bit head
//    and a tail, both subtracted with fused multiply-adds), e^r by the Taylor series to degree
//    7 in Horner form, times 2^n from exponent bits; z clamped to [-87, 87].
//  * s = 1/(1+e^-z) with IEEE division; v = s + b; group score = top1 + top2 of v.
//  * ties in every ranking go to the lower index; weights = (s_i / sum_j s_j) * scale with the
//    sum taken in selection order.
// Every operation is an explicitly rounded intrinsic (__fmaf_rn, __fadd_rn, __fmul_rn,
// __fdiv_rn) so the compiler cannot contract or reorder it.
#include "moe_device.cuh"

namespace moe {
namespace {

// (c0, c1) = (x0 * a + c0, x1 * a + c1): one packed fp32x2 fused multiply-add, i.e. two IEEE
// fmas each rounded once, exactly as two __fmaf_rn calls.
__device__ __forceinline__ void fma2_bcast(float& c0, float& c1, float x0, float x1, float a) {
  asm("{\n\t.reg .b64 d, x, w;\n\t"
      "mov.b64 d, {%0, %1};\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 w, {%4, %4};\n\t"
      "fma.rn.f32x2 d, x, w, d;\n\t"
      "mov.b64 {%0, %1}, d;\n\t}"
      : "+f"(c0), "+f"(c1)
      : "f"(x0), "f"(x1), "f"(a));
}

// ---------------------------------------------------------------------------------------
// Partial logits: partials[c][t][e] = sum over the c-th chunk of d of x[t][i] * w[e][i],
// one sequential FMA chain per (c, t, e).
// CTA tile BT tokens x BE experts of one chunk; thread tile TM x TN; k-steps of BK columns,
// staged through (dynamic) shared memory, k-major so the compute loop reads conflict-free, with
// the next step's global loads held in registers while the current step computes.
// ---------------------------------------------------------------------------------------
template <int BT, int BE, int TM, int TN, int BK>
constexpr int partials_smem_bytes() { return 2 * BK * (BT + BE) * 4; }

// Thread tiles of up to 64 outputs run two CTAs per SM (at most 128 registers a thread).
template <int BT, int BE, int TM, int TN, int BK>
__global__ void __launch_bounds__(256, TM * TN <= 64 ? 2 : 1)
    route_partials_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ wg,
                          float* __restrict__ partials, int T, int d, int E) {
  static_assert((BT / TM) * (BE / TN) == 256, "256 threads");
  pdl_wait();
  pdl_trigger();
  constexpr int XV = BT * BK / 8;            // 16-byte vectors of x per step (8 bf16)
  constexpr int WV = BE * BK / 4;            // 16-byte vectors of w per step (4 floats)
  constexpr int NX = (XV + 255) / 256, NW = (WV + 255) / 256;
  // static shared memory when the stages fit in 48 KB (addresses known at compile time),
  // dynamic otherwise
  constexpr int kSmemFloats = partials_smem_bytes<BT, BE, TM, TN, BK>() / 4;
  constexpr bool kStatic = kSmemFloats * 4 <= 48 * 1024;
  extern __shared__ __align__(16) float rsm[];
  __shared__ __align__(16) float rstat[kStatic ? kSmemFloats : 4];
  float* const rbase = kStatic ? rstat : rsm;
  float (*xs)[BK][BT] = reinterpret_cast<float (*)[BK][BT]>(rbase);
  float (*ws)[BK][BE] = reinterpret_cast<float (*)[BK][BE]>(rbase + 2 * BK * BT);

  const int tid = threadIdx.x;
  const int tx = tid % (BE / TN), ty = tid / (BE / TN);
  // Thread tile rows / columns. With a multiple of 4 per side they are groups of 4 consecutive
  // entries, one group per BT/(TM/4) rows (BE/(TN/4) columns), so each group is one
  // conflict-free 16-byte shared load; otherwise rows are consecutive and columns strided by
  // the thread count along the row.
  auto row_of = [&](int ty_, int i) {
    return TM % 4 == 0 ? (i / 4) * (BT / (TM / 4)) + ty_ * 4 + (i % 4) : ty_ * TM + i;
  };
  auto col_of = [&](int tx_, int j) {
    return TN % 4 == 0 ? (j / 4) * (BE / (TN / 4)) + tx_ * 4 + (j % 4) : tx_ + j * (BE / TN);
  };
  const int e0 = blockIdx.x * BE, t0 = blockIdx.y * BT, c = blockIdx.z;
  const int L = d / kRouteChunks;
  const int kbeg = c * L;
  const int nsteps = L / BK;

  float acc[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;

  uint4 rx[NX];
  float4 rw[NW];
  auto fetch = [&](int step) {
    const int k0 = kbeg + step * BK;
#pragma unroll
    for (int n = 0; n < NX; ++n) {
      const int q = tid + n * 256;
      rx[n] = make_uint4(0, 0, 0, 0);
      if (q < XV) {
        const int r = q % BT, kv = q / BT;   // consecutive threads: consecutive tokens
        const int t = t0 + r;
        if (t < T) rx[n] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * d + k0 + kv * 8));
      }
    }
#pragma unroll
    for (int n = 0; n < NW; ++n) {
      const int q = tid + n * 256;
      rw[n] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (q < WV) {
        const int r = q % BE, kv = q / BE;
        const int e = e0 + r;
        if (e < E) rw[n] = __ldg(reinterpret_cast<const float4*>(wg + (size_t)e * d + k0 + kv * 4));
      }
    }
  };
  auto stash = [&](int buf) {
#pragma unroll
    for (int n = 0; n < NX; ++n) {
      const int q = tid + n * 256;
      if (q < XV) {
        const int r = q % BT, kv = q / BT;
        xs[buf][kv * 8 + 0][r] = bf16_lo(rx[n].x);
        xs[buf][kv * 8 + 1][r] = bf16_hi(rx[n].x);
        xs[buf][kv * 8 + 2][r] = bf16_lo(rx[n].y);
        xs[buf][kv * 8 + 3][r] = bf16_hi(rx[n].y);
        xs[buf][kv * 8 + 4][r] = bf16_lo(rx[n].z);
        xs[buf][kv * 8 + 5][r] = bf16_hi(rx[n].z);
        xs[buf][kv * 8 + 6][r] = bf16_lo(rx[n].w);
        xs[buf][kv * 8 + 7][r] = bf16_hi(rx[n].w);
      }
    }
#pragma unroll
    for (int n = 0; n < NW; ++n) {
      const int q = tid + n * 256;
      if (q < WV) {
        const int r = q % BE, kv = q / BE;
        ws[buf][kv * 4 + 0][r] = rw[n].x;
        ws[buf][kv * 4 + 1][r] = rw[n].y;
        ws[buf][kv * 4 + 2][r] = rw[n].z;
        ws[buf][kv * 4 + 3][r] = rw[n].w;
      }
    }
  };

  fetch(0);
  stash(0);
  __syncthreads();
  for (int step = 0; step < nsteps; ++step) {
    const int buf = step & 1;
    if (step + 1 < nsteps) fetch(step + 1);   // in flight while this step computes
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[TM], b[TN];
#pragma unroll
      for (int i = 0; i < TM; ++i) a[i] = xs[buf][kk][row_of(ty, i)];
#pragma unroll
      for (int j = 0; j < TN; ++j) b[j] = ws[buf][kk][col_of(tx, j)];
#pragma unroll
      for (int i = 0; i < TM; ++i) {
        if constexpr (TN % 2 == 0) {
          // packed fp32x2 FMAs: two independent IEEE fmas, the same chain per output
#pragma unroll
          for (int j = 0; j < TN; j += 2)
            fma2_bcast(acc[i][j], acc[i][j + 1], b[j], b[j + 1], a[i]);
        } else {
#pragma unroll
          for (int j = 0; j < TN; ++j) acc[i][j] = __fmaf_rn(a[i], b[j], acc[i][j]);
        }
      }
    }
    if (step + 1 < nsteps) stash(buf ^ 1);
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int t = t0 + row_of(ty, i);
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int e = e0 + col_of(tx, j);
      if (e < E) partials[((size_t)c * T + t) * E + e] = acc[i][j];
    }
  }
}

// The k-step is BK columns, the largest of MAXBK, 16, 8 that divides a chunk.
template <int BT, int BE, int TM, int TN, int BK>
cudaError_t launch_partials_bk(const __nv_bfloat16* x, const float* wg, float* partials, int T,
                               int d, int E, cudaStream_t st, bool pdl) {
  constexpr int smem = partials_smem_bytes<BT, BE, TM, TN, BK>();
  auto kern = route_partials_kernel<BT, BE, TM, TN, BK>;
  const cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (err != cudaSuccess) return err;
  dim3 grid((E + BE - 1) / BE, (T + BT - 1) / BT, kRouteChunks);
  return launch_kernel(kern, grid, dim3(256), smem > 48 * 1024 ? smem : 0, st, pdl, x, wg,
                       partials, T, d, E);
}

template <int BT, int BE, int TM, int TN, int MAXBK>
cudaError_t launch_partials(const __nv_bfloat16* x, const float* wg, float* partials, int T, int d,
                            int E, cudaStream_t st, bool pdl) {
  const int L = d / kRouteChunks;
  if (MAXBK >= 32 && L % 32 == 0)
    return launch_partials_bk<BT, BE, TM, TN, (MAXBK >= 32 ? 32 : 16)>(x, wg, partials, T, d, E, st,
                                                                       pdl);
  if (L % 16 == 0) return launch_partials_bk<BT, BE, TM, TN, 16>(x, wg, partials, T, d, E, st, pdl);
  return launch_partials_bk<BT, BE, TM, TN, 8>(x, wg, partials, T, d, E, st, pdl);
}

// ---------------------------------------------------------------------------------------
// Partial logits for small batches, the CTA's whole slice resident. With few tokens the grid
// is only E/BE x 16 CTAs, and a kernel that stages one k-step at a time keeps a few KB in
// flight per SM: it waits on memory latency, not bandwidth. Here the CTA's BT rows of x and BE
// rows of w_gate over its chunk (L = d/16 columns) are all copied into shared memory at once
// with 16-byte cp.async, in G commit groups along k (rows past T or E are zero-filled), and the
// FMA chains run over each group as soon as it has landed. Nothing is overwritten, so the
// groups need no barrier other than the one after each wait.
// Shared layout: x rows [BT][L + 8] bf16, w rows [BE][L + 4] fp32, row-major with 16 bytes of
// padding, so a quarter-warp's 16-byte reads of 8 consecutive w rows hit distinct banks (the
// row stride is an odd number of 16-byte units when L % 8 == 0).
// Thread tile: rows ty*TM + i (TM even: one packed fp32x2 FMA covers two tokens against one
// weight), columns tx + j*(BE/TN). Every output is the same sequential chain over its chunk as
// in the staged kernel.
// ---------------------------------------------------------------------------------------
__host__ __device__ constexpr size_t resident_smem_bytes(int BT, int BE, int L) {
  return (size_t)BT * (L + 8) * 2 + (size_t)BE * (L + 4) * 4;
}

__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}

// wait until at most n of this thread's newest commit groups are still pending (n <= 3)
__device__ __forceinline__ void cp_async_wait_pending(int n) {
  if (n <= 0) asm volatile("cp.async.wait_group 0;" ::: "memory");
  else if (n == 1) asm volatile("cp.async.wait_group 1;" ::: "memory");
  else if (n == 2) asm volatile("cp.async.wait_group 2;" ::: "memory");
  else asm volatile("cp.async.wait_group 3;" ::: "memory");
}

template <int BT, int BE, int TM, int TN>
__global__ void __launch_bounds__(256, 1) route_partials_resident_kernel(
    const __nv_bfloat16* __restrict__ x, const float* __restrict__ wg, float* __restrict__ partials,
    int T, int d, int E, int G) {
  static_assert((BT / TM) * (BE / TN) == 256, "256 threads");
  static_assert(TM % 2 == 0, "token pairs");
  extern __shared__ __align__(16) unsigned char rres[];
  const int tid = threadIdx.x;
  const int e0 = blockIdx.x * BE, t0 = blockIdx.y * BT, c = blockIdx.z;
  const int L = d / kRouteChunks, kbeg = c * L;
  const int SX = L + 8, SW = L + 4;   // row strides (elements)
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(rres);
  float* ws = reinterpret_cast<float*>(rres + (size_t)BT * SX * 2);
  pdl_wait();
  pdl_trigger();

  // issue every copy of the slice: group g covers columns [g*KG, (g+1)*KG)
  const int KG = L / G, XV = KG / 8, WV = KG / 4;   // 16-byte vectors per row and group
  for (int g = 0; g < G; ++g) {
    const int kg = g * KG;
    for (int q = tid; q < BT * XV; q += 256) {
      const int r = q / XV, v = q - r * XV;   // consecutive threads: consecutive 16 bytes of a row
      const int t = t0 + r;
      const __nv_bfloat16* src = x + (size_t)(t < T ? t : 0) * d + kbeg + kg + v * 8;
      cp_async16_zfill(xs + r * SX + kg + v * 8, src, t < T ? 16 : 0);
    }
    for (int q = tid; q < BE * WV; q += 256) {
      const int r = q / WV, v = q - r * WV;
      const int e = e0 + r;
      const float* src = wg + (size_t)(e < E ? e : 0) * d + kbeg + kg + v * 4;
      cp_async16_zfill(ws + r * SW + kg + v * 4, src, e < E ? 16 : 0);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }

  const int tx = tid % (BE / TN), ty = tid / (BE / TN);
  float acc[TM][TN];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;
  const __nv_bfloat16* xrow = xs + (ty * TM) * SX;
  const float* wrow = ws + tx * SW;

  for (int g = 0; g < G; ++g) {
    cp_async_wait_pending(G - 1 - g);
    __syncthreads();   // every thread's copies of group g are visible
    const int kend = (g + 1) * KG;
    for (int k = g * KG; k < kend; k += 4) {
      float a[TM][4], b[TN][4];
#pragma unroll
      for (int i = 0; i < TM; ++i) {
        const uint2 u = *reinterpret_cast<const uint2*>(xrow + i * SX + k);
        a[i][0] = bf16_lo(u.x);
        a[i][1] = bf16_hi(u.x);
        a[i][2] = bf16_lo(u.y);
        a[i][3] = bf16_hi(u.y);
      }
#pragma unroll
      for (int j = 0; j < TN; ++j) {
        const float4 w = *reinterpret_cast<const float4*>(wrow + j * (BE / TN) * SW + k);
        b[j][0] = w.x;
        b[j][1] = w.y;
        b[j][2] = w.z;
        b[j][3] = w.w;
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int i = 0; i < TM; i += 2)
#pragma unroll
          for (int j = 0; j < TN; ++j)
            fma2_bcast(acc[i][j], acc[i + 1][j], a[i][kk], a[i + 1][kk], b[j][kk]);
    }
  }

#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int t = t0 + ty * TM + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int e = e0 + tx + j * (BE / TN);
      if (e < E) partials[((size_t)c * T + t) * E + e] = acc[i][j];
    }
  }
}

// Whether the resident kernel takes this shape: 16-byte aligned rows and chunks, and the slice
// within the per-CTA shared memory limit.
template <int BT, int BE>
bool resident_fits(const void* x, const void* wg, int d) {
  const int L = d / kRouteChunks;
  return L % 8 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
         (reinterpret_cast<uintptr_t>(wg) & 15) == 0 &&
         resident_smem_bytes(BT, BE, L) <= 227 * 1024;
}

template <int BT, int BE, int TM, int TN>
cudaError_t launch_partials_resident(const __nv_bfloat16* x, const float* wg, float* partials,
                                     int T, int d, int E, cudaStream_t st, bool pdl) {
  auto kern = route_partials_resident_kernel<BT, BE, TM, TN>;
  const int L = d / kRouteChunks;
  const size_t smem = resident_smem_bytes(BT, BE, L);
  const cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (err != cudaSuccess) return err;
  const int G = L % 32 == 0 ? 4 : L % 16 == 0 ? 2 : 1;
  dim3 grid((E + BE - 1) / BE, (T + BT - 1) / BT, kRouteChunks);
  return launch_kernel(kern, grid, dim3(256), smem, st, pdl, x, wg, partials, T, d, E, G);
}

// e^z by Cody-Waite reduction and a degree-7 Taylor polynomial (see the file comment).
__device__ __forceinline__ float route_exp(float z) {
  const float kLog2e = 1.44269504088896341f;
  const float kLn2Hi = 0.693359375f;      // 355/512: 9 significant bits
  const float kLn2Lo = -2.12194440e-4f;   // ln 2 - kLn2Hi
  z = fminf(fmaxf(z, -87.0f), 87.0f);
  const float n = rintf(__fmul_rn(z, kLog2e));
  float r = __fmaf_rn(-n, kLn2Hi, z);
  r = __fmaf_rn(-n, kLn2Lo, r);
  float p = 1.98412698e-4f;                // 1/7!
  p = __fmaf_rn(p, r, 1.38888889e-3f);     // 1/6!
  p = __fmaf_rn(p, r, 8.33333333e-3f);     // 1/5!
  p = __fmaf_rn(p, r, 4.16666667e-2f);     // 1/4!
  p = __fmaf_rn(p, r, 1.66666667e-1f);     // 1/3!
  p = __fmaf_rn(p, r, 0.5f);               // 1/2!
  p = __fmaf_rn(p, r, 1.0f);               // 1/1!
  p = __fmaf_rn(p, r, 1.0f);               // 1/0!
  const float two_n = __int_as_float((static_cast<int>(n) + 127) << 23);
  return __fmul_rn(p, two_n);
}

__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// k rounds of a warp-wide argmax over the eligible experts of one token under the total order
// (key desc, index asc); lane l holds candidates e = l + 32q. Each lane's best candidate is kept
// between rounds and only the lane whose candidate was taken looks again, so a round is one
// butterfly of shuffles (a strict total order: the argmax does not depend on how it is reduced).
// Returns, in lane i < k, the i-th choice. E <= 1024.
__device__ __forceinline__ int warp_topk(const float* v, const int* keep, int E, int gs, int k,
                                         int lane) {
  uint32_t elig = 0;   // bit q: candidate lane + 32q is in a kept group and not yet chosen
  for (int q = 0, e = lane; e < E; ++q, e += 32)
    if (keep[e / gs]) elig |= 1u << q;
  auto lane_best = [&](float& bv, int& be) {
    bv = -INFINITY;
    be = 0x7fffffff;
    for (uint32_t m = elig; m; m &= m - 1) {
      const int e = lane + 32 * (__ffs(m) - 1);
      if (be == 0x7fffffff || ranks_before(v[e], e, bv, be)) {
        bv = v[e];
        be = e;
      }
    }
  };
  float lv;
  int le;
  lane_best(lv, le);
  int sel_e = -1;
  for (int i = 0; i < k; ++i) {
    float bv = lv;
    int be = le;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (oe != 0x7fffffff && (be == 0x7fffffff || ranks_before(ov, oe, bv, be))) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) {
      elig &= ~(1u << (be >> 5));
      lane_best(lv, le);
    }
    if (lane == i) sel_e = be;
  }
  return sel_e;
}

// ---------------------------------------------------------------------------------------
// Selection for small batches: one CTA (256 threads) per token.
//  1. thread e: the 16 chunk partials of expert e (coalesced across threads), pairwise tree,
//     sigmoid, selection key v = s + bias;
//  2. warp w: scores of groups w, w+8, ...: the two largest keys of the group by a warp-wide
//     top-2 merge (values only: equal keys give equal scores whichever expert carries them);
//  3. thread g: rank of group g among all groups -> kept or not;
//  4. warp 0: k rounds of a warp-wide argmax over the eligible experts (key desc, index asc),
//     then the weights from the raw sigmoid scores in selection order.
// ---------------------------------------------------------------------------------------
constexpr int kSelThreads = 256;
constexpr int kWarmCtas = 64;   // CTAs that issue the L2 warm-up (about 1 MB each for DSV3)

__global__ void __launch_bounds__(kSelThreads) route_select_cta_kernel(
    const float* __restrict__ partials, const float* __restrict__ bias,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int T, int E, int k,
    int n_group, int topk_group, float route_scale, const void* warm, size_t warm_bytes,
    int warm_ctas) {
  extern __shared__ float sm[];
  float* s = sm;                 // [E] sigmoid scores
  float* v = s + E;              // [E] selection keys
  float* gscore = v + E;         // [64]
  int* keep = reinterpret_cast<int*>(gscore + 64);   // [64]
  float* sel_s = reinterpret_cast<float*>(keep + 64); // [32]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  if ((int)blockIdx.x < warm_ctas) {   // the first CTAs only start the L2 warm-up
    l2_warm(warm, warm_bytes, blockIdx.x, warm_ctas);
    return;
  }
  const int t = blockIdx.x - warm_ctas;

  for (int e = threadIdx.x; e < E; e += kSelThreads) {
    float p[kRouteChunks];
#pragma unroll
    for (int c = 0; c < kRouteChunks; ++c) p[c] = partials[((size_t)c * T + t) * E + e];
#pragma unroll
    for (int w = kRouteChunks; w > 1; w >>= 1)
#pragma unroll
      for (int j = 0; j < w / 2; ++j) p[j] = __fadd_rn(p[2 * j], p[2 * j + 1]);
    const float si = __fdiv_rn(1.0f, __fadd_rn(1.0f, route_exp(-p[0])));
    s[e] = si;
    v[e] = __fadd_rn(si, bias[e]);
  }
  __syncthreads();

  const int gs = E / n_group;
  for (int g = warp; g < n_group; g += kSelThreads / 32) {
    float a = -INFINITY, b = -INFINITY;  // this lane's two largest keys of group g
    for (int e = g * gs + lane; e < (g + 1) * gs; e += 32) {
      const float x = v[e];
      if (x > a) {
        b = a;
        a = x;
      } else if (x > b) {
        b = x;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float c = __shfl_xor_sync(0xffffffffu, a, off);
      const float d = __shfl_xor_sync(0xffffffffu, b, off);
      const float hi = fmaxf(a, c);
      b = fmaxf(fminf(a, c), fmaxf(b, d));
      a = hi;
    }
    if (lane == 0) gscore[g] = gs >= 2 ? __fadd_rn(a, b) : a;
  }
  __syncthreads();
  for (int g = threadIdx.x; g < n_group; g += kSelThreads) {
    int rank = 0;
    for (int h = 0; h < n_group; ++h) rank += ranks_before(gscore[h], h, gscore[g], g) ? 1 : 0;
    keep[g] = rank < topk_group;
  }
  __syncthreads();
  if (warp != 0) return;

  const int sel_e = warp_topk(v, keep, E, gs, k, lane);
  if (lane < k) sel_s[lane] = s[sel_e];
  __syncwarp();
  if (lane == 0) {
    float sum = 0.0f;
    for (int i = 0; i < k; ++i) sum = __fadd_rn(sum, sel_s[i]);
    for (int i = 0; i < k; ++i) sel_s[i] = __fmul_rn(__fdiv_rn(sel_s[i], sum), route_scale);
  }
  __syncwarp();
  if (lane < k) {
    topk_idx[(size_t)t * k + lane] = sel_e;
    topk_w[(size_t)t * k + lane] = sel_s[lane];
  }
}

// ---------------------------------------------------------------------------------------
// Selection for large batches: one warp per token, several tokens per CTA; each warp has its own
// shared-memory scratch. The operations and their order are those of the file comment:
//  1. lane l, experts e = l, l+32, ...: the 16 chunk partials (coalesced across lanes), pairwise
//     tree, sigmoid, selection key v = s + bias;
//  2. per group: the two largest keys by a warp-wide top-2 merge (values only: equal keys give
//     equal scores whichever expert carries them);
//  3. lane g: rank of group g among all groups -> kept or not;
//  4. k rounds of a warp-wide argmax over the eligible experts (key desc, index asc), then the
//     weights from the raw sigmoid scores in selection order.
// ---------------------------------------------------------------------------------------
__host__ __device__ constexpr int sel_scratch_floats(int E) { return 2 * E + 64 + 64 + 32; }

__global__ void __launch_bounds__(256) route_select_kernel(
    const float* __restrict__ partials, const float* __restrict__ bias,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int T, int E, int k,
    int n_group, int topk_group, float route_scale, const void* warm, size_t warm_bytes,
    int warm_ctas) {
  extern __shared__ float sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  pdl_trigger();
  if ((int)blockIdx.x < warm_ctas) {   // the first CTAs only start the L2 warm-up
    l2_warm(warm, warm_bytes, blockIdx.x, warm_ctas);
    return;
  }
  const int t = (blockIdx.x - warm_ctas) * (blockDim.x >> 5) + warp;
  if (t >= T) return;   // whole warps only: no block-wide barrier follows
  float* s = sm + warp * sel_scratch_floats(E);        // [E] sigmoid scores
  float* v = s + E;                                    // [E] selection keys
  float* gscore = v + E;                               // [64]
  int* keep = reinterpret_cast<int*>(gscore + 64);     // [64]
  float* sel_s = reinterpret_cast<float*>(keep + 64);  // [32]

#pragma unroll 4
  for (int e = lane; e < E; e += 32) {
    float p[kRouteChunks];
#pragma unroll
    for (int c = 0; c < kRouteChunks; ++c) p[c] = partials[((size_t)c * T + t) * E + e];
#pragma unroll
    for (int w = kRouteChunks; w > 1; w >>= 1)
#pragma unroll
      for (int j = 0; j < w / 2; ++j) p[j] = __fadd_rn(p[2 * j], p[2 * j + 1]);
    const float si = __fdiv_rn(1.0f, __fadd_rn(1.0f, route_exp(-p[0])));
    s[e] = si;
    v[e] = __fadd_rn(si, bias[e]);
  }
  __syncwarp();

  const int gs = E / n_group;
  for (int g = 0; g < n_group; ++g) {
    float a = -INFINITY, b = -INFINITY;  // this lane's two largest keys of group g
    for (int e = g * gs + lane; e < (g + 1) * gs; e += 32) {
      const float x = v[e];
      if (x > a) {
        b = a;
        a = x;
      } else if (x > b) {
        b = x;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float c = __shfl_xor_sync(0xffffffffu, a, off);
      const float d = __shfl_xor_sync(0xffffffffu, b, off);
      const float hi = fmaxf(a, c);
      b = fmaxf(fminf(a, c), fmaxf(b, d));
      a = hi;
    }
    if (lane == 0) gscore[g] = gs >= 2 ? __fadd_rn(a, b) : a;
  }
  __syncwarp();
  for (int g = lane; g < n_group; g += 32) {
    int rank = 0;
    for (int h = 0; h < n_group; ++h) rank += ranks_before(gscore[h], h, gscore[g], g) ? 1 : 0;
    keep[g] = rank < topk_group;
  }
  __syncwarp();

  const int sel_e = warp_topk(v, keep, E, gs, k, lane);
  if (lane < k) sel_s[lane] = s[sel_e];
  __syncwarp();
  if (lane == 0) {
    float sum = 0.0f;
    for (int i = 0; i < k; ++i) sum = __fadd_rn(sum, sel_s[i]);
    for (int i = 0; i < k; ++i) sel_s[i] = __fmul_rn(__fdiv_rn(sel_s[i], sum), route_scale);
  }
  __syncwarp();
  if (lane < k) {
    topk_idx[(size_t)t * k + lane] = sel_e;
    topk_w[(size_t)t * k + lane] = sel_s[lane];
  }
}

}  // namespace

cudaError_t launch_route(const moe_cfg& c, const void* x, const float* w_gate, const float* bias,
                         int32_t* topk_idx, float* topk_w, float* partials, uint32_t* status,
                         cudaStream_t st, bool pdl, const void* warm, size_t warm_bytes) {
  (void)status;
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  if (reinterpret_cast<uintptr_t>(warm) & 15) warm = nullptr;   // bulk prefetches need 16 bytes
  if (!warm) warm_bytes = 0;
  // extra CTAs at the front of the selection grid issue the warm-up on SMs of their own, off
  // the selection's path
  const int warm_ctas = warm_bytes ? kWarmCtas : 0;
  // The tile grows with T: larger thread tiles read shared memory less often per FMA (the small
  // tiles are bound by it), smaller CTA tiles keep the 16 chunks x E/BE x T/BT grid several
  // CTAs per SM deep. Measured on the DSV3 router (partials + selection, us, gate weights in
  // L2): T = 8 / 64 / 104 / 128: 21 / 25 / 31 / 31 with the resident slice (staged 32x32,
  // 64x32, 64x32, 64x64: 25 / 29 / 39 / 35); T = 256: 52 with 64x64 (32x32: 71); T = 512 /
  // 1024: 75 / 114 with 128x128 (32x32: 146 / 268).
  // Up to 128 tokens the whole per-CTA slice is resident (its copies all in flight at once).
  // The partial-dot kernel follows the caller's own work, so it is launched as usual.
  const int T = c.T, d = c.d, E = c.E;
  cudaError_t err;
  if (T <= 32 && resident_fits<32, 32>(xb, w_gate, d))
    err = launch_partials_resident<32, 32, 2, 2>(xb, w_gate, partials, T, d, E, st, false);
  else if (T <= 64 && resident_fits<64, 32>(xb, w_gate, d))
    err = launch_partials_resident<64, 32, 2, 4>(xb, w_gate, partials, T, d, E, st, false);
  else if (T <= 128 && resident_fits<128, 32>(xb, w_gate, d))
    err = launch_partials_resident<128, 32, 4, 4>(xb, w_gate, partials, T, d, E, st, false);
  else if (T >= 512)
    err = launch_partials<128, 128, 8, 8, 16>(xb, w_gate, partials, T, d, E, st, false);
  else if (T >= 128)
    err = launch_partials<64, 64, 4, 4, 32>(xb, w_gate, partials, T, d, E, st, false);
  else if (T >= 32)
    err = launch_partials<64, 32, 4, 2, 32>(xb, w_gate, partials, T, d, E, st, false);
  else
    err = launch_partials<32, 32, 2, 2, 32>(xb, w_gate, partials, T, d, E, st, false);
  if (err != cudaSuccess) return err;
  if (c.T < 1024) {   // a CTA per token keeps every expert's loads in flight at once
    const size_t smem1 = (size_t)sel_scratch_floats(c.E) * sizeof(float);
    return launch_kernel(route_select_cta_kernel, dim3(warm_ctas + c.T), dim3(kSelThreads), smem1,
                         st, pdl, partials, bias, topk_idx, topk_w, c.T, c.E, c.k, c.n_group,
                         c.topk_group, c.route_scale, warm, warm_bytes, warm_ctas);
  }
  // one warp per token; CTAs of up to 8 warps, fewer when T is small so the tokens still spread
  // over the SMs
  const int wpc = c.T >= 2432 ? 8 : c.T >= 1216 ? 4 : 2;
  const size_t smem = (size_t)wpc * sel_scratch_floats(c.E) * sizeof(float);
  err = ensure_smem_limit(reinterpret_cast<const void*>(route_select_kernel), smem);
  if (err != cudaSuccess) return err;
  return launch_kernel(route_select_kernel, dim3(warm_ctas + (c.T + wpc - 1) / wpc),
                       dim3(32 * wpc), smem, st, pdl, partials, bias, topk_idx, topk_w, c.T, c.E,
                       c.k, c.n_group, c.topk_group, c.route_scale, warm, warm_bytes, warm_ctas);
}

}  // namespace moe
