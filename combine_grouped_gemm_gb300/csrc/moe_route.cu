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

// ---------------------------------------------------------------------------------------
// Partial logits for large batches through a cp.async ring. The staged kernel above holds the
// next k-step in registers; here every thread copies its share of the next kRingStages - 1
// k-steps straight into shared memory (16-byte cp.async, nothing held in registers), so no
// warp waits on a global load before the step that needs it.
//  * Copies are coalesced: two threads per 32-byte x row slice, four per 64-byte w row slice.
//    Each thread copies into slots of its own in the ring, so it can convert and transpose what
//    it copied as soon as its own copies have landed, with no barrier in between.
//  * The compute tiles are k-major fp32 as in the staged kernel ([BK][128]), with the column
//    index XOR-swizzled per k row (x: bit 4 by k/8; w: bits 3-4 by (k/4)%4) so the transposing
//    stores are free of bank conflicts; the swizzle moves 16-column groups, so a thread's
//    4-row (4-column) float4 stays contiguous.
//  * Lanes: each half-warp covers 4 thread rows x 4 thread columns, so each 16-byte operand
//    load of a half-warp touches 64 contiguous bytes.
// CTA 128 tokens x 128 experts of one chunk, 256 threads of 8 x 8 outputs, BK = 16. Every
// output is the same sequential fused multiply-add chain over its chunk as in the other
// kernels.
// ---------------------------------------------------------------------------------------
constexpr int kRingStages = 4;
constexpr int kRingBK = 16;
constexpr size_t ring_smem_bytes() {
  return (size_t)kRingStages * (256 + 512) * 16 + (size_t)2 * 2 * kRingBK * 128 * 4;
}

__global__ void __launch_bounds__(256, 2)
    route_partials_ring_kernel(const __nv_bfloat16* __restrict__ x, const float* __restrict__ wg,
                               float* __restrict__ partials, int T, int d, int E) {
  constexpr int BT = 128, BE = 128, BK = kRingBK, S = kRingStages;
  extern __shared__ __align__(16) unsigned char rring[];
  uint4* xr = reinterpret_cast<uint4*>(rring);                    // [S][256] raw x pieces
  uint4* wr = xr + S * 256;                                       // [S][512] raw w pieces
  float (*xs)[BK][BT] = reinterpret_cast<float (*)[BK][BT]>(wr + S * 512);
  float (*ws)[BK][BE] = reinterpret_cast<float (*)[BK][BE]>(&xs[2][0][0]);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ty = (warp >> 1) * 4 + ((lane & 15) >> 2);
  const int tx = (warp & 1) * 8 + (lane >> 4) * 4 + (lane & 3);
  const int e0 = blockIdx.x * BE, t0 = blockIdx.y * BT, c = blockIdx.z;
  const int L = d / kRouteChunks, kbeg = c * L, nsteps = L / BK;

  // this thread's copy pieces: x row t0 + tid/2, columns 8*(tid%2)..+7 of the step;
  // w rows e0 + p/4, columns 4*(p%4)..+3 for p = tid and tid + 256
  const int xrow = tid >> 1, xhalf = tid & 1;
  const bool xok = t0 + xrow < T;
  const __nv_bfloat16* xsrc = x + (size_t)(xok ? t0 + xrow : 0) * d + kbeg + xhalf * 8;
  int wrow[2], wq[2];
  const float* wsrc[2];
  bool wok[2];
#pragma unroll
  for (int n = 0; n < 2; ++n) {
    const int p = tid + n * 256;
    wrow[n] = p >> 2;
    wq[n] = p & 3;
    wok[n] = e0 + wrow[n] < E;
    wsrc[n] = wg + (size_t)(wok[n] ? e0 + wrow[n] : 0) * d + kbeg + wq[n] * 4;
  }
  pdl_wait();
  pdl_trigger();

  auto issue = [&](int step) {
    const int slot = step % S, k0 = step * BK;
    cp_async16_zfill(xr + slot * 256 + tid, xsrc + k0, xok ? 16 : 0);
#pragma unroll
    for (int n = 0; n < 2; ++n)
      cp_async16_zfill(wr + slot * 512 + tid + n * 256, wsrc[n] + k0, wok[n] ? 16 : 0);
  };
  // convert / transpose this thread's landed pieces of a step into compute buffer buf
  auto stash = [&](int step, int buf) {
    const int slot = step % S;
    const uint4 v = xr[slot * 256 + tid];
    const int xk = xhalf * 8, xcol = xrow ^ (xhalf << 4);
    xs[buf][xk + 0][xcol] = bf16_lo(v.x);
    xs[buf][xk + 1][xcol] = bf16_hi(v.x);
    xs[buf][xk + 2][xcol] = bf16_lo(v.y);
    xs[buf][xk + 3][xcol] = bf16_hi(v.y);
    xs[buf][xk + 4][xcol] = bf16_lo(v.z);
    xs[buf][xk + 5][xcol] = bf16_hi(v.z);
    xs[buf][xk + 6][xcol] = bf16_lo(v.w);
    xs[buf][xk + 7][xcol] = bf16_hi(v.w);
#pragma unroll
    for (int n = 0; n < 2; ++n) {
      const float4 w = *reinterpret_cast<const float4*>(wr + slot * 512 + tid + n * 256);
      const int wk = wq[n] * 4, wcol = wrow[n] ^ (wq[n] << 3);
      ws[buf][wk + 0][wcol] = w.x;
      ws[buf][wk + 1][wcol] = w.y;
      ws[buf][wk + 2][wcol] = w.z;
      ws[buf][wk + 3][wcol] = w.w;
    }
  };

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

#pragma unroll
  for (int s = 0; s < S - 1; ++s) {
    if (s < nsteps) issue(s);
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  asm volatile("cp.async.wait_group %0;" ::"n"(S - 2) : "memory");
  stash(0, 0);
  __syncthreads();
  for (int step = 0; step < nsteps; ++step) {
    const int buf = step & 1;
    if (step + S - 1 < nsteps) issue(step + S - 1);
    asm volatile("cp.async.commit_group;" ::: "memory");
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      const int sx = (kk >> 3) << 4, sw = ((kk >> 2) & 3) << 3;
      const float4 a0 = *reinterpret_cast<const float4*>(&xs[buf][kk][(ty * 4) ^ sx]);
      const float4 a1 = *reinterpret_cast<const float4*>(&xs[buf][kk][(64 + ty * 4) ^ sx]);
      const float4 b0 = *reinterpret_cast<const float4*>(&ws[buf][kk][(tx * 4) ^ sw]);
      const float4 b1 = *reinterpret_cast<const float4*>(&ws[buf][kk][(64 + tx * 4) ^ sw]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; j += 2) fma2_bcast(acc[i][j], acc[i][j + 1], b[j], b[j + 1], a[i]);
    }
    if (step + 1 < nsteps) {
      asm volatile("cp.async.wait_group %0;" ::"n"(S - 2) : "memory");
      stash(step + 1, buf ^ 1);
    }
    __syncthreads();
  }

  // rows ty*4 + (i%4) (+64 for i >= 4), columns tx*4 + (j%4) (+64 for j >= 4)
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + (i >> 2) * 64 + ty * 4 + (i & 3);
    if (t >= T) continue;
    float* prow = partials + ((size_t)c * T + t) * E;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = e0 + h * 64 + tx * 4;
      if (e + 3 < E && (E & 3) == 0) {
        *reinterpret_cast<float4*>(prow + e) =
            make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (e + j < E) prow[e + j] = acc[i][4 * h + j];
      }
    }
  }
}

// Whether the ring kernel takes this shape: 16-byte aligned rows and k-steps.
bool ring_fits(const void* x, const void* wg, int d) {
  const int L = d / kRouteChunks;
  return L % kRingBK == 0 && L > 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0 &&
         (reinterpret_cast<uintptr_t>(wg) & 15) == 0;
}

cudaError_t launch_partials_ring(const __nv_bfloat16* x, const float* wg, float* partials, int T,
                                 int d, int E, cudaStream_t st, bool pdl) {
  const size_t smem = ring_smem_bytes();
  const cudaError_t err =
      ensure_smem_limit(reinterpret_cast<const void*>(route_partials_ring_kernel), smem);
  if (err != cudaSuccess) return err;
  dim3 grid((E + 127) / 128, (T + 127) / 128, kRouteChunks);
  return launch_kernel(route_partials_ring_kernel, grid, dim3(256), smem, st, pdl, x, wg,
                       partials, T, d, E);
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
//  4. thread e of a kept group: its rank among the eligible experts under the strict total
//     order (key desc, index asc), counted against every expert of the kept groups; the
//     expert of rank i < k is the i-th choice (the same choices in the same order as k rounds
//     of argmax, without their k dependent shuffle chains: 9,100 of the 14,500 cycles a token
//     took with them);
//  5. threads i < k: the weights from the raw sigmoid scores in selection order (each forms the
//     same sequential sum).
// ---------------------------------------------------------------------------------------
constexpr int kSelThreads = 256;
__host__ __device__ constexpr int sel_cta_scratch_floats(int E) { return 2 * E + 64 + 64 + 32 + 32; }
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
  int* sel_idx = reinterpret_cast<int*>(sel_s + 32);  // [32]
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

  // 4. ranks among the eligible experts; every eligible expert has a distinct rank
  for (int e = threadIdx.x; e < E; e += kSelThreads) {
    if (!keep[e / gs]) continue;
    const float ve = v[e];
    int rank = 0;
    for (int h = 0; h < n_group; ++h) {
      if (!keep[h]) continue;
      const int j0 = h * gs, j1 = j0 + gs;
      int j = j0;
      if ((gs & 3) == 0) {
        for (; j < j1; j += 4) {
          const float4 q = *reinterpret_cast<const float4*>(v + j);
          rank += ranks_before(q.x, j, ve, e) ? 1 : 0;
          rank += ranks_before(q.y, j + 1, ve, e) ? 1 : 0;
          rank += ranks_before(q.z, j + 2, ve, e) ? 1 : 0;
          rank += ranks_before(q.w, j + 3, ve, e) ? 1 : 0;
        }
      }
      for (; j < j1; ++j) rank += ranks_before(v[j], j, ve, e) ? 1 : 0;
    }
    if (rank < k) sel_idx[rank] = e;
  }
  __syncthreads();
  if (warp != 0) return;

  // 5. weights in selection order
  const int sel_e = lane < k ? sel_idx[lane] : 0;
  if (lane < k) sel_s[lane] = s[sel_e];
  __syncwarp();
  if (lane < k) {
    float sum = 0.0f;
    for (int i = 0; i < k; ++i) sum = __fadd_rn(sum, sel_s[i]);
    topk_idx[(size_t)t * k + lane] = sel_e;
    topk_w[(size_t)t * k + lane] = __fmul_rn(__fdiv_rn(sel_s[lane], sum), route_scale);
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

// ---------------------------------------------------------------------------------------
// Selection for large batches of the DeepSeek-V3 router shape (256 experts in 8 groups of
// 32): 8 lanes per token, 4 tokens per warp. Lane q of a token's segment holds experts
// 32g + 4q + m (g = 0..7, m = 0..3) as key slots j = 4g + m: 4 experts of every group, so the
// segment's 16-byte loads of one chunk partial row are 128 contiguous bytes. The operations
// and their order are those of the file comment:
//  1. per expert: the 16 chunk partials, pairwise tree, sigmoid, selection key v = s + bias
//     (v kept in registers, s in shared memory);
//  2. per group: the two largest keys (values only), each lane's own 4 then a 3-step butterfly
//     over the segment (equal keys give equal scores whichever lane holds them);
//  3. lane q: rank of group q among the 8 groups -> kept or not (a segment ballot);
//  4. k <= 8 rounds of a segment-wide argmax over the eligible experts (key desc, index asc);
//     each lane keeps its best eligible candidate between rounds and only the owner of the
//     chosen expert rescans; lane i of the segment records the i-th choice;
//  5. weights from the raw sigmoid scores in selection order (every lane of the segment forms
//     the same sequential sum).
// ---------------------------------------------------------------------------------------
constexpr int kSegThreads = 128;   // 4 warps, 16 tokens a CTA
constexpr int kSegE = 256, kSegGroups = 8;

__global__ void __launch_bounds__(kSegThreads) route_select_seg_kernel(
    const float* __restrict__ partials, const float* __restrict__ bias,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int T, int k, int topk_group,
    float route_scale, const void* warm, size_t warm_bytes, int warm_ctas) {
  constexpr int E = kSegE;
  extern __shared__ float s_all[];   // [16 tokens][E] sigmoid scores
  pdl_wait();
  pdl_trigger();
  if ((int)blockIdx.x < warm_ctas) {   // the first CTAs only start the L2 warm-up
    l2_warm(warm, warm_bytes, blockIdx.x, warm_ctas);
    return;
  }
  const int lane = threadIdx.x & 31, q = lane & 7, seg0 = lane & ~7;
  const int tl = (threadIdx.x >> 5) * 4 + (lane >> 3);   // token within the CTA
  const int t = (blockIdx.x - warm_ctas) * (kSegThreads / 8) + tl;
  const bool tok = t < T;
  const int tt = tok ? t : 0;   // rows past T compute on token 0 and write nothing
  float* s_row = s_all + tl * E;

  // 1. selection keys of experts 32g + 4q + m
  float v[32];
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const int col = 32 * g + 4 * q;
    float4 p[kRouteChunks];
#pragma unroll
    for (int c = 0; c < kRouteChunks; ++c)
      p[c] = *reinterpret_cast<const float4*>(partials + ((size_t)c * T + tt) * E + col);
#pragma unroll
    for (int w = kRouteChunks; w > 1; w >>= 1)
#pragma unroll
      for (int j = 0; j < w / 2; ++j) {
        p[j].x = __fadd_rn(p[2 * j].x, p[2 * j + 1].x);
        p[j].y = __fadd_rn(p[2 * j].y, p[2 * j + 1].y);
        p[j].z = __fadd_rn(p[2 * j].z, p[2 * j + 1].z);
        p[j].w = __fadd_rn(p[2 * j].w, p[2 * j + 1].w);
      }
    const float4 z = p[0];
    const float4 bb = *reinterpret_cast<const float4*>(bias + col);
    float4 sv;
    sv.x = __fdiv_rn(1.0f, __fadd_rn(1.0f, route_exp(-z.x)));
    sv.y = __fdiv_rn(1.0f, __fadd_rn(1.0f, route_exp(-z.y)));
    sv.z = __fdiv_rn(1.0f, __fadd_rn(1.0f, route_exp(-z.z)));
    sv.w = __fdiv_rn(1.0f, __fadd_rn(1.0f, route_exp(-z.w)));
    v[4 * g + 0] = __fadd_rn(sv.x, bb.x);
    v[4 * g + 1] = __fadd_rn(sv.y, bb.y);
    v[4 * g + 2] = __fadd_rn(sv.z, bb.z);
    v[4 * g + 3] = __fadd_rn(sv.w, bb.w);
    *reinterpret_cast<float4*>(s_row + col) = sv;
  }
  auto expert_of = [&](int j) { return 32 * (j >> 2) + 4 * q + (j & 3); };

  // 2. group scores: the two largest keys of each group, own 4 then the segment butterfly
  float gscore = 0.0f;   // lane q ends with group q's score
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    float a = -INFINITY, b = -INFINITY;
#pragma unroll
    for (int j = 4 * g; j < 4 * g + 4; ++j) {
      const float x = v[j];
      if (x > a) {
        b = a;
        a = x;
      } else if (x > b) {
        b = x;
      }
    }
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) {
      const float c = __shfl_xor_sync(0xffffffffu, a, off);
      const float d = __shfl_xor_sync(0xffffffffu, b, off);
      const float hi = fmaxf(a, c);
      b = fmaxf(fminf(a, c), fmaxf(b, d));
      a = hi;
    }
    if (q == g) gscore = __fadd_rn(a, b);
  }

  // 3. group q is kept when fewer than topk_group groups rank before it
  int rank = 0;
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    const float gh = __shfl_sync(0xffffffffu, gscore, seg0 + h);
    rank += ranks_before(gh, h, gscore, q) ? 1 : 0;
  }
  const uint32_t kept = (__ballot_sync(0xffffffffu, rank < topk_group) >> seg0) & 0xFFu;

  // 4. k rounds of the segment argmax (key desc, index asc)
  uint32_t elig = 0;   // bit j: key slot j is in a kept group and not yet chosen
#pragma unroll
  for (int g = 0; g < 8; ++g)
    if ((kept >> g) & 1u) elig |= 0xFu << (4 * g);
  float lv = -INFINITY;
  int le = 0x7fffffff;
  auto lane_best = [&]() {
    lv = -INFINITY;
    le = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (!((elig >> j) & 1u)) continue;
      const int e = expert_of(j);
      if (le == 0x7fffffff || ranks_before(v[j], e, lv, le)) {
        lv = v[j];
        le = e;
      }
    }
  };
  lane_best();
  int sel_e = 0;
  for (int i = 0; i < k; ++i) {
    float bv = lv;
    int be = le;
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      if (oe != 0x7fffffff && (be == 0x7fffffff || ranks_before(ov, oe, bv, be))) {
        bv = ov;
        be = oe;
      }
    }
    if (be == le) {   // this lane held the chosen expert: slot 4 * (be / 32) + be % 4
      elig &= ~(1u << (4 * (be >> 5) + (be & 3)));
      lane_best();
    }
    if (q == i) sel_e = be;
  }

  // 5. weights in selection order
  __syncwarp();
  const float si = (q < k) ? s_row[sel_e & (E - 1)] : 0.0f;
  float sum = 0.0f;
  for (int i = 0; i < k; ++i) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, si, seg0 + i));
  if (tok && q < k) {
    topk_idx[(size_t)t * k + q] = sel_e;
    topk_w[(size_t)t * k + q] = __fmul_rn(__fdiv_rn(si, sum), route_scale);
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
  else if (T >= 512 && ring_fits(xb, w_gate, d))
    err = launch_partials_ring(xb, w_gate, partials, T, d, E, st, false);
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
    const size_t smem1 = (size_t)sel_cta_scratch_floats(c.E) * sizeof(float);
    return launch_kernel(route_select_cta_kernel, dim3(warm_ctas + c.T), dim3(kSelThreads), smem1,
                         st, pdl, partials, bias, topk_idx, topk_w, c.T, c.E, c.k, c.n_group,
                         c.topk_group, c.route_scale, warm, warm_bytes, warm_ctas);
  }
  // the DeepSeek-V3 router shape from 2048 tokens: 8 lanes per token (1024 tokens: 106 us
  // against 99 us with a warp per token, whose CTAs spread over more SMs; 4096 / 16384 tokens:
  // 295 / 1080 us against 304 / 1109 us, router stage with the partial-dot kernel)
  if (c.T >= 2048 && c.E == kSegE && c.n_group == kSegGroups && c.k <= 8 &&
      (reinterpret_cast<uintptr_t>(bias) & 15) == 0 && (reinterpret_cast<uintptr_t>(partials) & 15) == 0) {
    const int per_cta = kSegThreads / 8;
    return launch_kernel(route_select_seg_kernel, dim3(warm_ctas + (c.T + per_cta - 1) / per_cta),
                         dim3(kSegThreads), (size_t)per_cta * kSegE * sizeof(float), st, pdl,
                         partials, bias, topk_idx, topk_w, c.T, c.k, c.topk_group, c.route_scale,
                         warm, warm_bytes, warm_ctas);
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
