// Dispatch kernels: per-source histogram, exclusive scan inside each destination rank, stable
// scatter of token rows into the rank-major receive buffer (optionally quantised to e4m3).
//
// Method: "7.13 Serving Mixture-of-Experts" (llm-stack-book), Expert Parallelism Mechanics,
// dispatch step (rows for the same destination made contiguous, one row per (token, expert));
// "One-Sided Expert-Parallel All-to-All for Mixture-of-Experts Inference over NVLink",
// abstract (each source pushes into rank-major buffers on the target with no metadata
// exchange first); "Serving Mixture-of-Experts", DeepEP section (FP8 E4M3 dispatch; fixed-size
// padded receive buffers, so no count has to be exchanged or read back by the host).
//
// Layout: destination rank r, source rank s, a segment of cap = (T/R)*min(k, E/R) rows. Inside
// a segment, rows are grouped by local expert (ascending) and by token index inside an expert.
// Each source computes its own offsets, so no rank needs another rank's counts.
#include "moe_device.cuh"
#include "moe_scale.cuh"

namespace moe {
namespace {

constexpr int kIndexWarps = 16;

// Choice i of token t is dispatched when its expert is in [0, E) and differs from the token's
// earlier choices; otherwise (input that the router never produces) it is skipped, its row_of
// is -1 and MOE_DEV_BOUNDS is reported. With distinct experts a token sends at most
// min(k, E/R) rows to one destination rank, so no segment can overflow.
// The token's k choices are read once (independent loads, then L1-resident local copies) and
// the valid ones marked in a bit mask.
constexpr int kMaxK = 32;
__device__ __forceinline__ uint32_t load_choices(const int32_t* __restrict__ topk_idx, int t,
                                                 int k, int E, int* ids) {
  const int32_t* row = topk_idx + (size_t)t * k;
  for (int i = 0; i < k; ++i) ids[i] = __ldg(row + i);
  uint32_t valid = 0;
  for (int i = 0; i < k; ++i) {
    const int e = ids[i];
    bool ok = e >= 0 && e < E;
    for (int j = 0; j < i && ok; ++j) ok = ids[j] != e;
    valid |= static_cast<uint32_t>(ok) << i;
  }
  return valid;
}

// Where the rows of a source go when the experts are placed on slots (redundant experts):
// slot p of G = R*S holds expert slot_expert[p] on rank p / S; expert e has n_copies[e] copies
// in slots copy_slot[e][0..], ascending. Source s sends its j-th row of expert e (in token
// order) to copy (j + s) mod n_copies[e], as that copy's row j / n_copies[e]: each source splits
// its own rows of an expert evenly over the copies, with no count exchanged.
struct Placement {
  const int32_t* slot_expert;   // [G]
  const int32_t* n_copies;      // [E]
  const int32_t* copy_slot;     // [E][max_copies]
  int max_copies;
  int slots_per_rank;           // S
};

// One CTA per logical source rank. Shared memory: run[16][E] (per-warp histogram, then
// running per-warp positions), mask[16][E] (lanes of the current 32-token chunk that chose e),
// cnt[E] (the source's rows per expert), off[G] (first row of each slot inside its segment;
// the slots are the experts themselves, G = E, without a placement).
__global__ void __launch_bounds__(kIndexWarps * 32) dispatch_index_kernel(
    const int32_t* __restrict__ topk_idx, int32_t* __restrict__ counts,
    int32_t* __restrict__ row_of, int32_t* __restrict__ src_tok, uint32_t* status, int T, int E,
    int k, int R, int cap, Placement pl) {
  extern __shared__ int32_t smi[];
  const bool placed = pl.slot_expert != nullptr;
  const int G = placed ? R * pl.slots_per_rank : E;
  int32_t* run = smi;                                              // [16][E]
  uint32_t* mask = reinterpret_cast<uint32_t*>(run + kIndexWarps * E);  // [16][E]
  int32_t* cnt = reinterpret_cast<int32_t*>(mask + kIndexWarps * E);    // [E]
  int32_t* off = cnt + E;                                               // [G]
  pdl_wait();
  pdl_trigger();

  const int s = blockIdx.x;
  const int Ts = T / R;
  const int Sg = G / R;   // slots per destination rank
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per = (Ts + kIndexWarps - 1) / kIndexWarps;
  const int my0 = s * Ts + min(Ts, warp * per);
  const int my1 = s * Ts + min(Ts, (warp + 1) * per);

  for (int i = threadIdx.x; i < 2 * kIndexWarps * E; i += blockDim.x) smi[i] = 0;
  __syncthreads();

  // 1. per-warp histograms of this source's choices
  int ids[kMaxK];
  for (int t = my0 + lane; t < my1; t += 32) {
    const uint32_t valid = load_choices(topk_idx, t, k, E, ids);
    if (valid != (k >= 32 ? 0xffffffffu : (1u << k) - 1u)) raise_status(status, MOE_DEV_BOUNDS);
    for (int i = 0; i < k; ++i)
      if ((valid >> i) & 1u) atomicAdd(&run[warp * E + ids[i]], 1);
  }
  __syncthreads();

  // 2. per expert: exclusive prefix over warps (each warp's first position), total count
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int acc = 0;
    for (int w = 0; w < kIndexWarps; ++w) {
      const int h = run[w * E + e];
      run[w * E + e] = acc;
      acc += h;
    }
    cnt[e] = acc;
  }
  __syncthreads();
  // rows of this source per slot: an expert's own count, or its copy's share (rows j with
  // j = c0 mod n, c0 = (c - s) mod n, for copy c of n)
  for (int p = threadIdx.x; p < G; p += blockDim.x) {
    int v = 0;
    if (!placed) {
      v = cnt[p];
    } else {
      const int e = pl.slot_expert[p];
      if (e >= 0 && e < E) {
        const int n = max(1, pl.n_copies[e]);
        int c = 0;
        while (c < n && c < pl.max_copies && pl.copy_slot[(size_t)e * pl.max_copies + c] != p) ++c;
        const int c0 = ((c - s) % n + n) % n;
        v = cnt[e] > c0 ? (cnt[e] - c0 + n - 1) / n : 0;
      }
    }
    off[p] = v;
    counts[(size_t)s * G + p] = v;
  }
  __syncthreads();

  // 3. exclusive scan of counts over slots, restarted at every destination rank
  if (warp == 0) {
    const int chunk = (G + 31) / 32;
    const int a = min(G, lane * chunk), b = min(G, (lane + 1) * chunk);
    int local = 0;
    for (int p = a; p < b; ++p) local += off[p];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    int ex = incl - local;
    for (int p = a; p < b; ++p) {
      const int c = off[p];
      off[p] = ex;  // global exclusive sum for now
      ex += c;
    }
  }
  __syncthreads();
  // rebase to the destination rank's first slot (read all bases before overwriting)
  int base_vals[4];
  int nb = 0;
  for (int p = threadIdx.x; p < G && nb < 4; p += blockDim.x) base_vals[nb++] = off[(p / Sg) * Sg];
  __syncthreads();
  nb = 0;
  for (int p = threadIdx.x; p < G && nb < 4; p += blockDim.x) off[p] -= base_vals[nb++];
  __syncthreads();

  // 4. stable positions: walk the warp's tokens in chunks of 32, one token per lane
  const uint32_t lt = (1u << lane) - 1u;
  for (int base = my0; base < my1; base += 32) {
    const int t = base + lane;
    const bool valid = t < my1;
    const uint32_t vmask = valid ? load_choices(topk_idx, t, k, E, ids) : 0u;
    if (valid)
      for (int i = 0; i < k; ++i)
        if ((vmask >> i) & 1u) atomicOr(&mask[warp * E + ids[i]], 1u << lane);
    __syncwarp();
    if (valid)
      for (int i = 0; i < k; ++i) {
        if (!((vmask >> i) & 1u)) {
          row_of[(size_t)t * k + i] = -1;
          continue;
        }
        const int e = ids[i];
        const uint32_t m = mask[warp * E + e];
        const int j = run[warp * E + e] + __popc(m & lt);   // the source's j-th row of e
        int p = e, pos = j;
        if (placed) {
          const int n = max(1, pl.n_copies[e]);
          const int c = (j + s) % n;
          p = c < pl.max_copies ? pl.copy_slot[(size_t)e * pl.max_copies + c] : -1;
          pos = j / n;
          if (p < 0 || p >= G) {
            raise_status(status, MOE_DEV_BOUNDS);
            row_of[(size_t)t * k + i] = -1;
            continue;
          }
        }
        const int r = p / Sg;
        const int in_seg = off[p] + pos;
        if (in_seg < 0 || in_seg >= cap) {   // cannot happen with distinct experts; never written
          raise_status(status, MOE_DEV_BOUNDS);
          row_of[(size_t)t * k + i] = -1;
          continue;
        }
        const int row = (r * R + s) * cap + in_seg;
        row_of[(size_t)t * k + i] = row;
        if (src_tok) src_tok[row] = t;
      }
    __syncwarp();
    if (valid)
      for (int i = 0; i < k; ++i) {
        if (!((vmask >> i) & 1u)) continue;
        const int e = ids[i];
        const uint32_t m = mask[warp * E + e];
        if (m != 0u && (m & lt) == 0u) {  // lowest lane that chose e in this chunk
          run[warp * E + e] += __popc(m);
          mask[warp * E + e] = 0u;
        }
      }
    __syncwarp();
  }
}

// bf16 payload: block (token t, column slice); each 16-byte vector of x[t] is read once and
// written to each of the token's k receive rows.
__global__ void __launch_bounds__(128) dispatch_copy_bf16_kernel(
    const uint4* __restrict__ x, const int32_t* __restrict__ row_of, uint4* __restrict__ recv,
    int d, int k, int slice_vecs) {
  __shared__ int32_t rows[32];
  const int t = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x < k) rows[threadIdx.x] = row_of[(size_t)t * k + threadIdx.x];
  __syncthreads();
  const int vpr = d / 8;  // 16-byte vectors per row
  const int v0 = blockIdx.y * slice_vecs, v1 = min(vpr, v0 + slice_vecs);
  for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
    const uint4 val = __ldg(x + (size_t)t * vpr + v);
    for (int i = 0; i < k; ++i) {
      const int row = rows[i];
      if (row >= 0) recv[(size_t)row * vpr + v] = val;
    }
  }
}

// e4m3 payload: 16 threads per 128-column block, 8 columns per thread. amax over the block,
// scale = amax/448 (1 if amax is 0), or with pow2 the smallest power of two not below it,
// code = e4m3(x / scale) with IEEE division, nearest even, saturating. The codes and the scale
// are written to each of the token's rows; the scales are block-major, recv_scales[block][row]
// with sc_ld rows per block.
__global__ void __launch_bounds__(128) dispatch_copy_e4m3_kernel(
    const uint4* __restrict__ x, const int32_t* __restrict__ row_of, uint2* __restrict__ recv,
    float* __restrict__ recv_scales, long long sc_ld, int d, int k, int slice_vecs, int pow2) {
  __shared__ int32_t rows[32];
  const int t = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  // row_of == nullptr: quantise token t into row t (the shared expert's input)
  if (threadIdx.x < k) rows[threadIdx.x] = row_of ? row_of[(size_t)t * k + threadIdx.x] : t;
  __syncthreads();
  const int vpr = d / 8;
  const int v0 = blockIdx.y * slice_vecs, v1 = min(vpr, v0 + slice_vecs);
  for (int vb = v0; vb < v1; vb += blockDim.x) {
    const int v = vb + threadIdx.x;  // v0 and blockDim are multiples of 16: groups align
    const bool in = v < v1;
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (in) raw = __ldg(x + (size_t)t * vpr + v);
    float f[8] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y),
                  bf16_lo(raw.z), bf16_hi(raw.z), bf16_lo(raw.w), bf16_hi(raw.w)};
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale =
        pow2 ? pow2_block_scale(amax) : (amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int j = 0; j < 4; j += 2) {
      const __nv_fp8x2_storage_t p = __nv_cvt_float2_to_fp8x2(
          make_float2(__fdiv_rn(f[j], scale), __fdiv_rn(f[j + 1], scale)), __NV_SATFINITE,
          __NV_E4M3);
      lo |= static_cast<uint32_t>(p) << (8 * j);
    }
#pragma unroll
    for (int j = 4; j < 8; j += 2) {
      const __nv_fp8x2_storage_t p = __nv_cvt_float2_to_fp8x2(
          make_float2(__fdiv_rn(f[j], scale), __fdiv_rn(f[j + 1], scale)), __NV_SATFINITE,
          __NV_E4M3);
      hi |= static_cast<uint32_t>(p) << (8 * (j - 4));
    }
    if (in) {
      const bool leader = (threadIdx.x & 15) == 0;
      for (int i = 0; i < k; ++i) {
        const int row = rows[i];
        if (row < 0) continue;
        recv[(size_t)row * vpr + v] = make_uint2(lo, hi);
        if (leader) recv_scales[(long long)(v / 16) * sc_ld + row] = scale;
      }
    }
  }
}

// Column slices so that the grid covers every SM about twice even for few tokens; slices are
// whole 128-column blocks.
void copy_grid(int T, int d, int* nslice_out, int* slice_vecs_out) {
  const int vpr = d / 8;
  int nslice = 1;
  while (T * nslice < 2 * 152 && vpr / (nslice * 2) >= 128) nslice *= 2;
  int slice_vecs = (vpr + nslice - 1) / nslice;
  slice_vecs = (slice_vecs + 15) / 16 * 16;
  *slice_vecs_out = slice_vecs;
  *nslice_out = (vpr + slice_vecs - 1) / slice_vecs;
}

}  // namespace

cudaError_t launch_quant_rows_e4m3(const void* x, int T, int d, void* out, float* scales,
                                   cudaStream_t st, bool pdl, bool pow2) {
  int nslice, slice_vecs;
  copy_grid(T, d, &nslice, &slice_vecs);
  return launch_kernel(dispatch_copy_e4m3_kernel, dim3(T, nslice), dim3(128), 0, st, pdl,
                       static_cast<const uint4*>(x), static_cast<const int32_t*>(nullptr),
                       static_cast<uint2*>(out), scales, (long long)T, d, 1, slice_vecs,
                       pow2 ? 1 : 0);
}

cudaError_t launch_dispatch(const moe_cfg& c, const void* x, const int32_t* topk_idx, void* recv,
                            float* recv_scales, int32_t* counts, int32_t* row_of,
                            int32_t* src_tok, uint32_t* status, cudaStream_t st, bool pdl,
                            bool clear_src_tok, const moe_placement* placement) {
  const moe_cfg cs = slot_cfg(c, placement);   // the receive layout is over the slots
  const int cap = cap_of(cs);
  cudaError_t err;
  const bool memset_first = src_tok && clear_src_tok;
  if (memset_first) {
    err = cudaMemsetAsync(src_tok, 0xff, sizeof(int32_t) * (size_t)cs.R * cs.R * cap, st);
    if (err != cudaSuccess) return err;
  }
  Placement pl{};
  if (placement) {
    pl.slot_expert = placement->slot_expert;
    pl.n_copies = placement->n_copies;
    pl.copy_slot = placement->copy_slot;
    pl.max_copies = placement->max_copies;
    pl.slots_per_rank = placement->slots_per_rank;
  }
  const size_t smem = sizeof(int32_t) * ((size_t)(2 * kIndexWarps + 1) * c.E + cs.E);
  err = ensure_smem_limit(reinterpret_cast<const void*>(dispatch_index_kernel), smem);
  if (err != cudaSuccess) return err;
  // (after the memset the index kernel is launched as usual: its predecessor is not a kernel)
  err = launch_kernel(dispatch_index_kernel, dim3(c.R), dim3(kIndexWarps * 32), smem, st,
                      pdl && !memset_first,
                      topk_idx, counts, row_of, src_tok, status, c.T, c.E, c.k, c.R, cap, pl);
  if (err != cudaSuccess || recv == nullptr) return err;   // gather mode: indices only

  int nslice, slice_vecs;
  copy_grid(c.T, c.d, &nslice, &slice_vecs);
  dim3 grid(c.T, nslice);
  if (is_fp8(c)) {
    return launch_kernel(dispatch_copy_e4m3_kernel, grid, dim3(128), 0, st, pdl,
                         static_cast<const uint4*>(x), static_cast<const int32_t*>(row_of),
                         static_cast<uint2*>(recv), recv_scales, (long long)c.R * c.R * cap, c.d,
                         c.k, slice_vecs, pow2_scales(c) ? 1 : 0);
  }
  return launch_kernel(dispatch_copy_bf16_kernel, grid, dim3(128), 0, st, pdl,
                       static_cast<const uint4*>(x), static_cast<const int32_t*>(row_of),
                       static_cast<uint4*>(recv), c.d, c.k, slice_vecs);
}

}  // namespace moe
