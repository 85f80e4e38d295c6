// Combine kernel: weighted gather-sum of each token's k expert-output rows back to token order,
// plus the shared expert's row, in fp32, rounded once to bf16.
//
// Method: "7.13 Serving Mixture-of-Experts" (llm-stack-book), Expert Parallelism Mechanics,
// combine step (a token's k partial results weighted-summed by its gate weights); DeepEP
// section (the combine stays in BF16).
#include "moe_device.cuh"

namespace moe {
namespace {

// Block (token t, column slice), 128 threads, one 16-byte vector (8 columns) per thread per
// iteration: k gathered row vectors and the shared row, fp32 FMAs in selection order.
// Rows outside [0, recv_rows) are skipped: a negative one silently (a choice the dispatch
// skipped), one past the buffer with MOE_DEV_BOUNDS in status (input the dispatch never writes).
__global__ void __launch_bounds__(128) combine_kernel(const uint4* __restrict__ ebuf,
                                                      const int32_t* __restrict__ row_of,
                                                      const float* __restrict__ topk_w,
                                                      const uint4* __restrict__ shared_out,
                                                      uint4* __restrict__ y, int d, int k,
                                                      int slice_vecs, long long recv_rows,
                                                      uint32_t* status) {
  __shared__ int32_t rows[32];
  pdl_wait();
  pdl_trigger();
  __shared__ float wts[32];
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    int row = row_of[(size_t)t * k + threadIdx.x];
    if (row >= recv_rows) {
      if (blockIdx.y == 0) raise_status(status, MOE_DEV_BOUNDS);
      row = -1;
    }
    rows[threadIdx.x] = row;
    wts[threadIdx.x] = topk_w[(size_t)t * k + threadIdx.x];
  }
  __syncthreads();
  const int vpr = d / 8;
  const int v0 = blockIdx.y * slice_vecs, v1 = min(vpr, v0 + slice_vecs);
  for (int v = v0 + threadIdx.x; v < v1; v += blockDim.x) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    // rows in groups of 8 whose loads are all issued before the first is used
    for (int i0 = 0; i0 < k; i0 += 8) {
      uint4 e[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int row = (i0 + u < k) ? rows[i0 + u] : -1;
        e[u] = row >= 0 ? __ldg(ebuf + (size_t)row * vpr + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (i0 + u >= k || rows[i0 + u] < 0) continue;
        const float w = wts[i0 + u];
        acc[0] = __fmaf_rn(w, bf16_lo(e[u].x), acc[0]);
        acc[1] = __fmaf_rn(w, bf16_hi(e[u].x), acc[1]);
        acc[2] = __fmaf_rn(w, bf16_lo(e[u].y), acc[2]);
        acc[3] = __fmaf_rn(w, bf16_hi(e[u].y), acc[3]);
        acc[4] = __fmaf_rn(w, bf16_lo(e[u].z), acc[4]);
        acc[5] = __fmaf_rn(w, bf16_hi(e[u].z), acc[5]);
        acc[6] = __fmaf_rn(w, bf16_lo(e[u].w), acc[6]);
        acc[7] = __fmaf_rn(w, bf16_hi(e[u].w), acc[7]);
      }
    }
    if (shared_out) {
      const uint4 s = __ldg(shared_out + (size_t)t * vpr + v);
      acc[0] += bf16_lo(s.x);
      acc[1] += bf16_hi(s.x);
      acc[2] += bf16_lo(s.y);
      acc[3] += bf16_hi(s.y);
      acc[4] += bf16_lo(s.z);
      acc[5] += bf16_hi(s.z);
      acc[6] += bf16_lo(s.w);
      acc[7] += bf16_hi(s.w);
    }
    uint4 out;
    out.x = pack_bf16x2(acc[0], acc[1]);
    out.y = pack_bf16x2(acc[2], acc[3]);
    out.z = pack_bf16x2(acc[4], acc[5]);
    out.w = pack_bf16x2(acc[6], acc[7]);
    y[(size_t)t * vpr + v] = out;
  }
}

}  // namespace

cudaError_t launch_combine(const moe_cfg& c, const void* ebuf, const int32_t* row_of,
                           const float* topk_w, const void* shared_out, void* y,
                           uint32_t* status, cudaStream_t st, bool pdl) {
  const int vpr = c.d / 8;
  int nslice = 1;
  while (c.T * nslice < 2 * 152 && vpr / (nslice * 2) >= 128) nslice *= 2;
  const int slice_vecs = (vpr + nslice - 1) / nslice;
  nslice = (vpr + slice_vecs - 1) / slice_vecs;
  dim3 grid(c.T, nslice);
  return launch_kernel(combine_kernel, grid, dim3(128), 0, st, pdl,
                       static_cast<const uint4*>(ebuf), row_of, topk_w,
                       static_cast<const uint4*>(shared_out), static_cast<uint4*>(y), c.d, c.k,
                       slice_vecs, (long long)c.R * c.R * cap_of(c), status);
}

}  // namespace moe
