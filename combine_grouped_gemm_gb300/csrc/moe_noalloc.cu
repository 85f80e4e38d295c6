// moe_route_noalloc: the router for callers that cannot hand the library any device memory
// beyond their own inputs and outputs.
//
// Who needs it: a plugin running inside another framework that does not own (or cannot reach)
// that framework's allocator; a deployment that reserves every byte of device memory at start-
// up under a fixed memory plan; a latency-critical caller that must not enter the driver's
// allocator on the hot path (cudaMalloc/cudaFree can synchronise the whole device). Such a
// caller owns x, the gate weights, the bias and the two outputs, but has no workspace to give.
//
// The router's only scratch is its table of 16 partial dot products per (token, expert). Here
// that table lives in a file-scope device array of a fixed size, allocated with the library
// image when it is loaded on a device and held by every device that loads the library until
// the process exits. Its device address is looked up once per device context
// (cudaGetSymbolAddress with that device current) on the first call made there; make that
// first call before any stream capture begins. Every call shares the one array: the kernels write every entry they
// later read, so nothing has to be cleared between calls, but two calls whose kernels overlap
// on the GPU (different streams, or different host threads on one device) race on it.
#include <mutex>

#include "moe_internal.h"

namespace moe {
namespace {

// 8 MiB: room for 16 partials x T x E fp32 with T*E up to 131072 (e.g. 512 tokens x 256
// experts).
constexpr size_t kNoallocScratchFloats = 2u * 1024u * 1024u;
static __device__ __align__(256) float g_route_scratch[kNoallocScratchFloats];

// The array's device address belongs to the CUDA context that loaded the library's module on
// a device. It is looked up once per context (cudaGetSymbolAddress with that device current)
// and cached under the context's unique ID, so a context created after a device reset (which
// loads the module again, elsewhere) gets a fresh lookup instead of a dangling address.
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

struct ScratchEntry {
  unsigned long long ctx_id;
  float* ptr;
};
constexpr int kMaxContexts = 64;
std::mutex g_scratch_mutex;
ScratchEntry g_scratch[kMaxContexts] = {};
int g_scratch_used = 0;

// ID of the current context (0 if it cannot be read: the address is then looked up anew).
unsigned long long current_ctx_id() {
  static CtxGetIdFn get_id = nullptr;
  static CtxGetCurrentFn get_cur = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_id || !get_cur || get_cur(&ctx) != CUDA_SUCCESS || !ctx ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_route_scratch in the current context.
cudaError_t scratch_on_current_device(float** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);   // fails when no device can be used
  if (err != cudaSuccess) return err;
  (void)dev;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  unsigned long long id = current_ctx_id();   // 0 before the runtime made a context current
  if (id != 0)
    for (int i = 0; i < g_scratch_used; ++i)
      if (g_scratch[i].ctx_id == id) {
        *out = g_scratch[i].ptr;
        return cudaSuccess;
      }
  void* p = nullptr;
  err = cudaGetSymbolAddress(&p, g_route_scratch);   // makes the device's context current
  if (err != cudaSuccess) return err;
  if (id == 0) id = current_ctx_id();
  if (id != 0 && g_scratch_used < kMaxContexts)
    g_scratch[g_scratch_used++] = ScratchEntry{id, static_cast<float*>(p)};
  *out = static_cast<float*>(p);
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

extern "C" int moe_route_noalloc(const moe_cfg* cfg, const void* x, const float* w_gate,
                                 const float* bias, int32_t* topk_idx, float* topk_w,
                                 cudaStream_t stream) {
  using namespace moe;
  if (!cfg) return MOE_ERR_INVALID_ARG;
  const int rc = validate(*cfg);
  if (rc != MOE_OK) return rc;
  const void* ptrs[] = {x, w_gate, bias, topk_idx, topk_w};
  for (const void* p : ptrs) {
    if (!p) return MOE_ERR_INVALID_ARG;
    if (!aligned16(p)) return MOE_ERR_MISALIGNED;
  }
  // the partial table must fit the fixed array
  if ((size_t)kRouteChunks * (size_t)cfg->T * (size_t)cfg->E > kNoallocScratchFloats)
    return MOE_ERR_UNSUPPORTED;
  float* scratch = nullptr;
  cudaError_t err = scratch_on_current_device(&scratch);
  if (err == cudaSuccess)
    err = launch_route(*cfg, x, w_gate, bias, topk_idx, topk_w, scratch, nullptr, stream);
  return err == cudaSuccess ? MOE_OK : cuda_fail(err);
}
