// Top-t selection without any allocation and without a caller workspace.
//
// lc_select_topt needs scratch for the order-preserving codes of the scores
// (n_heads * T * 4 bytes), which its caller passes in as a workspace.  Some
// callers cannot provide one: code that runs under a memory planner that
// hands out every buffer before serving starts and forbids allocation on the
// hot path, or a plug-in that only receives the input and output pointers of
// an already-planned graph.  This variant keeps its scratch in a fixed
// device array that is part of the library image, so it needs neither
// cudaMalloc nor a workspace.
//
// The array lives as long as the library is loaded, on every GPU that loads
// it (kNoAllocMaxScores codes, 4 MiB).  Its device address is looked up once
// per device, on the first call made with that device current; do that first
// call before any stream capture.  The address is kept together with the
// unique ID of the CUDA context it belongs to: after the device's context has
// been torn down and recreated (cudaDeviceReset), the module is loaded again
// at a new address, so the next call sees a new context ID and looks the
// address up again (that call, too, belongs before any capture).  All calls
// share the array, so calls whose
// work overlaps on the GPU (different streams, or different host threads on
// the same device) race and must be serialised by the caller.  Every call
// rewrites all the codes it reads before reading them, so nothing has to be
// cleared between calls.
#include <cuda.h>

#include <mutex>

#include "../../include/lc.h"
#include "lc_common.cuh"
#include "lc_kernels.cuh"

namespace {

constexpr size_t kNoAllocMaxScores = static_cast<size_t>(LC_NOALLOC_MAX_SCORES);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint32_t g_score_codes[kNoAllocMaxScores];

std::mutex g_mu;

// The array's address on one device and the ID of the context it belongs to.
struct Scratch {
  unsigned long long ctx_id;
  uint32_t* ptr;
};
Scratch g_scratch[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
std::once_flag g_ctx_fn_once;

// Unique ID of the current CUDA context (false if there is none or the driver
// entry points are unavailable).
bool current_context_id(unsigned long long* id) {
  std::call_once(g_ctx_fn_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<CtxGetIdFn>(fn);
  });
  if (!g_ctx_current || !g_ctx_id) return false;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_score_codes on the current device: looked up on the
// first call, and again whenever the current context is not the one the
// cached address belongs to.  Without a context ID the address is looked up
// on every call and not cached.
lc_status scratch_for_current_device(uint32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  Scratch& e = g_scratch[dev];
  unsigned long long id = 0;
  if (e.ptr && current_context_id(&id) && id == e.ctx_id) {
    *out = e.ptr;
    return LC_OK;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_score_codes) != cudaSuccess || !p) return LC_ERR_CUDA;
  if (current_context_id(&id)) e = {id, static_cast<uint32_t*>(p)};
  *out = static_cast<uint32_t*>(p);
  return LC_OK;
}

}  // namespace

extern "C" lc_status lc_select_topt_noalloc(int n_heads, int T, int t, const float* u,
                                            int32_t* idx, void* stream) {
  if (n_heads < 1 || T < 1 || t < 1 || t > T || !u || !idx) return LC_ERR_INVALID_ARG;
  if (static_cast<size_t>(n_heads) * static_cast<size_t>(T) > kNoAllocMaxScores)
    return LC_ERR_UNSUPPORTED;
  uint32_t* codes = nullptr;
  lc_status s = scratch_for_current_device(&codes);
  if (s != LC_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (lc::launch_encode_scores(u, codes, static_cast<size_t>(n_heads) * T, st) != cudaSuccess)
    return LC_ERR_CUDA;
  if (lc::launch_select_topt(codes, n_heads, T, t, idx, st) != cudaSuccess) return LC_ERR_CUDA;
  return LC_OK;
}
