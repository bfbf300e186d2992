// k3moe_noalloc.cu -- k3moe_route_noalloc: the router step with its logits
// scratch in a statically allocated device array instead of caller memory.
//
// Who needs this: callers that must not allocate device memory at the point
// where they route tokens.  Examples are code that runs while a CUDA graph
// is being captured (a cudaMalloc there fails or breaks the capture), code
// that runs inside another framework's memory pool or under a fixed memory
// budget (where a stray allocation can fail or fragment the pool), and
// embedded or latency-bound services that allow no allocation after start-up.
// They pass inputs and outputs only; the scratch comes from a file-scope
// __device__ array that every GPU loading this library holds until the
// process exits.
#include <cuda.h>

#include <cstdio>
#include <mutex>

#include "../../include/k3moe.h"
#include "k3moe_internal.h"

namespace {

// Router logits [T, E] of the most recent call: at most this many floats
// (512 KiB per device), e.g. 64 tokens x 2048 experts or 146 x 896.
constexpr size_t kNoAllocLogits = 131072;
__device__ __align__(256) float g_noalloc_logits[kNoAllocLogits];

// The array's device address belongs to one CUDA context (the module is
// loaded per context), so the cache is keyed by the current context, not
// by the device ordinal: a primary context rebuilt after cudaDeviceReset,
// or a second context on the same device, gets its own entry.  Outside
// stream capture every call asks the runtime again and refreshes the entry;
// during capture the entry of the current context is used as it stands.
constexpr int kMaxContexts = 64;
struct ScratchEntry {
  CUcontext ctx;
  float* ptr;
};
ScratchEntry g_scratch[kMaxContexts] = {};
int g_scratch_n = 0;
std::mutex g_scratch_mu;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// cuCtxGetCurrent from the driver, through the runtime's entry-point query
// (the library does not link libcuda directly).
CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

int noalloc_fail(int code, const char* msg) {
  k3::set_thread_error(msg);  // reported by k3moe_last_error(NULL)
  return code;
}

}  // namespace

extern "C" {

// See include/k3moe.h.
int k3moe_route_noalloc(const void* x, int T, const void* router_w, const float* bias, int E, int H, int K,
                        int norm_topk, float routed_scaling, int32_t* topk_idx, float* topk_w, void* cuda_stream) {
  if (T < 0) return noalloc_fail(K3MOE_EINVAL, "T < 0");
  if (T == 0) return K3MOE_OK;
  if (!x || !router_w || !bias || !topk_idx || !topk_w) return noalloc_fail(K3MOE_EINVAL, "a pointer is NULL");
  if (H <= 0 || H % 128 || K < 1 || K > 32 || K > E || E > 2048)
    return noalloc_fail(K3MOE_EINVAL, "need H % 128 == 0, 1 <= K <= 32, K <= E <= 2048");
  if ((size_t)T * (size_t)E > kNoAllocLogits)
    return noalloc_fail(K3MOE_EINVAL, "T * E exceeds the static scratch (131072 router logits)");
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(router_w) & 15u))
    return noalloc_fail(K3MOE_EINVAL, "x and router_w must be 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  // Make the current device's primary context current (cudaSetDevice
  // initialises it; a no-op when it already is), then identify it.
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess)
    return noalloc_fail(K3MOE_ECUDA, "no usable CUDA device");
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  CUcontext ctx = nullptr;
  if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS || !ctx)
    return noalloc_fail(K3MOE_ECUDA, "cuCtxGetCurrent failed");
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return noalloc_fail(K3MOE_ECUDA, "cudaStreamIsCapturing failed");
  float* scratch = nullptr;
  {
    // Set-up with the device current: the host-side name of the array is
    // not a device address, so ask the runtime for this context's copy.
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchEntry* ent = nullptr;
    for (int i = 0; i < g_scratch_n; ++i)
      if (g_scratch[i].ctx == ctx) ent = &g_scratch[i];
    if (!ent || cs == cudaStreamCaptureStatusNone) {
      if (cs != cudaStreamCaptureStatusNone)
        return noalloc_fail(K3MOE_ESTATE, "first call on this CUDA context made during stream capture; "
                                          "call once outside capture first");
      void* p = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_logits);
      if (e != cudaSuccess || !p) return noalloc_fail(K3MOE_ECUDA, "cudaGetSymbolAddress of the scratch failed");
      if (!ent) {
        if (g_scratch_n == kMaxContexts) return noalloc_fail(K3MOE_ECUDA, "too many CUDA contexts");
        ent = &g_scratch[g_scratch_n++];
        ent->ctx = ctx;
      }
      ent->ptr = static_cast<float*>(p);
    }
    scratch = ent->ptr;
  }
  cudaError_t e = k3::launch_dense_gemv(static_cast<const uint16_t*>(router_w), E, H, static_cast<const uint16_t*>(x),
                                        T, E, scratch, nullptr, s);
  if (e == cudaSuccess)
    e = k3::launch_topk(scratch, T, E, E, bias, K, norm_topk, routed_scaling, topk_idx, topk_w, s);
  if (e != cudaSuccess) return noalloc_fail(K3MOE_ECUDA, cudaGetErrorString(e));
  return K3MOE_OK;
}

}  // extern "C"
