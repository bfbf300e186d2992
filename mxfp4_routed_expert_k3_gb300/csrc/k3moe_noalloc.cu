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
#include <cstdio>
#include <mutex>

#include "../../include/k3moe.h"
#include "k3moe_internal.h"

namespace {

// Router logits [T, E] of the most recent call: at most this many floats
// (512 KiB per device), e.g. 64 tokens x 2048 experts or 146 x 896.
constexpr size_t kNoAllocLogits = 131072;
__device__ __align__(256) float g_noalloc_logits[kNoAllocLogits];

constexpr int kMaxDevices = 64;
float* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

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
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return noalloc_fail(K3MOE_ECUDA, "cudaGetDevice failed or device ordinal too large");
  float* scratch = nullptr;
  {
    // Set-up, once per device, with that device current: the host-side
    // name of the array is not a device address, so ask the runtime.
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
      void* p = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_logits);
      if (e != cudaSuccess || !p) return noalloc_fail(K3MOE_ECUDA, "cudaGetSymbolAddress of the scratch failed");
      g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    scratch = g_scratch_ptr[dev];
  }
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  cudaError_t e = k3::launch_dense_gemv(static_cast<const uint16_t*>(router_w), E, H, static_cast<const uint16_t*>(x),
                                        T, E, scratch, nullptr, s);
  if (e == cudaSuccess)
    e = k3::launch_topk(scratch, T, E, E, bias, K, norm_topk, routed_scaling, topk_idx, topk_w, s);
  if (e != cudaSuccess) return noalloc_fail(K3MOE_ECUDA, cudaGetErrorString(e));
  return K3MOE_OK;
}

}  // extern "C"
