// k3moe_umma.cu -- tensor-core path (tcgen05 + TMEM + TMA).
#include "k3moe_umma.h"

namespace k3 {

UmmaPlan umma_plan(const Dims&, int) { return UmmaPlan{}; }
bool umma_path_enabled(const UmmaPlan& p, const Dims&, int T) { return p.enabled && T >= p.min_tokens; }
cudaError_t umma_dense(const UmmaPlan&, const uint16_t*, int, int, const uint16_t*, int, int, float*, uint16_t*,
                       cudaStream_t) {
  return cudaErrorNotSupported;
}
int umma_dense_launches() { return 1; }
cudaError_t umma_experts(const UmmaPlan&, const uint8_t*, const uint8_t*, const Work&, int, const Dims&,
                         cudaStream_t) {
  return cudaErrorNotSupported;
}
int umma_expert_launches() { return 2; }

}  // namespace k3
