// The step kernel for bf16 queries and caches.
#include "attn_step.cuh"

namespace cpa {
template cudaError_t launch_step<0>(const AttnParams &, const StepWs &, cudaStream_t);
}  // namespace cpa
