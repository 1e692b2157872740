// The step kernel for binary16 queries and caches.
#include "attn_step.cuh"

namespace cpa {
template cudaError_t launch_step<1>(const AttnParams &, const StepWs &, cudaStream_t);
}  // namespace cpa
