// The step kernel for caches of OCP FP8 E4M3 codes (bf16 or binary16 queries).
#include "attn_step.cuh"

namespace cpa {
template cudaError_t launch_step<2>(const AttnParams &, const StepWs &, cudaStream_t);
}  // namespace cpa
