// cpa_attention_forward_noalloc: the attention step for callers that cannot
// allocate device memory.
//
// Some callers are not allowed to call cudaMalloc: a plugin inside a host
// runtime that owns every device buffer and hands the plugin only its inputs
// and outputs; a serving loop that forbids allocation after start-up because
// cudaMalloc/cudaFree can synchronise the device and may fail under memory
// pressure in the middle of a step.  Such callers cannot provide the scratch
// workspace that cpa_attention_forward needs, so this entry point keeps that
// scratch in a fixed array compiled into the library instead.
//
// The array below lives in the device memory of every GPU that loads the
// library, for as long as the process runs.  Host code must not hand the
// array's name to a kernel: on the host that name is only a stand-in, not a
// device address.  The real address is looked up with cudaGetSymbolAddress
// on every call, for the device and context current at that moment: a cached
// address would go stale when the module is loaded again (after
// cudaDeviceReset, or in another context on the same device).  The lookup is
// host-side and allocates nothing; only the first one in a context may have to
// load the module, which is why the first call belongs before any stream
// capture.
#include "cpa_internal.cuh"

namespace cpa {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[CPA_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch array in the current context, or nullptr.
void *scratch_for_current_context() {
  void *ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
    cudaGetLastError();  // clear the (non-sticky) error so a later call can retry
    return nullptr;
  }
  return ptr;
}

}  // namespace
}  // namespace cpa

using namespace cpa;

extern "C" size_t cpa_noalloc_scratch_bytes(void) { return CPA_NOALLOC_SCRATCH_BYTES; }

extern "C" int cpa_attention_forward_noalloc(const void *q, const void *k_cache,
                                             const void *v_cache, const int32_t *block_table,
                                             const int32_t *query_start_loc,
                                             const int32_t *seq_lens, int32_t num_seqs,
                                             float scale, void *out, void *stream,
                                             const cpa_desc *desc) {
  if (!desc || num_seqs < 0) return CPA_ERR_ARG;
  // the scratch replaces the caller's workspace: size it, check the limit
  cpa_desc d = *desc;
  d.workspace = nullptr;
  d.workspace_bytes = 0;
  const size_t need = cpa_workspace_bytes(&d, num_seqs);
  if (need == 0) {
    // invalid description: the regular checks report the exact error
    return attention(q, k_cache, v_cache, block_table, query_start_loc, seq_lens, num_seqs,
                     scale, out, stream, &d, NewRows{}, 0);
  }
  if (need > (size_t)CPA_NOALLOC_SCRATCH_BYTES) return CPA_ERR_WORKSPACE;
  void *scratch = scratch_for_current_context();
  if (!scratch) return CPA_ERR_CUDA;
  d.workspace = scratch;
  d.workspace_bytes = CPA_NOALLOC_SCRATCH_BYTES;
  // The status word starts at zero in every no-alloc call (the word reports
  // this call only); the work queue and merge counters are reset by the call
  // itself.  The clear runs on the caller's stream only once the call has
  // passed every check, right before its first launch.
  const WorkspaceLayout w = workspace_layout(d, num_seqs);
  return attention(q, k_cache, v_cache, block_table, query_start_loc, seq_lens, num_seqs,
                   scale, out, stream, &d, NewRows{}, w.clear);
}

extern "C" int cpa_noalloc_read_device_status(void *stream, int32_t *status_out) {
  if (!status_out) return CPA_ERR_ARG;
  void *scratch = scratch_for_current_context();
  if (!scratch) return CPA_ERR_CUDA;
  uint32_t word = 0;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&word, scratch, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return CPA_ERR_CUDA;
  if (cudaMemsetAsync(scratch, 0, sizeof word, s) != cudaSuccess) return CPA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return CPA_ERR_CUDA;
  *status_out = word ? CPA_ERR_DEVICE : CPA_OK;
  return CPA_OK;
}
