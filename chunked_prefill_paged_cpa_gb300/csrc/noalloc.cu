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
// device address.  The real address is looked up once per device with
// cudaGetSymbolAddress and cached.
#include <mutex>

#include "cpa_internal.cuh"

namespace cpa {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[CPA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on the
// first call made on that device).  Returns nullptr on failure.
void *scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
      cudaGetLastError();  // clear the (non-sticky) error so a later call can retry
      return nullptr;
    }
    g_scratch_ptr[dev] = ptr;
  }
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace cpa

using namespace cpa;

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
    // invalid description: let the regular entry point report the exact error
    return cpa_attention_forward(q, k_cache, v_cache, block_table, query_start_loc,
                                 seq_lens, num_seqs, scale, out, stream, &d);
  }
  if (need > (size_t)CPA_NOALLOC_SCRATCH_BYTES) return CPA_ERR_WORKSPACE;
  void *scratch = scratch_for_current_device();
  if (!scratch) return CPA_ERR_CUDA;
  // The merge counters and the status word must start at zero; a previous
  // call on this device left the array as it finished (or was aborted), so
  // clear them on the caller's stream before the launch.
  const WorkspaceLayout w = workspace_layout(d, num_seqs);
  if (cudaMemsetAsync(scratch, 0, w.part_o, (cudaStream_t)stream) != cudaSuccess)
    return CPA_ERR_CUDA;
  d.workspace = scratch;
  d.workspace_bytes = CPA_NOALLOC_SCRATCH_BYTES;
  return cpa_attention_forward(q, k_cache, v_cache, block_table, query_start_loc, seq_lens,
                               num_seqs, scale, out, stream, &d);
}
