// Internal declarations shared by the libcpa translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "cpa.h"

namespace cpa {

// Device status bits (OR-ed into the status word at the start of the
// workspace; host reads it with cpa_read_device_status).
enum : uint32_t {
  STATUS_BAD_PAGE = 1u,   // block_table entry outside [0, num_pages)
  STATUS_BAD_SLOT = 2u,   // slot_mapping entry >= num_pages * page_size
  STATUS_TIMEOUT = 4u,    // a bounded wait gave up
};

// Workspace layout (byte offsets from desc->workspace, all 256-aligned):
//   [0, 256)   header: uint32 status word
//   counters   uint32 [num_seqs * Hkv]   split-merge arrival counts
//   part_o     split partial outputs (float), part_ml their (max, sum) pairs.
// With the streaming decode kernel (bf16 fast path) a partial slot holds the
// G rows of one (sequence, kv head) contribution and there are
// num_seqs * Hkv + kDecodeMaxWorkers slots; otherwise the row kernel keeps
// one slot per (sequence, query head, split).
struct WorkspaceLayout {
  size_t counters, part_o, part_ml, total;
  int max_splits;
  bool fast_decode;
};

// Keys handled by one split of a long decode in the row kernel.
constexpr int kSplitKeys = 512;
// Streaming decode kernel limits.
constexpr int kDecodeMaxSeqs = 4096;
constexpr int kDecodeMaxWorkers = 4096;  // CTAs x warps of its persistent grid

WorkspaceLayout workspace_layout(const cpa_desc &d, int num_seqs);

struct AttnParams {
  const void *q;
  const void *k_cache;
  const void *v_cache;
  const int32_t *block_table;
  const int32_t *query_start_loc;
  const int32_t *seq_lens;
  void *out;
  int num_seqs;
  int num_tokens;
  int Hq, Hkv, D, page_size;
  int64_t num_pages;
  int max_pages;
  float scale_log2;          // scale * log2(e): scores live in the log2 domain
  int max_splits;
  int rows_mode;              // row kernel: 0 all tokens, 1 only q_len > 1, 2 only q_len == 1
  // Streaming decode kernel beside the chunk kernel: its first decode_early
  // CTAs start at once, the rest as the chunk kernel's chunk_grid CTAs finish.
  // The page stream is split between the two groups on the device so both end
  // about together.  0 = every CTA starts at once (even split).
  int decode_early;
  int chunk_grid;
  // Fused append (cpa_append_attention_forward): the step's new k/v rows
  // [num_tokens][Hkv][D] and their cache slots.  The attention kernels take
  // the step's own keys and values from k_new/v_new and the decode kernel also
  // writes every new row into the cache.  fused = 0: the cache already holds
  // them (cpa_kv_append ran first).
  int fused;
  const void *k_new;
  const void *v_new;
  const int64_t *slot_mapping;
  uint32_t *status;
  uint32_t *counters;
  float *part_o;
  float2 *part_ml;
};

// The step's new rows for a fused append (nullptr k: no append in this call).
struct NewRows {
  const void *k = nullptr, *v = nullptr;
  const int64_t *slots = nullptr;
};

// The attention call behind every entry point (cpa_api.cu): validates the
// arguments, optionally zeroes the first clear_bytes of the workspace on the
// stream once they pass, then launches.
int attention(const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_table, const int32_t *query_start_loc,
              const int32_t *seq_lens, int32_t num_seqs, float scale, void *out,
              void *stream, const cpa_desc *desc, const NewRows &nr, size_t clear_bytes);

cudaError_t launch_kv_append(const void *k, const void *v, const int64_t *slots,
                             void *k_cache, void *v_cache, int64_t num_tokens,
                             int Hkv, int D, int page_size, int64_t num_pages,
                             int elem_bytes, uint32_t *status, cudaStream_t stream);

cudaError_t launch_attention_rows(const AttnParams &p, int dtype, cudaStream_t stream);

// Streaming split-KV decode kernel (bf16; head_dim 64/128; GQA group 2/4/8
// with group * head_dim <= 512).
bool decode_fast_path(int dtype, int D, int G);
cudaError_t launch_attention_decode(const AttnParams &p, int grid, cudaStream_t stream);
int decode_grid(int device);

// Prefill-chunk tiles on tcgen05 (bf16; head_dim 64/128; GQA group 1/2/4/8).
bool chunk_tc_path(int dtype, int D, int G);
cudaError_t launch_attention_chunk(const AttnParams &p, int grid, cudaStream_t stream);
int chunk_grid_estimate(const AttnParams &p, int sms);

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

}  // namespace cpa
