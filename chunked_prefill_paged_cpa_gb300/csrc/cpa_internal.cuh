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

// Workspace layout (byte offsets from desc->workspace, all 256-aligned).
// Both layouts start with a 256-byte header whose first word is the device
// status word.
//  - Row kernel (fp32 and shapes the step kernel does not take):
//      counters  uint32 [num_seqs * Hkv]      split-merge arrival counts
//      part_o / part_ml  one partial (o, (max, sum)) per (sequence, query
//                        head, split of kSplitKeys keys)
//  - Step kernel (16-bit queries, head_dim 64/128, GQA group 1/2/4/8):
//      header    status word; queue sizes, decode slice pages, ticket
//      list      the step's work queue, one 32-byte entry per item
//      dec_ctr   uint32 [num_seqs * Hkv]      decode segments' arrival counts
//      chunk_ctr uint32 [2 * chunk units]     per (tile pair, tile) counts
//      dec_o / dec_ml   one partial per decode slice: G rows x D, (max, sum)
//      chunk_o / chunk_ml  one partial per split chunk unit: two 128-row tiles
//      q16       E4M3 cache with bf16 queries: their binary16 copy [T][Hq][D]
//    Capacities, for a grid of up to kMaxStepGrid CTAs: decode slices <=
//    Hkv * num_seqs + 32 * kMaxStepGrid; chunk units <= max(kMaxStepGrid,
//    Hkv * (ceil(num_tokens * G / 256) + num_seqs)); split chunk units <=
//    kMaxStepGrid.  The plan kernel zeroes the counters and the ticket of
//    every step, so nothing but the status word carries over between calls.
struct WorkspaceLayout {
  bool step;
  size_t total;
  size_t clear;  // bytes to zero before a call on a workspace in unknown state
  // row kernel
  size_t counters, part_o, part_ml;
  int max_splits;
  // step kernel
  size_t list, dec_ctr, chunk_ctr, dec_o, dec_ml, chunk_o, chunk_ml, q16;
  int cap_dec, cap_chunk, cap_split;
};

// Keys handled by one split of a long decode in the row kernel.
constexpr int kSplitKeys = 512;
// Sequences per step on the step kernel (its plan scans them in shared memory).
constexpr int kDecodeMaxSeqs = 4096;
// Largest persistent grid of the step kernel (one CTA per SM, capped here);
// the workspace is sized for it, so its size is plain host arithmetic.
constexpr int kMaxStepGrid = 256;

// Layout for this description and at most num_seqs sequences.
WorkspaceLayout workspace_layout(const cpa_desc &d, int num_seqs);

// Device pointers into the step kernel's workspace.
struct StepWs {
  int *hdr;            // [0] chunk units, [1] decode slices, [2] items, [3] pages per slice, [4] ticket
  int *list;           // 8 ints per queue entry
  uint32_t *dec_ctr;
  uint32_t *chunk_ctr;
  float *dec_o;
  float2 *dec_ml;
  float *chunk_o;
  float2 *chunk_ml;
  int grid;            // CTAs of the step kernel (one per SM)
};

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
  // Fused append (cpa_append_attention_forward, step kernel): the step's new
  // k/v rows [num_tokens][Hkv][D] and their cache slots; the plan kernel
  // copies them into the cache before the step kernel reads it.  fused = 0:
  // the cache already holds them (cpa_kv_append ran first).
  int fused;
  const void *k_new;
  const void *v_new;
  const int64_t *slot_mapping;
  // Element types: act_f16 = q, k/v rows and out are binary16 (else bf16 on
  // the step kernel); kv_e4m3 = the caches hold E4M3 codes of K / k_scale and
  // V / v_scale; q16 = the plan kernel's binary16 copy of bf16 queries.
  int act_f16;
  int kv_e4m3;
  float k_scale, v_scale;
  void *q16;
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

// Append of new rows; `quant` 0: copy elem_bytes-wide elements; 1 / 2: E4M3
// codes of bf16 / binary16 rows divided by k_scale (K) and v_scale (V).
cudaError_t launch_kv_append(const void *k, const void *v, const int64_t *slots,
                             void *k_cache, void *v_cache, int64_t num_tokens,
                             int Hkv, int D, int page_size, int64_t num_pages,
                             int elem_bytes, int quant, float k_scale, float v_scale,
                             uint32_t *status, cudaStream_t stream);

cudaError_t launch_attention_rows(const AttnParams &p, int dtype, cudaStream_t stream);

// fp32 steps: the chunk rows (q_len > 1) on the tensor cores, kind::tf32
// (attn_chunk_tf32.cu); the decode rows then go to the row kernel (rows_mode 2).
cudaError_t launch_chunk_tf32(const AttnParams &p, cudaStream_t stream);

// Number of SMs of a device (cached); 0 if it cannot be queried.
int sm_count(int device);

// The step kernel (attn_step.cuh, one translation unit per cache mode):
// 16-bit queries, head_dim 64/128, GQA group 1/2/4/8.  KVM 0: bf16 queries and
// caches; 1: binary16 queries and caches; 2: E4M3 caches.
bool step_path(int dtype, int D, int G);
template <int KVM>
cudaError_t launch_step(const AttnParams &p, const StepWs &w, cudaStream_t stream);

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

}  // namespace cpa
