// C ABI of libcpa: argument validation, workspace layout and launches.
// Declared and documented in include/cpa.h.
#include <algorithm>

#include "cpa_internal.cuh"

namespace cpa {

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The persistent step kernel takes every supported shape with 16-bit queries;
// fp32 runs on the row kernel.
bool step_path(int dtype, int D, int G) {
  if (dtype != CPA_BF16 && dtype != CPA_F16) return false;
  if (D != 64 && D != 128) return false;
  return G == 1 || G == 2 || G == 4 || G == 8;
}

int sm_count(int device) {
  static int sms[64] = {};
  if (device < 0 || device >= 64) return 0;
  if (!sms[device]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    sms[device] = n;
  }
  return sms[device];
}

WorkspaceLayout workspace_layout(const cpa_desc &d, int num_seqs) {
  WorkspaceLayout w{};
  const int G = d.num_q_heads / d.num_kv_heads;
  const int Hkv = d.num_kv_heads, D = d.head_dim;
  w.step = step_path(d.dtype, D, G);
  size_t off = 256;  // header
  if (!w.step) {
    const int64_t max_keys = (int64_t)d.max_pages_per_seq * d.page_size;
    w.max_splits = (int)((max_keys + kSplitKeys - 1) / kSplitKeys);
    if (w.max_splits < 1) w.max_splits = 1;
    w.counters = off;
    off = align_up(off + sizeof(uint32_t) * (size_t)num_seqs * Hkv, 256);
    w.part_o = off;
    const size_t rows = (size_t)num_seqs * d.num_q_heads * w.max_splits;
    off = align_up(off + sizeof(float) * rows * D, 256);
    w.part_ml = off;
    off = align_up(off + sizeof(float2) * rows, 256);
    w.total = off;
    w.clear = 256;  // the status word; every call zeroes its counters itself
    return w;
  }
  // capacities for a persistent grid of up to kMaxStepGrid CTAs (one per SM)
  const int64_t tok = d.num_tokens > 0 ? d.num_tokens : 0;
  w.cap_dec = Hkv * num_seqs + 32 * kMaxStepGrid;
  w.cap_chunk = (int)std::max<int64_t>(kMaxStepGrid,
                                       (int64_t)Hkv * ((tok * G + 255) / 256 + num_seqs));
  w.cap_split = kMaxStepGrid;
  w.list = off;
  off = align_up(off + (size_t)32 * (w.cap_dec + w.cap_chunk), 256);
  w.dec_ctr = off;
  off = align_up(off + sizeof(uint32_t) * (size_t)num_seqs * Hkv, 256);
  w.chunk_ctr = off;
  off = align_up(off + sizeof(uint32_t) * 2 * (size_t)w.cap_chunk, 256);
  w.dec_o = off;
  off = align_up(off + sizeof(float) * (size_t)w.cap_dec * G * D, 256);
  w.dec_ml = off;
  off = align_up(off + sizeof(float2) * (size_t)w.cap_dec * G, 256);
  w.chunk_o = off;
  off = align_up(off + sizeof(float) * (size_t)w.cap_split * 2 * 128 * D, 256);
  w.chunk_ml = off;
  off = align_up(off + sizeof(float2) * (size_t)w.cap_split * 2 * 128, 256);
  if (d.kv_dtype == CPA_KV_E4M3 && d.dtype == CPA_BF16) {
    w.q16 = off;
    off = align_up(off + 2 * (size_t)tok * d.num_q_heads * D, 256);
  }
  w.total = off;
  w.clear = 256;  // the status word; the plan kernel zeroes the rest it uses
  return w;
}

// Shape checks shared by both calls.
static int check_shape(const cpa_desc *d) {
  if (!d) return CPA_ERR_ARG;
  if (d->num_q_heads <= 0 || d->num_kv_heads <= 0 || d->head_dim <= 0 ||
      d->page_size <= 0 || d->num_pages <= 0 || d->num_tokens < 0)
    return CPA_ERR_ARG;
  if (d->num_q_heads % d->num_kv_heads != 0) return CPA_ERR_ARG;
  if (d->dtype != CPA_F32 && d->dtype != CPA_BF16 && d->dtype != CPA_F16)
    return CPA_ERR_UNSUPPORTED;
  if (d->kv_dtype != CPA_KV_SAME && d->kv_dtype != CPA_KV_E4M3) return CPA_ERR_UNSUPPORTED;
  if (d->kv_dtype == CPA_KV_E4M3) {
    if (d->dtype == CPA_F32) return CPA_ERR_UNSUPPORTED;  // 16-bit queries only
    const float ks = d->k_scale, vs = d->v_scale;
    if (!(ks > 0.f) || !(vs > 0.f) || ks > 3.0e38f || vs > 3.0e38f) return CPA_ERR_ARG;
  }
  if (d->head_dim != 64 && d->head_dim != 128) return CPA_ERR_UNSUPPORTED;
  if (d->page_size != 16) return CPA_ERR_UNSUPPORTED;
  const int G = d->num_q_heads / d->num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return CPA_ERR_UNSUPPORTED;
  if (d->num_tokens > INT32_MAX / 2) return CPA_ERR_UNSUPPORTED;
  return CPA_OK;
}

static bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace cpa

using namespace cpa;

extern "C" const char *cpa_status_string(int status) {
  switch (status) {
    case CPA_OK: return "CPA_OK";
    case CPA_ERR_ARG: return "CPA_ERR_ARG: malformed argument";
    case CPA_ERR_UNSUPPORTED: return "CPA_ERR_UNSUPPORTED: shape or dtype not supported";
    case CPA_ERR_WORKSPACE: return "CPA_ERR_WORKSPACE: workspace missing, misaligned or too small";
    case CPA_ERR_CUDA: return "CPA_ERR_CUDA: CUDA runtime or launch error";
    case CPA_ERR_DEVICE: return "CPA_ERR_DEVICE: a kernel met an out-of-range index";
    default: return "unknown cpa_status";
  }
}

extern "C" size_t cpa_workspace_bytes(const cpa_desc *desc, int32_t num_seqs) {
  if (check_shape(desc) != CPA_OK || num_seqs < 0 || desc->max_pages_per_seq <= 0) return 0;
  return workspace_layout(*desc, num_seqs).total;
}

extern "C" int cpa_kv_append(const void *k, const void *v, const int64_t *slot_mapping,
                             void *k_cache, void *v_cache, const cpa_desc *desc,
                             void *stream) {
  int rc = check_shape(desc);
  if (rc != CPA_OK) return rc;
  if (desc->num_tokens == 0) return CPA_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return CPA_ERR_ARG;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8))
    return CPA_ERR_ARG;
  uint32_t *status = nullptr;
  if (desc->workspace) {
    if (!aligned(desc->workspace, 256) || desc->workspace_bytes < 256) return CPA_ERR_WORKSPACE;
    status = static_cast<uint32_t *>(desc->workspace);
  }
  const int eb = desc->dtype == CPA_F32 ? 4 : 2;
  const int quant = desc->kv_dtype == CPA_KV_E4M3 ? (desc->dtype == CPA_F16 ? 2 : 1) : 0;
  cudaError_t e = launch_kv_append(k, v, slot_mapping, k_cache, v_cache, desc->num_tokens,
                                   desc->num_kv_heads, desc->head_dim, desc->page_size,
                                   desc->num_pages, eb, quant, desc->k_scale, desc->v_scale,
                                   status, (cudaStream_t)stream);
  return e == cudaSuccess ? CPA_OK : CPA_ERR_CUDA;
}

namespace cpa {

// Attention over the packed batch; with `nr.k` set the append of the step's
// new rows is part of the call (fused into the attention kernels where they
// take the shape, else one append launch ahead of them on the same stream).
// With clear_bytes > 0 the first clear_bytes of the workspace are zeroed on
// the stream once every argument has passed its checks, just before the
// first launch (a call that is rejected or has nothing to do leaves the
// workspace untouched).
int attention(const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_table, const int32_t *query_start_loc,
              const int32_t *seq_lens, int32_t num_seqs, float scale, void *out,
              void *stream, const cpa_desc *desc, const NewRows &nr, size_t clear_bytes) {
  int rc = check_shape(desc);
  if (rc != CPA_OK) return rc;
  if (num_seqs < 0) return CPA_ERR_ARG;
  if (num_seqs == 0 || desc->num_tokens == 0) return CPA_OK;
  if (desc->num_tokens < num_seqs) return CPA_ERR_ARG;  // every sequence has q_len >= 1
  if (!q || !k_cache || !v_cache || !block_table || !query_start_loc || !seq_lens || !out)
    return CPA_ERR_ARG;
  if (desc->max_pages_per_seq <= 0) return CPA_ERR_ARG;
  if (!(scale > 0.f) || scale != scale) return CPA_ERR_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(block_table, 4) || !aligned(query_start_loc, 4) || !aligned(seq_lens, 4))
    return CPA_ERR_ARG;
  const WorkspaceLayout w = workspace_layout(*desc, num_seqs);
  if (!desc->workspace || !aligned(desc->workspace, 256) || desc->workspace_bytes < w.total)
    return CPA_ERR_WORKSPACE;
  char *ws = static_cast<char *>(desc->workspace);

  AttnParams p{};
  p.q = q;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_table = block_table;
  p.query_start_loc = query_start_loc;
  p.seq_lens = seq_lens;
  p.out = out;
  p.num_seqs = num_seqs;
  p.num_tokens = (int)desc->num_tokens;
  p.Hq = desc->num_q_heads;
  p.Hkv = desc->num_kv_heads;
  p.D = desc->head_dim;
  p.page_size = desc->page_size;
  p.num_pages = desc->num_pages;
  p.max_pages = desc->max_pages_per_seq;
  p.act_f16 = desc->dtype == CPA_F16;
  p.kv_e4m3 = desc->kv_dtype == CPA_KV_E4M3;
  p.k_scale = p.kv_e4m3 ? desc->k_scale : 1.f;
  p.v_scale = p.kv_e4m3 ? desc->v_scale : 1.f;
  // scores live in the log2 domain; an E4M3 cache's K scale folds in here
  p.scale_log2 = scale * p.k_scale * 1.4426950408889634f;
  if (!(p.scale_log2 > 0.f) || p.scale_log2 > 3.0e38f) return CPA_ERR_ARG;
  p.max_splits = w.max_splits;
  p.status = reinterpret_cast<uint32_t *>(ws);
  cudaStream_t st = (cudaStream_t)stream;
  int grid = 0;
  if (w.step) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CPA_ERR_CUDA;
    grid = std::min(sm_count(dev), kMaxStepGrid);
    if (grid <= 0) return CPA_ERR_CUDA;
    if (num_seqs > kDecodeMaxSeqs) return CPA_ERR_UNSUPPORTED;
    // tensor-map row coordinates and page-stream offsets are 32-bit
    if ((int64_t)p.num_pages * p.Hkv * p.page_size >= INT32_MAX) return CPA_ERR_UNSUPPORTED;
    if ((int64_t)num_seqs * p.Hkv * p.max_pages > INT32_MAX) return CPA_ERR_UNSUPPORTED;
  }
  if (clear_bytes > 0) {
    if (clear_bytes > desc->workspace_bytes) return CPA_ERR_WORKSPACE;
    if (cudaMemsetAsync(desc->workspace, 0, clear_bytes, st) != cudaSuccess) return CPA_ERR_CUDA;
  }
  if (w.step) {
    // One launch pair for the whole step: the plan (with the append when it
    // is fused into the call), then the persistent step kernel.
    StepWs sw{};
    sw.hdr = reinterpret_cast<int *>(ws + 64);
    sw.list = reinterpret_cast<int *>(ws + w.list);
    sw.dec_ctr = reinterpret_cast<uint32_t *>(ws + w.dec_ctr);
    sw.chunk_ctr = reinterpret_cast<uint32_t *>(ws + w.chunk_ctr);
    sw.dec_o = reinterpret_cast<float *>(ws + w.dec_o);
    sw.dec_ml = reinterpret_cast<float2 *>(ws + w.dec_ml);
    sw.chunk_o = reinterpret_cast<float *>(ws + w.chunk_o);
    sw.chunk_ml = reinterpret_cast<float2 *>(ws + w.chunk_ml);
    sw.grid = grid;
    if (nr.k) {
      p.fused = 1;
      p.k_new = nr.k;
      p.v_new = nr.v;
      p.slot_mapping = nr.slots;
    }
    if (w.q16) p.q16 = ws + w.q16;
    cudaError_t e;
    if (p.kv_e4m3) e = launch_step<2>(p, sw, st);
    else if (p.act_f16) e = launch_step<1>(p, sw, st);
    else e = launch_step<0>(p, sw, st);
    return e == cudaSuccess ? CPA_OK : CPA_ERR_CUDA;
  }
  // row kernel: the append (if any) first, on the same stream
  if (nr.k) {
    // fp32 only (every 16-bit shape runs on the step kernel): a plain copy
    if (launch_kv_append(nr.k, nr.v, nr.slots, const_cast<void *>(k_cache),
                         const_cast<void *>(v_cache), desc->num_tokens, p.Hkv, p.D,
                         p.page_size, p.num_pages, 4, 0, 1.f, 1.f, p.status, st) != cudaSuccess)
      return CPA_ERR_CUDA;
  }
  // the split-merge counters start at zero in every call, whatever an earlier
  // call (one that gave up a bounded wait, say) or the caller left there
  if (cudaMemsetAsync(ws + w.counters, 0, w.part_o - w.counters, st) != cudaSuccess)
    return CPA_ERR_CUDA;
  p.counters = reinterpret_cast<uint32_t *>(ws + w.counters);
  p.part_o = reinterpret_cast<float *>(ws + w.part_o);
  p.part_ml = reinterpret_cast<float2 *>(ws + w.part_ml);
  p.rows_mode = 0;
  if (desc->dtype == CPA_F32) {
    // the chunk rows on the tensor cores (tf32), the decode rows on the row kernel
    if (launch_chunk_tf32(p, st) != cudaSuccess) return CPA_ERR_CUDA;
    p.rows_mode = 2;
  }
  return launch_attention_rows(p, desc->dtype, st) == cudaSuccess ? CPA_OK : CPA_ERR_CUDA;
}

}  // namespace cpa

extern "C" int cpa_attention_forward(const void *q, const void *k_cache, const void *v_cache,
                                     const int32_t *block_table,
                                     const int32_t *query_start_loc, const int32_t *seq_lens,
                                     int32_t num_seqs, float scale, void *out, void *stream,
                                     const cpa_desc *desc) {
  return attention(q, k_cache, v_cache, block_table, query_start_loc, seq_lens, num_seqs, scale,
                   out, stream, desc, NewRows{}, 0);
}

extern "C" int cpa_append_attention_forward(const void *q, const void *k, const void *v,
                                            const int64_t *slot_mapping, void *k_cache,
                                            void *v_cache, const int32_t *block_table,
                                            const int32_t *query_start_loc,
                                            const int32_t *seq_lens, int32_t num_seqs,
                                            float scale, void *out, void *stream,
                                            const cpa_desc *desc) {
  int rc = check_shape(desc);
  if (rc != CPA_OK) return rc;
  if (num_seqs < 0) return CPA_ERR_ARG;
  if (num_seqs == 0 || desc->num_tokens == 0) return CPA_OK;
  if (!k || !v || !slot_mapping) return CPA_ERR_ARG;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(slot_mapping, 8)) return CPA_ERR_ARG;
  NewRows nr;
  nr.k = k;
  nr.v = v;
  nr.slots = slot_mapping;
  return attention(q, k_cache, v_cache, block_table, query_start_loc, seq_lens, num_seqs, scale,
                   out, stream, desc, nr, 0);
}

extern "C" int cpa_read_device_status(const cpa_desc *desc, void *stream, int32_t *status_out) {
  if (!desc || !desc->workspace || !status_out) return CPA_ERR_ARG;
  if (!aligned(desc->workspace, 256) || desc->workspace_bytes < 256) return CPA_ERR_WORKSPACE;
  uint32_t word = 0;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&word, desc->workspace, sizeof word, cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return CPA_ERR_CUDA;
  if (cudaMemsetAsync(desc->workspace, 0, sizeof word, s) != cudaSuccess) return CPA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return CPA_ERR_CUDA;
  *status_out = word ? CPA_ERR_DEVICE : CPA_OK;
  return CPA_OK;
}
