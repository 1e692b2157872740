// Row attention: one CTA per (query token, kv head, KV split), CUDA cores.
//
// A CTA computes the G query heads that share kv head g (GQA group) for one
// packed token against the keys [k0, k1) of one split of its visible range.
// It serves every decode of a step (q_len == 1; long contexts are split over
// the KV axis and merged in the same launch by the last-arriving split), and
// the rows of prefill chunks that have no tensor-core tile path.
//
// Visibility ("vllm-learning-book 05. Chunked Prefill", section 3): row i of a
// sequence with q_len new tokens and ctx cached tokens sees keys
// 0 .. ctx - q_len + i.  Softmax is computed online in the log2 domain and
// pieces are combined with log-sum-exp weights ("Chunked Prefill 技术深度解析",
// section 7.2, incremental softmax).
#include "cpa_internal.cuh"

namespace cpa {
namespace {

constexpr int kWarps = 4;

template <typename Elem, int DL>
struct RowLoad;

template <>
struct RowLoad<float, 2> {
  __device__ static void load(const float *p, float (&x)[2]) {
    float2 v = __ldg(reinterpret_cast<const float2 *>(p));
    x[0] = v.x; x[1] = v.y;
  }
};
template <>
struct RowLoad<float, 4> {
  __device__ static void load(const float *p, float (&x)[4]) {
    float4 v = __ldg(reinterpret_cast<const float4 *>(p));
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  }
};
template <>
struct RowLoad<__nv_bfloat16, 2> {
  __device__ static void load(const __nv_bfloat16 *p, float (&x)[2]) {
    uint32_t w = __ldg(reinterpret_cast<const unsigned int *>(p));
    x[0] = bf16_lo(w); x[1] = bf16_hi(w);
  }
};
template <>
struct RowLoad<__nv_bfloat16, 4> {
  __device__ static void load(const __nv_bfloat16 *p, float (&x)[4]) {
    uint2 w = __ldg(reinterpret_cast<const uint2 *>(p));
    x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
  }
};

__device__ __forceinline__ void store_out(float *p, float v) { *p = v; }
__device__ __forceinline__ void store_out(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ int owner_seq(const int32_t *qsl, int num_seqs, int t) {
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(qsl + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <typename Elem, int D, int G>
__global__ void __launch_bounds__(kWarps * 32)
attn_rows_kernel(const AttnParams p) {
  constexpr int DL = D / 32;
  const int t = blockIdx.x, g = blockIdx.y, split = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int s = owner_seq(p.query_start_loc, p.num_seqs, t);
  const int qs = __ldg(p.query_start_loc + s);
  const int q_len = __ldg(p.query_start_loc + s + 1) - qs;
  if (t - qs >= q_len) return;  // token past query_start_loc[num_seqs]: not owned
  if ((q_len == 1 && p.rows_mode == 1) || (q_len > 1 && p.rows_mode == 2)) return;
  int ctx = __ldg(p.seq_lens + s);
  const int cap = p.max_pages * p.page_size;
  if (ctx > cap) {  // contract violation: never read past the block table row
    if (threadIdx.x == 0) atomicOr(p.status, STATUS_BAD_PAGE);
    ctx = cap;
  }
  const int vis = ctx - q_len + (t - qs) + 1;
  if (vis <= 0) return;  // malformed row (q_len > ctx); host contract forbids it
  int nsplit = 1;
  if (q_len == 1) {
    nsplit = (vis + kSplitKeys - 1) / kSplitKeys;
    if (nsplit > p.max_splits) nsplit = p.max_splits;
  }
  if (split >= nsplit) return;
  const int per = (nsplit == 1) ? vis : kSplitKeys;
  const int k0 = split * per;
  const int k1 = (split == nsplit - 1) ? vis : k0 + per;

  const Elem *q = static_cast<const Elem *>(p.q);
  const Elem *kc = static_cast<const Elem *>(p.k_cache);
  const Elem *vc = static_cast<const Elem *>(p.v_cache);
  const int32_t *bt = p.block_table + (int64_t)s * p.max_pages;

  float qr[G][DL];
#pragma unroll
  for (int gh = 0; gh < G; ++gh) {
    RowLoad<Elem, DL>::load(q + ((int64_t)t * p.Hq + g * G + gh) * D + lane * DL, qr[gh]);
#pragma unroll
    for (int e = 0; e < DL; ++e) qr[gh][e] *= p.scale_log2;
  }

  float m[G], l[G], o[G][DL];
#pragma unroll
  for (int gh = 0; gh < G; ++gh) {
    m[gh] = -INFINITY;
    l[gh] = 0.f;
#pragma unroll
    for (int e = 0; e < DL; ++e) o[gh][e] = 0.f;
  }

  for (int j = k0 + warp; j < k1; j += kWarps) {
    const int page = __ldg(bt + j / p.page_size);
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0) atomicOr(p.status, STATUS_BAD_PAGE);
      continue;
    }
    const int64_t row = (((int64_t)page * p.Hkv + g) * p.page_size + (j % p.page_size)) * D;
    float kx[DL], vx[DL];
    RowLoad<Elem, DL>::load(kc + row + lane * DL, kx);
    RowLoad<Elem, DL>::load(vc + row + lane * DL, vx);
#pragma unroll
    for (int gh = 0; gh < G; ++gh) {
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < DL; ++e) dot = fmaf(qr[gh][e], kx[e], dot);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      const float m_new = fmaxf(m[gh], dot);
      const float alpha = exp2f(m[gh] - m_new);
      const float pj = exp2f(dot - m_new);
      l[gh] = l[gh] * alpha + pj;
#pragma unroll
      for (int e = 0; e < DL; ++e) o[gh][e] = fmaf(o[gh][e], alpha, pj * vx[e]);
      m[gh] = m_new;
    }
  }

  // combine the warps' partial softmax states
  __shared__ float sm_m[kWarps][G], sm_l[kWarps][G];
  __shared__ float sm_o[kWarps][G][D];
#pragma unroll
  for (int gh = 0; gh < G; ++gh) {
    if (lane == 0) { sm_m[warp][gh] = m[gh]; sm_l[warp][gh] = l[gh]; }
#pragma unroll
    for (int e = 0; e < DL; ++e) sm_o[warp][gh][lane * DL + e] = o[gh][e];
  }
  __syncthreads();

  Elem *out = static_cast<Elem *>(p.out);
  for (int idx = threadIdx.x; idx < G * D; idx += kWarps * 32) {
    const int gh = idx / D, d = idx - gh * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][gh]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float a = exp2f(sm_m[w][gh] - M);
      L = fmaf(sm_l[w][gh], a, L);
      O = fmaf(sm_o[w][gh][d], a, O);
    }
    const int h = g * G + gh;
    if (nsplit == 1) {
      store_out(out + ((int64_t)t * p.Hq + h) * D + d, O / L);
    } else {
      const int64_t slot = ((int64_t)s * p.Hq + h) * p.max_splits + split;
      p.part_o[slot * D + d] = O;
      if (d == 0) p.part_ml[slot] = make_float2(M, L);
    }
  }
  if (nsplit == 1) return;

  // last-arriving split of this (sequence, kv head) merges all splits
  __shared__ int is_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(p.counters + (int64_t)s * p.Hkv + g, 1u);
    is_last = (prev == (unsigned)(nsplit - 1));
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int idx = threadIdx.x; idx < G * D; idx += kWarps * 32) {
    const int gh = idx / D, d = idx - gh * D;
    const int h = g * G + gh;
    const int64_t base = ((int64_t)s * p.Hq + h) * p.max_splits;
    float M = -INFINITY;
    for (int k = 0; k < nsplit; ++k) M = fmaxf(M, __ldcg(&p.part_ml[base + k].x));
    float L = 0.f, O = 0.f;
    for (int k = 0; k < nsplit; ++k) {
      const float2 ml = __ldcg(&p.part_ml[base + k]);
      const float a = exp2f(ml.x - M);
      L = fmaf(ml.y, a, L);
      O = fmaf(__ldcg(&p.part_o[(base + k) * D + d]), a, O);
    }
    store_out(out + ((int64_t)t * p.Hq + h) * D + d, O / L);
  }
  if (threadIdx.x == 0) p.counters[(int64_t)s * p.Hkv + g] = 0u;  // ready for next launch
}

template <typename Elem, int D>
cudaError_t launch_d(const AttnParams &p, cudaStream_t stream) {
  const dim3 grid(p.num_tokens, p.Hkv, p.rows_mode == 1 ? 1 : p.max_splits);
  switch (p.Hq / p.Hkv) {
    case 1: attn_rows_kernel<Elem, D, 1><<<grid, kWarps * 32, 0, stream>>>(p); break;
    case 2: attn_rows_kernel<Elem, D, 2><<<grid, kWarps * 32, 0, stream>>>(p); break;
    case 4: attn_rows_kernel<Elem, D, 4><<<grid, kWarps * 32, 0, stream>>>(p); break;
    case 8: attn_rows_kernel<Elem, D, 8><<<grid, kWarps * 32, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_rows(const AttnParams &p, int dtype, cudaStream_t stream) {
  if (p.num_tokens == 0) return cudaSuccess;
  if (dtype == CPA_F32) {
    return p.D == 64 ? launch_d<float, 64>(p, stream) : launch_d<float, 128>(p, stream);
  }
  return p.D == 64 ? launch_d<__nv_bfloat16, 64>(p, stream)
                   : launch_d<__nv_bfloat16, 128>(p, stream);
}

}  // namespace cpa
