// fp32 prefill-chunk attention on the tensor cores (tcgen05.mma kind::tf32).
//
// Serves the chunk rows (q_len > 1) of fp32 steps; their decode rows stay on
// the row kernel.  One CTA per (128-row query tile of a chunk, kv head): the G
// query heads that share the kv head are packed into the tile's rows (row r:
// packed row m * 128 + r of the chunk = token (m * 128 + r) / G, head
// g * G + (m * 128 + r) % G), one thread per row.  Per 64-key KV tile:
//   - the keys' K rows and V rows are gathered from the paged cache into
//     shared memory with plain loads, V transposed (head_dim-major), so that
//     every MMA operand is K-major with a 128-byte swizzle;
//   - S = Q K^T into TMEM (M 128, N 64, K-steps of 8 along head_dim);
//   - the online softmax in registers, in the log2 domain; O in TMEM is
//     rescaled when a row's maximum moves; P (fp32) goes to shared memory;
//   - O += P V into TMEM (N = head_dim, K-steps of 8 keys).
// Each step waits for the one before: this serves a parity configuration of a
// few hundred rows, whose step is launch latency.  The tensor core rounds the
// MMA inputs to tf32 (10 mantissa bits); accumulation, softmax and the output
// stay fp32.
//
// Visibility ("vllm-learning-book 05. Chunked Prefill", section 3): row i of a
// chunk of q_len tokens whose sequence holds ctx keys in all sees keys
// 0 .. ctx - q_len + i.  The softmax runs over KV tiles incrementally
// ("Chunked Prefill 技术深度解析", section 7.2).
#include <algorithm>

#include "cpa_internal.cuh"
#include "ptx.cuh"

namespace cpa {
namespace {

constexpr int kTileRows = 128;  // query rows per tile (M)
constexpr int kTileKeys = 64;   // keys per KV tile
constexpr int kTf32Threads = 128;

template <int D>
struct Tf32Layout {
  static constexpr int Q_BYTES = kTileRows * D * 4;
  static constexpr int K_BYTES = kTileKeys * D * 4;
  static constexpr int VT_BYTES = D * kTileKeys * 4;
  static constexpr int P_BYTES = kTileRows * kTileKeys * 4;
  static constexpr int OFF_K = Q_BYTES;
  static constexpr int OFF_VT = OFF_K + K_BYTES;
  static constexpr int OFF_P = OFF_VT + VT_BYTES;
  static constexpr int SMEM = OFF_P + P_BYTES + 1024;  // + slack for the 1 KB alignment
};

// Byte offset of element (row, k) of a K-major operand of `rows` rows with a
// 128-byte swizzle: panels of 32 fp32 along k (rows x 128 B each, 1 KB
// aligned), and a row's 16-byte chunks XOR-ed with its index in its 8-row group.
__device__ __forceinline__ uint32_t sw128(int row, int k, int rows) {
  return (uint32_t)((k >> 5) * rows * 128 + row * 128 + ((((k >> 2) & 7) ^ (row & 7)) << 4) +
                    (k & 3) * 4);
}

// The chunk tile of CTA b: sequences with q_len > 1 own ceil(q_len * G / 128)
// tiles each, in sequence order.  Warp 0 scans 32 sequences at a time.
// seq = -1: no such tile (the grid is an upper bound).
template <int G>
__device__ __forceinline__ void find_tile(const AttnParams &p, int b, int lane, int &seq,
                                          int &tile) {
  seq = -1;
  tile = 0;
  int base = 0;
  for (int s0 = 0; s0 < p.num_seqs; s0 += 32) {
    const int s = s0 + lane;
    int nt = 0;
    if (s < p.num_seqs) {
      const int ql = __ldg(p.query_start_loc + s + 1) - __ldg(p.query_start_loc + s);
      if (ql > 1) nt = (int)(((int64_t)ql * G + kTileRows - 1) / kTileRows);
    }
    int incl = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int lo = base + incl - nt;
    const unsigned hit = __ballot_sync(0xffffffffu, nt > 0 && b >= lo && b < lo + nt);
    if (hit) {
      const int src = __ffs(hit) - 1;
      seq = s0 + src;
      tile = b - __shfl_sync(0xffffffffu, lo, src);
      return;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
}

template <int D, int G>
__global__ void __launch_bounds__(kTf32Threads, 1) attn_chunk_tf32_kernel(const AttnParams p) {
  using L = Tf32Layout<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char *sQ = smem, *sK = smem + L::OFF_K, *sVT = smem + L::OFF_VT, *sP = smem + L::OFF_P;
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ int s_seq, s_tile;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = blockIdx.y;

  if (warp == 0) {
    int seq, tile;
    find_tile<G>(p, blockIdx.x, lane, seq, tile);
    if (lane == 0) {
      s_seq = seq;
      s_tile = tile;
    }
  }
  __syncthreads();
  const int s = s_seq, mt = s_tile;
  if (s < 0) return;
  if (warp == 0) ptx::tmem_alloc(&tmem_base, 256);  // S: columns 0..63, O: 128..128+D-1
  if (tid == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tm = tmem_base, lane_off = (uint32_t)(warp * 32) << 16;
  const uint32_t tS = tm + lane_off, tO = tm + 128 + lane_off;

  const int qs = __ldg(p.query_start_loc + s), q_len = __ldg(p.query_start_loc + s + 1) - qs;
  int ctx = __ldg(p.seq_lens + s);
  const int cap = p.max_pages * p.page_size;
  if (ctx > cap) {  // contract violation: never read past the block-table row
    if (tid == 0) atomicOr(p.status, STATUS_BAD_PAGE);
    ctx = cap;
  }
  // this thread's row
  const int lr = mt * kTileRows + tid;
  const int tl = lr / G, t = qs + tl, h = g * G + (lr - tl * G);
  const int vis = ctx - q_len + tl + 1;  // keys the row sees
  const bool valid = tl < q_len && t < p.num_tokens && vis > 0;  // (a token past the batch: malformed)
  const int vis_row = valid ? vis : 1;   // rows without output still see key 0 (finite math)
  // keys loaded: those the tile's last row sees (at least key 0)
  const int last_tl = (int)(min((int64_t)mt * kTileRows + kTileRows - 1, (int64_t)q_len * G - 1) / G);
  const int n_keys = max(1, min(ctx - q_len + last_tl + 1, ctx));
  const int n_tiles = (n_keys + kTileKeys - 1) / kTileKeys;

  // Q tile (rows without output are zero)
  const float *q = static_cast<const float *>(p.q);
#pragma unroll 4
  for (int c = 0; c < D / 4; ++c) {
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (valid) x = __ldg(reinterpret_cast<const float4 *>(q + ((int64_t)t * p.Hq + h) * D) + c);
    *reinterpret_cast<float4 *>(sQ + sw128(tid, c * 4, kTileRows)) = x;
  }

  const float *kc = static_cast<const float *>(p.k_cache);
  const float *vc = static_cast<const float *>(p.v_cache);
  const int32_t *bt = p.block_table + (int64_t)s * p.max_pages;
  constexpr uint32_t idesc_qk = ptx::idesc_tf32_f32(kTileRows, kTileKeys);
  constexpr uint32_t idesc_pv = ptx::idesc_tf32_f32(kTileRows, D);
  float m_run = -INFINITY, l_run = 0.f;
  uint32_t phase = 0;
  bool ok = true;
  for (int j = 0; j < n_tiles; ++j) {
    // K rows and V^T of keys j*64 .. j*64+63; zero past n_keys or for a bad page
    for (int i = tid; i < kTileKeys * (D / 4); i += kTf32Threads) {
      const int n = i / (D / 4), c = i - n * (D / 4);
      const int key = j * kTileKeys + n;
      float4 kx = make_float4(0.f, 0.f, 0.f, 0.f), vx = kx;
      if (key < n_keys) {
        const int page = __ldg(bt + key / p.page_size);
        if (page >= 0 && page < p.num_pages) {
          const int64_t row = (((int64_t)page * p.Hkv + g) * p.page_size + key % p.page_size) * D;
          kx = __ldg(reinterpret_cast<const float4 *>(kc + row) + c);
          vx = __ldg(reinterpret_cast<const float4 *>(vc + row) + c);
        } else if (c == 0) {
          atomicOr(p.status, STATUS_BAD_PAGE);
        }
      }
      *reinterpret_cast<float4 *>(sK + sw128(n, c * 4, kTileKeys)) = kx;
      *reinterpret_cast<float *>(sVT + sw128(c * 4 + 0, n, D)) = vx.x;
      *reinterpret_cast<float *>(sVT + sw128(c * 4 + 1, n, D)) = vx.y;
      *reinterpret_cast<float *>(sVT + sw128(c * 4 + 2, n, D)) = vx.z;
      *reinterpret_cast<float *>(sVT + sw128(c * 4 + 3, n, D)) = vx.w;
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      ptx::tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < D / 8; ++ks) {
        const uint64_t a = ptx::smem_desc_sw128(sQ + (ks >> 2) * kTileRows * 128 + (ks & 3) * 32, 16, 1024);
        const uint64_t b = ptx::smem_desc_sw128(sK + (ks >> 2) * kTileKeys * 128 + (ks & 3) * 32, 16, 1024);
        ptx::mma_tf32_ss(tm, a, b, idesc_qk, ks > 0);
      }
      ptx::mma_commit(&bar);
    }
    ok = __syncthreads_and(ptx::mbar_wait(&bar, phase & 1)) != 0;
    ++phase;
    if (!ok) break;
    ptx::tc_fence_after();

    // softmax of this tile's scores, in the log2 domain
    uint32_t sa[32], sb[32];
    ptx::tmem_ld32(tS, sa);
    ptx::tmem_ld32(tS + 32, sb);
    ptx::tmem_wait_ld_regs(sa);
    ptx::tmem_wait_ld_regs(sb);
    const int key0 = j * kTileKeys;
    float x[kTileKeys];
    float tmax = -INFINITY;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      x[c] = key0 + c < vis_row ? __uint_as_float(sa[c]) * p.scale_log2 : -INFINITY;
      x[32 + c] = key0 + 32 + c < vis_row ? __uint_as_float(sb[c]) * p.scale_log2 : -INFINITY;
      tmax = fmaxf(tmax, fmaxf(x[c], x[32 + c]));
    }
    const float m_new = fmaxf(m_run, tmax);  // finite: every row sees key 0 in tile 0
    const float alpha = exp2f(m_run - m_new);
    float rs = 0.f;
#pragma unroll
    for (int c = 0; c < kTileKeys; ++c) {
      x[c] = exp2f(x[c] - m_new);
      rs += x[c];
    }
    l_run = l_run * alpha + rs;
    m_run = m_new;
    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        ptx::tmem_ld32(tO + c * 32, o);
        ptx::tmem_wait_ld_regs(o);
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        ptx::tmem_st32(tO + c * 32, o);
      }
      ptx::tmem_wait_st();
    }
#pragma unroll
    for (int c = 0; c < kTileKeys / 4; ++c)
      *reinterpret_cast<float4 *>(sP + sw128(tid, c * 4, kTileRows)) =
          make_float4(x[4 * c], x[4 * c + 1], x[4 * c + 2], x[4 * c + 3]);
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      ptx::tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < kTileKeys / 8; ++ks) {
        const uint64_t a = ptx::smem_desc_sw128(sP + (ks >> 2) * kTileRows * 128 + (ks & 3) * 32, 16, 1024);
        const uint64_t b = ptx::smem_desc_sw128(sVT + (ks >> 2) * D * 128 + (ks & 3) * 32, 16, 1024);
        ptx::mma_tf32_ss(tm + 128, a, b, idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
      }
      ptx::mma_commit(&bar);
    }
    ok = __syncthreads_and(ptx::mbar_wait(&bar, phase & 1)) != 0;
    ++phase;
    if (!ok) break;
    ptx::tc_fence_after();
  }

  if (ok) {
    float *out = static_cast<float *>(p.out);
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      ptx::tmem_ld32(tO + c * 32, o);
      ptx::tmem_wait_ld_regs(o);
      if (valid) {
        float *dst = out + ((int64_t)t * p.Hq + h) * D + c * 32;
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4 *>(dst + e) =
              make_float4(__uint_as_float(o[e]) / l_run, __uint_as_float(o[e + 1]) / l_run,
                          __uint_as_float(o[e + 2]) / l_run, __uint_as_float(o[e + 3]) / l_run);
      }
    }
  } else {
    // a wait gave up: flag it, and give the MMAs in flight one more bounded
    // wait before their TMEM is freed
    if (tid == 0) atomicOr(p.status, STATUS_TIMEOUT);
    ptx::mbar_wait(&bar, (phase - 1) & 1);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tm, 256);
  }
}

template <int D, int G>
cudaError_t launch_dg(const AttnParams &p, cudaStream_t stream) {
  using L = Tf32Layout<D>;
  cudaError_t e = cudaFuncSetAttribute(attn_chunk_tf32_kernel<D, G>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
  if (e != cudaSuccess) return e;
  // upper bound on the chunk tiles: every chunk has at least two tokens
  const int64_t tiles = ((int64_t)p.num_tokens * G + kTileRows - 1) / kTileRows +
                        std::min<int64_t>(p.num_seqs, p.num_tokens / 2);
  if (tiles > INT32_MAX) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)tiles, (unsigned)p.Hkv);
  attn_chunk_tf32_kernel<D, G><<<grid, kTf32Threads, L::SMEM, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const AttnParams &p, cudaStream_t stream) {
  switch (p.Hq / p.Hkv) {
    case 1: return launch_dg<D, 1>(p, stream);
    case 2: return launch_dg<D, 2>(p, stream);
    case 4: return launch_dg<D, 4>(p, stream);
    case 8: return launch_dg<D, 8>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_chunk_tf32(const AttnParams &p, cudaStream_t stream) {
  if (p.num_tokens < 2) return cudaSuccess;  // no chunk in the step
  if (p.D == 64) return launch_d<64>(p, stream);
  if (p.D == 128) return launch_d<128>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace cpa
