// KV append: scatter the step's new K/V rows into their cache slots.
//
// "Chunked Prefill on an M5 Max", section "Wiring it into the loop": each
// chunk extends the KV cache instead of rebuilding it, and appending is part
// of a chunk's fixed cost.  "Chunked Prefill 技术深度解析", section 4.2: the
// cache is made of 16-token pages.  The copy is a pure byte move, so it is
// bit-exact; an E4M3 cache stores instead each element's code of x / scale
// (one correctly rounded binary32 division, then round to nearest even with
// saturation at +-448), so it too is exactly defined.
//
// Layout: k, v [T][Hkv][D]; caches [num_pages][Hkv][page_size][D].  One
// thread moves one 16-byte chunk of one (token, kv head) row of K and the
// matching chunk of V, so a warp covers 512 contiguous source bytes and
// 256-byte contiguous destination rows.
#include "cpa_internal.cuh"
#include "ptx.cuh"

namespace cpa {

// QUANT 0: copy; 1 / 2: bf16 / binary16 rows to E4M3 codes (8 per 16 bytes in).
template <int QUANT>
__global__ void __launch_bounds__(256)
kv_append_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                 const int64_t *__restrict__ slots, void *__restrict__ k_cache,
                 void *__restrict__ v_cache, int64_t num_tokens, int Hkv,
                 int chunks_per_row, int page_size, int64_t num_slots,
                 float k_scale, float v_scale, uint32_t *status) {
  const int64_t total = num_tokens * Hkv * chunks_per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / chunks_per_row;          // t * Hkv + g
    const int c = (int)(i - row * chunks_per_row);
    const int64_t t = row / Hkv;
    const int g = (int)(row - t * Hkv);
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (status && c == 0) atomicOr(status, STATUS_BAD_SLOT);
      continue;
    }
    const int64_t page = slot / page_size;
    const int64_t off = slot - page * page_size;
    const int64_t dst = ((page * Hkv + g) * page_size + off) * chunks_per_row + c;
    if (QUANT == 0) {
      static_cast<uint4 *>(k_cache)[dst] = __ldg(k + i);
      static_cast<uint4 *>(v_cache)[dst] = __ldg(v + i);
    } else {
      static_cast<uint2 *>(k_cache)[dst] = ptx::quantise8_e4m3<QUANT == 2>(__ldg(k + i), k_scale);
      static_cast<uint2 *>(v_cache)[dst] = ptx::quantise8_e4m3<QUANT == 2>(__ldg(v + i), v_scale);
    }
  }
}

cudaError_t launch_kv_append(const void *k, const void *v, const int64_t *slots,
                             void *k_cache, void *v_cache, int64_t num_tokens,
                             int Hkv, int D, int page_size, int64_t num_pages,
                             int elem_bytes, int quant, float k_scale, float v_scale,
                             uint32_t *status, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int chunks_per_row = D * elem_bytes / 16;  // 16-byte pieces of an input row
  const int64_t total = num_tokens * Hkv * chunks_per_row;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 4096) blocks = 4096;
  auto kern = quant == 1 ? kv_append_kernel<1> : quant == 2 ? kv_append_kernel<2> : kv_append_kernel<0>;
  kern<<<(unsigned)blocks, threads, 0, stream>>>(
      (const uint4 *)k, (const uint4 *)v, slots, k_cache, v_cache, num_tokens, Hkv,
      chunks_per_row, page_size, num_pages * page_size, k_scale, v_scale, status);
  return cudaGetLastError();
}

}  // namespace cpa
