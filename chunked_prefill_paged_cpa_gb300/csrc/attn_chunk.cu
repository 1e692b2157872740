// Prefill-chunk attention on the 5th-generation tensor cores (tcgen05, TMEM).
//
// A chunk of q_len new tokens attends to everything its sequence already has
// in the paged cache plus a causal mask inside the chunk ("vllm-learning-book
// 05. Chunked Prefill", section 3; "Chunked Prefill 技术深度解析", section 4.1;
// "How Chunked Prefill Stops Decode Starvation", "The fix").  That is a dense
// contraction: one CTA computes two 128-row query tiles against every key
// they can see.
//
// Tile rows (BM = 128) pack the G query heads that share kv head g (GQA):
// row r = (token m*TM + r/G of the chunk, head g*G + r%G), TM = 128/G tokens.
// Each K/V byte read from the paged cache therefore serves all G heads, and
// the two tiles of a CTA (m = 2mp, 2mp+1) share every K/V tile.
//
// Per CTA (352 threads, one CTA per SM):
//   warps 0-3  softmax for tile 0, warps 4-7 softmax for tile 1; one thread
//              per row.  Two short rolled passes over S in TMEM: the tile's
//              row max (causal mask on diagonal tiles only), then exp2 against
//              the running max (log2 domain), row sum, and P in bf16 written
//              back into TMEM over S chunk by chunk.  The running max (and with
//              it the TMEM O accumulator) moves only when it grew by more than
//              2^8.
//   warp 8     TMA producer: both Q tiles (3-d tensor map over q, 128-byte
//              swizzle), then per KV tile of BN = 128 keys the 8 pages of K
//              and of V of kv head g (2-d tensor map over the cache rows);
//              pages past the sequence are read from an out-of-range row and
//              arrive as zeros.  K ring of 3 stages, V ring of 2; K runs
//              one tile ahead of V.  With the append fused into the call, the
//              chunk's own pages come from the step's k/v rows instead (tensor
//              maps over those), chosen once per tile.
//   warps 9-10 warp 9 allocates the 512 TMEM columns (S0, S1, O0, O1); lane 0
//              of warp 9 + i issues tile i's tcgen05.mma: S_i = Q_i K_j^T
//              (both operands from shared memory) and O_i += P_i V_j (P from
//              TMEM, V MN-major in shared memory).  The two tiles ping-pong:
//              while one warpgroup runs its softmax, the tensor core runs the
//              other tile's PV and next QK^T.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "cpa_internal.cuh"
#include "ptx.cuh"

namespace cpa {
namespace {

constexpr int kPage = 16;
constexpr int BM = 128;          // rows per query tile
constexpr int BN = 128;          // keys per KV tile (8 pages)
constexpr int kThreads = 352;
constexpr int kProducerWarp = 8, kMmaWarp = 9;  // MMA issuers: warps 9 and 10
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct ChunkCfg {
  static constexpr int PANELS = D / 64;          // 128-byte swizzle panels along head_dim
  static constexpr int Q_BYTES = BM * D * 2;     // one query tile
  static constexpr int KV_BYTES = BN * D * 2;    // one K (or V) tile
  static constexpr int PAGE_BYTES = 16 * D * 2;  // one page of one kv head
  static constexpr int KST = 3, VST = 2;       // K and V ring depths
  static constexpr int OFF_Q = 0;                // two query tiles
  static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + KST * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + VST * KV_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;  // barriers, scan scratch, 1 KB alignment
};

struct Bars {
  uint64_t q_full, q_empty, k_full[3], k_empty[3], v_full[2], v_empty[2], s_full[2], p_full[2],
      o_final[2];
  uint32_t tmem_base;
  uint32_t mma_lock;  // held by the issuer queueing a batch of MMAs
};

__device__ __forceinline__ int seq_work(const AttnParams &p, int s, int G) {
  const int q_len = __ldg(p.query_start_loc + s + 1) - __ldg(p.query_start_loc + s);
  if (q_len < 2) return 0;
  const int mt = (q_len * G + BM - 1) / BM;
  return p.Hkv * ((mt + 1) / 2);
}

// One work item = two consecutive 128-row query tiles (m = 2mp, 2mp+1) of one
// (chunk sequence, kv head).  Every warp locates its items on its own with a
// warp-level prefix sum over the sequences, so the warp roles never have to
// synchronise with each other between items.
struct Item {
  int s, qs, q_len, ctx, g, mp, mt, n_kv0, n_kv1, n_kv, n_pages;
};

__device__ int warp_total_items(const AttnParams &p, int G) {
  const int lane = threadIdx.x & 31;
  int local = 0;
  for (int s = lane; s < p.num_seqs; s += 32) local += seq_work(p, s, G);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
  return local;
}

template <int G>
__device__ bool warp_find_item(const AttnParams &p, int item, Item &it) {
  constexpr int TM = BM / G;
  const int lane = threadIdx.x & 31;
  const int S = p.num_seqs;
  const int per = (S + 31) / 32;
  const int s0 = lane * per, s1 = min(S, s0 + per);
  int local = 0;
  for (int s = s0; s < s1; ++s) local += seq_work(p, s, G);
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const int excl = incl - local;
  int fs = -1, fli = 0;
  if (item >= excl && item < incl) {
    int acc = excl;
    for (int s = s0; s < s1; ++s) {
      const int c = seq_work(p, s, G);
      if (item < acc + c) { fs = s; fli = item - acc; break; }
      acc += c;
    }
  }
  const unsigned who = __ballot_sync(0xffffffffu, fs >= 0);
  if (!who) return false;
  const int src = __ffs(who) - 1;
  it.s = __shfl_sync(0xffffffffu, fs, src);
  const int li = __shfl_sync(0xffffffffu, fli, src);
  it.qs = __ldg(p.query_start_loc + it.s);
  it.q_len = __ldg(p.query_start_loc + it.s + 1) - it.qs;
  it.mt = (it.q_len * G + BM - 1) / BM;
  const int npair = (it.mt + 1) / 2;
  it.g = li % p.Hkv;
  it.mp = npair - 1 - li / p.Hkv;  // later tiles (more keys) first
  int ctx = __ldg(p.seq_lens + it.s);
  const int cap = p.max_pages * kPage;
  if (ctx > cap) ctx = cap;
  if (ctx < it.q_len) ctx = it.q_len;  // malformed metadata; never read past the row
  it.ctx = ctx;
  const int m0 = 2 * it.mp, m1 = m0 + 1;
  it.n_kv0 = (ctx - it.q_len + min(m0 * TM + TM - 1, it.q_len - 1)) / BN + 1;
  it.n_kv1 = m1 < it.mt ? (ctx - it.q_len + min(m1 * TM + TM - 1, it.q_len - 1)) / BN + 1 : 0;
  it.n_kv = max(it.n_kv0, it.n_kv1);
  it.n_pages = (ctx + kPage - 1) / kPage;
  return true;
}

// The work items of one CTA, wave by wave: item w*grid + b in even waves and
// (w+1)*grid - 1 - b in odd ones.  Items come longest first (later query tiles
// see more keys), so a CTA whose first item is long gets a short second one;
// plain round-robin gave the CTA with the longest item the longest of the
// second wave too.  Every warp of the CTA walks the same sequence.
struct ItemSeq {
  int b, grid, total, w;
  __device__ int next() {
    for (;;) {
      const int wv = w++;
      if ((int64_t)wv * grid >= total) return total;
      const int it = (wv & 1) ? (wv + 1) * grid - 1 - b : wv * grid + b;
      if (it < total) return it;
    }
  }
};

// Keys at positions >= n of a 32-column chunk become -inf.
__device__ __forceinline__ void mask_chunk(uint32_t (&sr)[32], int n) {
#pragma unroll
  for (int e = 0; e < 32; ++e)
    if (e >= n) sr[e] = __float_as_uint(-INFINITY);
}

// p = exp2(s * scale - m) for 32 columns as 16 bf16 pairs in `pw`; the fp32
// row sum (packed pairs) goes to four independent accumulators, so it is not
// one long dependency chain.
__device__ __forceinline__ void exp_chunk_regs(const uint32_t (&sr)[32], uint64_t sc2, uint64_t nm2,
                                               uint64_t (&rs2)[4], uint32_t (&pw)[16]) {
#pragma unroll
  for (int h = 0; h < 16; ++h) {
    const uint64_t x2 = ptx::ffma2(ptx::pack2(__uint_as_float(sr[2 * h]), __uint_as_float(sr[2 * h + 1])),
                                   sc2, nm2);
    float x0, x1;
    ptx::unpack2(x2, x0, x1);
    const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
    rs2[h & 3] = ptx::fadd2(rs2[h & 3], ptx::pack2(p0, p1));
    pw[h] = ptx::pack_bf16x2(p0, p1);
  }
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
attn_chunk_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_kin,
                  const __grid_constant__ CUtensorMap tm_vin, int kv_rows) {
  using C = ChunkCfg<D>;
  constexpr int TM = BM / G;  // tokens per tile
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char *sQ = smem + C::OFF_Q;
  unsigned char *sK = smem + C::OFF_K;
  unsigned char *sV = smem + C::OFF_V;
  Bars *bs = reinterpret_cast<Bars *>(smem + C::OFF_BAR);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int total = warp_total_items(p, G);  // identical in every warp
  if ((int)blockIdx.x >= total) return;      // uniform over the CTA

  if (tid == 0) {
    ptx::mbar_init(&bs->q_full, 1);
    ptx::mbar_init(&bs->q_empty, 2);
    for (int i = 0; i < 3; ++i) {
      ptx::mbar_init(&bs->k_full[i], 1);
      ptx::mbar_init(&bs->k_empty[i], 2);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bs->v_full[i], 1);
      ptx::mbar_init(&bs->v_empty[i], 2);
      ptx::mbar_init(&bs->s_full[i], 1);
      ptx::mbar_init(&bs->p_full[i], 128);
      ptx::mbar_init(&bs->o_final[i], 1);
    }
    ptx::fence_mbar_init();
    bs->mma_lock = 0u;
  }
  if (warp == kMmaWarp) ptx::tmem_alloc(&bs->tmem_base, 512);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bs->tmem_base;  // S_i at columns 128*i, O_i at 256 + 128*i

  if (warp == kProducerWarp) {
    // ------------------------------- TMA producer -------------------------------
    if (lane == 0) {
      ptx::prefetch_tmap(&tm_q);
      ptx::prefetch_tmap(&tm_k);
      ptx::prefetch_tmap(&tm_v);
      if (p.fused) {
        ptx::prefetch_tmap(&tm_kin);
        ptx::prefetch_tmap(&tm_vin);
      }
    }
    uint32_t kvc = 0;  // K/V tiles loaded so far by this CTA
    bool ok = true;
    int n = 0;
    ItemSeq seq{(int)blockIdx.x, (int)gridDim.x, total, 0};
    for (int item = seq.next(); ok && item < total; item = seq.next(), ++n) {
      Item it;
      if (!warp_find_item<G>(p, item, it)) break;
      // the Q buffers are free once every MMA of the previous item completed
      if (n > 0 && !ptx::mbar_wait(&bs->q_empty, (n - 1) & 1)) { ok = false; break; }
      if (lane == 0) {
        const int ntiles = it.n_kv1 > 0 ? 2 : 1;
        ptx::mbar_arrive_expect_tx(&bs->q_full, ntiles * C::Q_BYTES);
        for (int i = 0; i < ntiles; ++i)
#pragma unroll
          for (int pl = 0; pl < C::PANELS; ++pl)
            ptx::tma_load_3d(sQ + i * C::Q_BYTES + pl * BM * 128, &tm_q, pl * 64, it.g * G,
                             it.qs + (2 * it.mp + i) * TM, &bs->q_full);
      }
      // With the append fused in, the chunk's own keys and values are read
      // from the step's k/v rows: a page made only of new tokens is loaded
      // from there (encoded below as -2 - its first token).  A page holding
      // both cached and new rows (a chunk that starts inside a page) is read
      // from the cache, after this warp has written its new rows there and
      // fenced them against the bulk-copy proxy; other CTAs may write the same
      // bytes, with the same values.
      const int prefix = it.ctx - it.q_len;
      const int first_new_page = (prefix + kPage - 1) / kPage;  // first page of new tokens only
      if (p.fused && (prefix % kPage) != 0) {
        constexpr int CPR = D * 2 / 16;  // 16-byte pieces per row
        const int nnew = min(it.q_len, first_new_page * kPage - prefix);
        const int total = nnew * 2 * CPR;
        const uint4 *kin = static_cast<const uint4 *>(p.k_new);
        const uint4 *vin = static_cast<const uint4 *>(p.v_new);
        uint4 *kc4 = static_cast<uint4 *>(const_cast<void *>(p.k_cache));
        uint4 *vc4 = static_cast<uint4 *>(const_cast<void *>(p.v_cache));
        const int64_t num_slots = p.num_pages * kPage;
#pragma unroll
        for (int u = 0; u < (15 * 2 * CPR + 31) / 32; ++u) {
          const int c = lane + 32 * u;
          if (c < total) {
            const int r = c / (2 * CPR), part = c - r * 2 * CPR;
            const bool isv = part >= CPR;
            const int ch = isv ? part - CPR : part;
            const int64_t t = it.qs + r;
            const int64_t slot = __ldg(p.slot_mapping + t);
            const uint4 w = __ldg((isv ? vin : kin) + (t * p.Hkv + it.g) * CPR + ch);
            if (slot >= num_slots) {
              atomicOr(p.status, STATUS_BAD_SLOT);
            } else if (slot >= 0) {
              const int64_t pg = slot / kPage, off = slot - pg * kPage;
              (isv ? vc4 : kc4)[((pg * p.Hkv + it.g) * kPage + off) * CPR + ch] = w;
            }
          }
        }
        ptx::fence_proxy_async_global();
        __syncwarp();
      }
      // page ids of the item, 32 at a time in this warp's registers (lane l
      // holds page 32 b + l of block b), the next block prefetched
      const int32_t *bt = p.block_table + (int64_t)it.s * p.max_pages;
      auto load_block = [&](int b) -> int {
        const int pi = 32 * b + lane;
        if (pi >= it.n_pages) return kv_rows;  // past the sequence: zero fill
        if (p.fused && pi >= first_new_page) return -2 - (it.qs + pi * kPage - prefix);
        const int page = __ldg(bt + pi);
        if (page < 0 || page >= p.num_pages) {
          atomicOr(p.status, STATUS_BAD_PAGE);
          return kv_rows;
        }
        return (page * p.Hkv + it.g) * kPage;
      };
      // V lags K by one tile, so the block before the current one is kept too
      int blk_prev = kv_rows, blk_cur = load_block(0), blk_next = load_block(1), blk = 0;
      auto load_tile = [&](unsigned char *dst, bool is_v, uint64_t *bar, int j) {
        const int b = j >> 2;
        while (blk < b) {  // warp-uniform
          blk_prev = blk_cur;
          blk_cur = blk_next;
          ++blk;
          blk_next = load_block(blk + 1);
        }
        const int src = (b == blk) ? blk_cur : blk_prev;  // b is blk or blk - 1
        int rows[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rows[i] = __shfl_sync(0xffffffffu, src, (j & 3) * 8 + i);
        // The source is chosen once per tile: every page from the cache,
        // every page from the step's rows, or (once per item at most) the
        // tile where they meet, page by page.  A per-page choice in every
        // tile made the whole kernel ~30 % slower.
        const int p0 = 8 * j;
        const bool some_new = p.fused && max(p0, first_new_page) < min(p0 + 8, it.n_pages);
        const bool all_new = some_new && p0 >= first_new_page && p0 + 8 <= it.n_pages;
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(bar, C::KV_BYTES);
          if (is_v) {
            // V page-major: one box per page holds all its panels
            if (!some_new) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                ptx::tma_load_3d(dst + i * C::PAGE_BYTES, &tm_v, 0, rows[i], 0, bar);
            } else if (all_new) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                ptx::tma_load_4d(dst + i * C::PAGE_BYTES, &tm_vin, 0, -2 - rows[i], 0, it.g, bar);
            } else {
              for (int i = 0; i < 8; ++i) {
                if (rows[i] <= -2)
                  ptx::tma_load_4d(dst + i * C::PAGE_BYTES, &tm_vin, 0, -2 - rows[i], 0, it.g, bar);
                else
                  ptx::tma_load_3d(dst + i * C::PAGE_BYTES, &tm_v, 0, rows[i], 0, bar);
              }
            }
          } else {
            if (!some_new) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int pl = 0; pl < C::PANELS; ++pl)
                  ptx::tma_load_2d(dst + pl * BN * 128 + i * kPage * 128, &tm_k, pl * 64, rows[i], bar);
            } else if (all_new) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int pl = 0; pl < C::PANELS; ++pl)
                  ptx::tma_load_3d(dst + pl * BN * 128 + i * kPage * 128, &tm_kin, pl * 64, it.g,
                                   -2 - rows[i], bar);
            } else {
              for (int i = 0; i < 8; ++i)
                for (int pl = 0; pl < C::PANELS; ++pl) {
                  unsigned char *d = dst + pl * BN * 128 + i * kPage * 128;
                  if (rows[i] <= -2)
                    ptx::tma_load_3d(d, &tm_kin, pl * 64, it.g, -2 - rows[i], bar);
                  else
                    ptx::tma_load_2d(d, &tm_k, pl * 64, rows[i], bar);
                }
            }
          }
        }
      };
      // K runs one tile ahead of V: K_t, then V_{t-1}
      for (int t = 0; t <= it.n_kv; ++t) {
        if (t < it.n_kv) {
          const uint32_t kc = kvc + t, st = kc % C::KST;
          if (kc >= C::KST && !ptx::mbar_wait(&bs->k_empty[st], ((kc / C::KST) - 1) & 1)) {
            ok = false;
            break;
          }
          load_tile(sK + st * C::KV_BYTES, false, &bs->k_full[st], t);
        }
        if (t >= 1) {
          const uint32_t vc = kvc + t - 1, st = vc % C::VST;
          if (vc >= C::VST && !ptx::mbar_wait(&bs->v_empty[st], ((vc / C::VST) - 1) & 1)) {
            ok = false;
            break;
          }
          load_tile(sV + st * C::KV_BYTES, true, &bs->v_full[st], t - 1);
        }
      }
      kvc += it.n_kv;
    }
    if (!ok && lane == 0) atomicOr(p.status, STATUS_TIMEOUT);
  } else if (warp >= kMmaWarp) {
    // ------------------------------ MMA issuers --------------------------------
    // One issuing thread per query tile slot (warp 9: tile 0, warp 10: tile 1).
    // Issuing a tcgen05.mma stalls while the tensor pipe's queue is full, so a
    // single issuer for both tiles would notice one tile's P only after it got
    // the other tile's MMAs queued.  A commit tracks the issuing thread's own
    // operations, which is what each tile's s_full / o_final need.  The K/V
    // stage and Q release barriers take one arrival per tile: a tile that reads
    // a stage the other tile does not read (the later tile sees more keys; the
    // second tile may be absent) commits twice, so both arrivals come after
    // its reads.  Both issuers wait on q_full for every item, so neither ever
    // skips a phase of it.
    const int ti = warp - kMmaWarp;
    // A tile's batch (PV_j and the next QK^T) enters the tensor pipe as a
    // whole: interleaved one MMA at a time, both tiles' S would complete
    // together and their softmaxes would run together instead of each one
    // overlapping the other tile's MMAs.
    auto lock = [&]() -> bool {
      for (uint32_t i = 0; i < (1u << 22); ++i) {
        if (atomicCAS(&bs->mma_lock, 0u, 1u) == 0u) return true;
        __nanosleep(32);
      }
      return false;
    };
    auto unlock = [&]() { atomicExch(&bs->mma_lock, 0u); };
    constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(BM, BN, false, false);
    constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(BM, D, false, true);
    const uint32_t tS = tmem + ti * 128, tO = tmem + 256 + ti * 128;
    // Every shared-memory descriptor this issuer uses, built once: the issuing
    // warp shares its scheduler with two softmax warps, so each instruction
    // between MMAs costs several cycles and delays the tensor pipe's queue.
    constexpr int KS = D / 16, VS = BN / 16;
    uint64_t qdesc[KS], kdesc[C::KST][KS], vdesc[C::VST][VS];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int o = (ks >> 2) * BM * 128 + (ks & 3) * 32;  // panel, 16-element step
      qdesc[ks] = ptx::smem_desc_sw128(sQ + ti * C::Q_BYTES + o, 16, 1024);
#pragma unroll
      for (int st = 0; st < C::KST; ++st)
        kdesc[st][ks] = ptx::smem_desc_sw128(sK + st * C::KV_BYTES + o, 16, 1024);
    }
#pragma unroll
    for (int st = 0; st < C::VST; ++st)
#pragma unroll
      for (int ks = 0; ks < VS; ++ks)
        vdesc[st][ks] = ptx::smem_desc_sw128(sV + st * C::KV_BYTES + ks * C::PAGE_BYTES,
                                             kPage * 128, 1024);
    uint32_t kvm = 0;   // K/V tiles loaded so far for this CTA (both tiles agree)
    uint32_t pcnt = 0;  // P tiles of this slot consumed
    bool ok = true;
    int n = 0;
    ItemSeq seq{(int)blockIdx.x, (int)gridDim.x, total, 0};
    for (int item = seq.next(); ok && item < total; item = seq.next(), ++n) {
      Item it;
      if (!warp_find_item<G>(p, item, it)) break;
      if (lane == 0) {
        const int n_mine = ti ? it.n_kv1 : it.n_kv0;
        const int n_other = ti ? it.n_kv0 : it.n_kv1;
        // QK^T MMAs only; the caller commits
        auto issue_qk = [&](uint32_t kvidx) {
          const uint32_t st = kvidx % C::KST;
#pragma unroll
          for (int s3 = 0; s3 < C::KST; ++s3) {
            if (st == (uint32_t)s3) {
#pragma unroll
              for (int ks = 0; ks < KS; ++ks)
                ptx::mma_bf16_ss(tS, qdesc[ks], kdesc[s3][ks], idesc_qk, ks > 0 ? 1u : 0u);
            }
          }
        };
        auto release_k = [&](uint32_t kvidx) {
          ptx::mma_commit(&bs->k_empty[kvidx % C::KST]);
          if ((int)(kvidx - kvm) >= n_other) ptx::mma_commit(&bs->k_empty[kvidx % C::KST]);
        };
        ok = ptx::mbar_wait(&bs->q_full, n & 1);
        if (ok && n_mine > 0) {
          ok = ptx::mbar_wait(&bs->k_full[kvm % C::KST], (kvm / C::KST) & 1) && lock();
          if (ok) {
            ptx::tc_fence_after();
            issue_qk(kvm);
            unlock();
            ptx::mma_commit(&bs->s_full[ti]);
            release_k(kvm);
          }
        }
        for (int j = 0; ok && j < n_mine; ++j) {
          const uint32_t kv = kvm + j;
          const int vst = kv % C::VST;
          const bool more = j + 1 < n_mine;
          // everything the batch reads is resident before it starts, so its
          // MMAs go to the tensor pipe back to back; the commits follow them
          if (!ptx::mbar_wait(&bs->p_full[ti], pcnt & 1) ||
              !ptx::mbar_wait(&bs->v_full[vst], (kv / C::VST) & 1) ||
              (more && !ptx::mbar_wait(&bs->k_full[(kv + 1) % C::KST], ((kv + 1) / C::KST) & 1)) ||
              !lock()) {
            ok = false;
            break;
          }
          ++pcnt;
          ptx::tc_fence_after();
#pragma unroll
          for (int s2 = 0; s2 < C::VST; ++s2) {
            if (vst == s2) {
#pragma unroll
              for (int ks = 0; ks < VS; ++ks)
                ptx::mma_bf16_ts(tO, tS + ks * 8, vdesc[s2][ks], idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
            }
          }
          if (more) issue_qk(kv + 1);
          // the batch is queued: the other tile may queue its own behind it
          // while this thread's commits wait for these MMAs
          unlock();
          if (more) {
            ptx::mma_commit(&bs->s_full[ti]);
            release_k(kv + 1);
          } else {
            ptx::mma_commit(&bs->o_final[ti]);
          }
          ptx::mma_commit(&bs->v_empty[vst]);
          if (j >= n_other) ptx::mma_commit(&bs->v_empty[vst]);
        }
        if (ok && n_mine > 0) {
          ptx::mma_commit(&bs->q_empty);
          if (n_other == 0) ptx::mma_commit(&bs->q_empty);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      kvm += it.n_kv;
    }
    if (!ok && lane == 0) atomicOr(p.status, STATUS_TIMEOUT);
  } else {
    // ------------------------------- softmax ------------------------------------
    const int ti = warp >> 2;                 // query tile slot of this warpgroup
    const int quarter = warp & 3;             // TMEM lane quarter this warp may access
    const int r = quarter * 32 + lane;        // tile row
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tmem + ti * 128 + lane_off;
    const uint32_t tO = tmem + 256 + ti * 128 + lane_off;
    const float sl2 = p.scale_log2;
    uint32_t scnt = 0, ocnt = 0, kvb = 0;
    bool ok = true;
    ItemSeq seq{(int)blockIdx.x, (int)gridDim.x, total, 0};
    for (int item = seq.next(); ok && item < total; item = seq.next()) {
      Item it;
      if (!warp_find_item<G>(p, item, it)) break;
      const int n_mine = ti ? it.n_kv1 : it.n_kv0;
      const int ctx = it.ctx, q_len = it.q_len;
      const int tok = (2 * it.mp + ti) * TM + r / G;  // index within the chunk
      const bool row_valid = tok < q_len;
      const int last = row_valid ? ctx - q_len + tok : 0;
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < n_mine; ++j, ++scnt) {
        // waits are combined over the warp so a timeout never splits it
        // before a warp-collective TMEM access
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bs->s_full[ti], scnt & 1))) { ok = false; break; }
        ptx::tc_fence_after();
        const int key0 = j * BN;
        const bool diag = key0 + BN - 1 > last;  // tile holds keys past `last`
        const int nvis = last - key0 + 1;        // visible keys of this row in the tile
        // Pass 1: the tile's row max (rolled; TMEM loads are cheap).
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t sa[32];
          ptx::tmem_ld32(tS + c * 32, sa);
          ptx::tmem_wait_ld_regs(sa);
          if (diag) mask_chunk(sa, nvis - c * 32);
#pragma unroll
          for (int h = 0; h < 16; ++h)
            mx[h & 3] = ptx::max3(mx[h & 3], __uint_as_float(sa[2 * h]), __uint_as_float(sa[2 * h + 1]));
        }
        const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;  // log2 domain
        // The reference moves only when the max grew by more than 2^8 (or on
        // the first tile), so every p stays below 2^8; moving it rescales O
        // and l first (S_j complete implies PV_{j-1} complete: same issuing
        // thread, in order).  TMEM loads/stores are warp-collective, so the
        // warp rescales if any of its rows needs it (the others scale by 1).
        const bool move = tmax > m_run + kRescaleThreshold;  // m_run = -inf: any visible key
        const float alpha = (move && m_run != -INFINITY) ? ptx::ex2(m_run - tmax) : 1.f;
        if (move) m_run = tmax;
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
        }
        l_run *= alpha;
        // Pass 2 (rolled over pairs of 32-column chunks, the second chunk's
        // load in flight while the first is converted): P = exp2(S * scale -
        // m_run) in bf16, each chunk's 16 columns stored straight over S
        // columns already read.
        const float mref = (m_run == -INFINITY) ? 0.f : m_run;
        const uint64_t sc2 = ptx::pack2(sl2, sl2);
        const uint64_t nm2 = ptx::pack2(-mref, -mref);
        uint64_t rs2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll 1
        for (int c = 0; c < 4; c += 2) {
          uint32_t sa[32], sb[32], w16[16];
          ptx::tmem_ld32(tS + c * 32, sa);
          ptx::tmem_ld32(tS + (c + 1) * 32, sb);
          ptx::tmem_wait_ld_regs(sa);
          if (diag) mask_chunk(sa, nvis - c * 32);
          exp_chunk_regs(sa, sc2, nm2, rs2, w16);
          ptx::tmem_st16(tS + c * 16, w16);
          ptx::tmem_wait_ld_regs(sb);
          if (diag) mask_chunk(sb, nvis - (c + 1) * 32);
          exp_chunk_regs(sb, sc2, nm2, rs2, w16);
          ptx::tmem_st16(tS + (c + 1) * 16, w16);
        }
        {
          const uint64_t r2 = ptx::fadd2(ptx::fadd2(rs2[0], rs2[1]), ptx::fadd2(rs2[2], rs2[3]));
          float rs0, rs1;
          ptx::unpack2(r2, rs0, rs1);
          l_run += rs0 + rs1;
        }
        // Cache slots at or past ctx in the last page may hold anything (NaN
        // included) and 0 * NaN is NaN inside PV: zero those V rows before PV
        // runs.  Both warpgroups may write the same zeros; rows past the last
        // page were loaded out of range and are zero already.
        if (key0 + BN > ctx) {
          const uint32_t kv = kvb + j;
          if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bs->v_full[kv % C::VST], (kv / C::VST) & 1))) {
            ok = false;
            break;
          }
          if (r >= ctx - key0 && r < it.n_pages * kPage - key0) {
            unsigned char *vrow = sV + (kv % C::VST) * C::KV_BYTES + (r / kPage) * C::PAGE_BYTES +
                                  (r % kPage) * 128;
#pragma unroll
            for (int pl = 0; pl < C::PANELS; ++pl)
#pragma unroll
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4 *>(vrow + pl * kPage * 128 + c * 16) = make_uint4(0, 0, 0, 0);
          }
          ptx::fence_proxy_async_smem();
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&bs->p_full[ti]);
      }
      kvb += it.n_kv;
      if (!ok || n_mine == 0) continue;
      // epilogue: O / l
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bs->o_final[ti], ocnt & 1))) { ok = false; break; }
      ++ocnt;
      ptx::tc_fence_after();
      const float inv = 1.f / l_run;
      __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out) +
                           ((int64_t)(it.qs + tok) * p.Hq + it.g * G + r % G) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        ptx::tmem_ld32(tO + c * 32, o);
        ptx::tmem_wait_ld_regs(o);
        if (row_valid) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t wds[4];
#pragma unroll
            for (int h = 0; h < 4; ++h)
              wds[h] = ptx::pack_bf16x2(__uint_as_float(o[q4 * 8 + h * 2]) * inv,
                                        __uint_as_float(o[q4 * 8 + h * 2 + 1]) * inv);
            *reinterpret_cast<uint4 *>(out + c * 32 + q4 * 8) =
                make_uint4(wds[0], wds[1], wds[2], wds[3]);
          }
        }
      }
      // O is read; the next item's first PV may overwrite it after p_full
      ptx::tc_fence_before();
    }
    if (!ok && lane == 0) atomicOr(p.status, STATUS_TIMEOUT);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

template <int D, int G>
cudaError_t launch_dg(const AttnParams &p, int grid, cudaStream_t stream) {
  using C = ChunkCfg<D>;
  auto encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap tq, tk, tv;
  // q viewed as [T][Hq][D]: box = 64 dims x G heads x BM/G tokens
  {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.Hq, (cuuint64_t)p.num_tokens};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)p.Hq * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(BM / G)};
    cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(p.q), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int64_t rows = p.num_pages * p.Hkv * kPage;
  {
    // K: cache rows [rows][D], box = one 64-dim panel of one page (16 rows)
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kPage};
    cuuint32_t estr[2] = {1, 1};
    if (encode(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(p.k_cache), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // V: the same rows viewed as (64 dims, row, panel), box = a whole page with
    // its panels outermost, i.e. [panel][16 rows][64 dims] in shared memory --
    // each page is exactly the B operand of one 16-key step of PV.
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)C::PANELS};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)kPage, (cuuint32_t)C::PANELS};
    cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(p.v_cache), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_chunk_kernel<D, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  CUtensorMap tkin = tk, tvin = tv;  // unused unless the append is fused
  if (p.fused) {
    // the step's new k rows [T][Hkv][D]: box = one 64-dim panel of one kv head
    // for 16 consecutive tokens, the same [16][64] swizzled layout as a cache page
    {
      cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.Hkv, (cuuint64_t)p.num_tokens};
      cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)p.Hkv * D * 2};
      cuuint32_t box[3] = {64, 1, (cuuint32_t)kPage};
      cuuint32_t estr[3] = {1, 1, 1};
      if (encode(&tkin, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(p.k_new), dims,
                 strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
    // the step's new v rows viewed as (64 dims, token, panel, kv head): box =
    // 16 tokens of one kv head with its panels outermost, as a cache V page
    {
      cuuint64_t dims[4] = {64, (cuuint64_t)p.num_tokens, (cuuint64_t)C::PANELS,
                            (cuuint64_t)p.Hkv};
      cuuint64_t strides[3] = {(cuuint64_t)p.Hkv * D * 2, 128, (cuuint64_t)D * 2};
      cuuint32_t box[4] = {64, (cuuint32_t)kPage, (cuuint32_t)C::PANELS, 1};
      cuuint32_t estr[4] = {1, 1, 1, 1};
      if (encode(&tvin, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(p.v_new), dims,
                 strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
  }
  attn_chunk_kernel<D, G><<<grid, kThreads, C::SMEM, stream>>>(p, tq, tk, tv, tkin, tvin,
                                                                (int)rows);
  return cudaGetLastError();
}

}  // namespace

bool chunk_tc_path(int dtype, int D, int G) {
  if (dtype != CPA_BF16) return false;
  if (D != 64 && D != 128) return false;
  return G == 1 || G == 2 || G == 4 || G == 8;
}

int chunk_grid_estimate(const AttnParams &p, int sms) {
  // Persistent grid: one CTA per expected work item (pairs of 128-row tiles),
  // assuming the step's chunk tokens are num_tokens - num_seqs + 1 (one chunk
  // among decodes); any count is correct, this only sets the SM split.
  const int G = p.Hq / p.Hkv;
  const int64_t chunk_tokens = (int64_t)p.num_tokens - p.num_seqs + 1;
  const int64_t pairs = (chunk_tokens * G + 2 * BM - 1) / (2 * BM);
  const int64_t est = (int64_t)p.Hkv * pairs;
  return (int)(est < 1 ? 1 : (est > sms ? sms : est));
}

cudaError_t launch_attention_chunk(const AttnParams &p, int grid, cudaStream_t stream) {
  const int G = p.Hq / p.Hkv;
  if (p.D == 128) {
    switch (G) {
      case 1: return launch_dg<128, 1>(p, grid, stream);
      case 2: return launch_dg<128, 2>(p, grid, stream);
      case 4: return launch_dg<128, 4>(p, grid, stream);
      case 8: return launch_dg<128, 8>(p, grid, stream);
    }
  } else {
    switch (G) {
      case 1: return launch_dg<64, 1>(p, grid, stream);
      case 2: return launch_dg<64, 2>(p, grid, stream);
      case 4: return launch_dg<64, 4>(p, grid, stream);
      case 8: return launch_dg<64, 8>(p, grid, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace cpa
