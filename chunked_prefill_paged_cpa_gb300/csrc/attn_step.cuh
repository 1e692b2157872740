// One attention step over a packed hybrid batch, in one persistent launch on
// the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// The batch holds prefill chunks (q_len > 1: each query row sees all earlier
// K/V of its sequence in the paged cache plus a causal mask inside the chunk)
// and single-token decodes ("vllm-learning-book 05. Chunked Prefill", sections
// 3 and 4; "Chunked Prefill 技术深度解析", section 4.1).  Both kinds of work are
// cut into items and handed to the CTAs of one persistent grid from a device
// queue, so a step has no padding and no SM waits for a kernel boundary
// (same page, section 4: one packed batch instead of padded per-kind batches).
//
//   chunk unit   two 128-row query tiles of one (chunk, kv head) against a
//                range of 128-key KV tiles.  Rows pack the G query heads of the
//                kv head (row = token * G + head), so each K/V byte serves all
//                G heads.  A chunk whose tile pairs are fewer than the SMs has
//                each pair's KV range split over several units; the last unit
//                to finish merges their partial results with log-sum-exp
//                weights ("Chunked Prefill 技术深度解析", section 7.2).
//   decode slice up to P pages of one (decode, kv head) segment.  The G query
//                rows are the N = 16 side of S^T = K Q^T (M = 128 keys) and of
//                O^T = V^T P^T (M = 128 dims), so the page stream runs through
//                the tensor cores, not through per-key FMAs.  A segment cut
//                into several slices is merged the same way by its last slice.
//
// A small plan kernel runs first (programmatic dependent launch: the step
// kernel's prologue overlaps it).  It enumerates the items and queues them
// longest first (chunk units, then decode slices by size), zeroes the queue
// ticket and every merge counter of this step, and -- when the append is fused
// into the call -- copies the step's new K/V rows into the cache, so the step
// kernel reads every key and value from the cache.
//
// Step kernel, per CTA (352 threads, one CTA per SM):
//   warp 8     producer: claims items from the queue, publishes them to the
//              other warps through a ring of item slots, and issues the TMA
//              loads: the query tile(s) (chunk: two 128-row tiles; decode: the
//              G rows of one token), then the item's K/V tiles of 8 pages
//              (K panel-major, V page-major, 128-byte swizzle; K ring of 3
//              stages, V ring of 2, K one tile ahead).  Pages past the item's
//              range arrive as zeros (out-of-range rows).
//   warps 9-10 MMA issuers, one per query tile (chunk) or pipeline (decode).
//   warps 0-7  two softmax warpgroups.  Chunk: one thread per query row, the
//              scores in TMEM, P written back into TMEM.  Decode: one thread
//              per key of the 128-key block, the block's row maxima reduced
//              over the warpgroup, P^T written to shared memory.  The running
//              maximum (and with it the accumulator) moves only when it grew
//              by more than 2^8.  Decode pipelines take alternate blocks of a
//              slice and merge at its end through TMEM.
//
// Cache modes (template KVM): 0 bf16 queries and cache; 1 binary16 queries
// and cache; 2 a cache of OCP FP8 E4M3 codes.  In mode 2 each page of codes
// lands in the upper half of its page's 16-bit destination in the K/V stage,
// and the eight softmax warps widen it in place to binary16 (exact), one page
// per warp, every fill in the producer's order, before the MMAs read it; the
// MMAs then take binary16 operands (queries converted to binary16 by the plan
// kernel when they are bf16), k_scale is folded into the softmax scale and
// v_scale into the output.  The widening also zeroes the rows of cache slots
// past the sequence.
//
// This header is compiled once per cache mode (attn_step_<mode>.cu).
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "cpa_internal.cuh"
#include "ptx.cuh"

namespace cpa {
namespace {

constexpr int kPage = 16;
constexpr int BM = 128;          // rows per query tile
constexpr int BN = 128;          // keys per KV tile (8 pages)
constexpr int kThreads = 352;
constexpr int kProducerWarp = 8, kMmaWarp = 9;  // MMA issuers: warps 9 and 10
constexpr int kItemSlots = 4;
constexpr int kDecN = 16;        // N of the decode MMAs: the G query rows, padded
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kPlanThreads = 1024;  // block size of the plan kernel (its side work)
constexpr int kPlanWorkers = 256;   // threads of block 0 that build the queue
// A tile pair's KV range is split over several units only into pieces of at
// least this many KV tiles: each unit pays a query load, a pipeline fill and
// a partial-result merge.
constexpr int kMinUnitTiles = 8;
// Decode slices are queued longest first, bucketed by their 8-page blocks.
constexpr int kSizeBuckets = kPlanWorkers;

enum : int { KIND_CHUNK = 0, KIND_DECODE = 1, KIND_DONE = 2 };

template <int D>
struct StepCfg {
  static constexpr int PANELS = D / 64;          // 128-byte swizzle panels along head_dim
  static constexpr int Q_BYTES = BM * D * 2;     // one query tile
  static constexpr int KV_BYTES = BN * D * 2;    // one K (or V) tile
  static constexpr int PAGE_BYTES = 16 * D * 2;  // one page of one kv head
  static constexpr int KST = 3, VST = 2;         // K and V ring depths
  static constexpr int OFF_Q = 0;                // two query tiles
  static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
  static constexpr int OFF_V = OFF_K + KST * KV_BYTES;
  // decode, inside the query-tile region (1 KB aligned): two Q^T buffers (16
  // rows each, alternate items), each pipeline's P^T (16 rows x 128 keys),
  // and a third V stage
  static constexpr int QT_BYTES = PANELS * kDecN * 128;
  static constexpr int OFF_QT = OFF_Q;           // + QT_BYTES * buffer
  static constexpr int OFF_PT = OFF_Q + 2 * QT_BYTES;  // + 4096 * pipeline
  static constexpr int OFF_VX = OFF_Q + 16384;
  // The decode PV uses M = 128 rows of V^T; at head_dim 64 its upper half reads
  // the next 2 KB (never used): keep that inside the allocation.
  static constexpr int PAD = D == 64 ? 2048 : 0;
  // E4M3 cache: where a page of codes (16 rows x D bytes) lands inside the
  // 16-bit stage, within page i's own destination: K at K8_OFF + i * 2 KB
  // (the last panel's slot of the page at D = 128, the slot's second half at
  // D = 64), V at V8_OFF + i * PAGE_BYTES (the page's second half)
  static constexpr int PAGE8 = 16 * D;
  static constexpr int K8_OFF = D == 128 ? BN * 128 : 1024;
  static constexpr int V8_OFF = PAGE_BYTES / 2;
  static constexpr int OFF_BAR = OFF_V + VST * KV_BYTES + PAD;
  static constexpr int BAR_BYTES = 2048;
  static constexpr int SMEM = OFF_BAR + BAR_BYTES + 1024;  // barriers and scratch, 1 KB alignment
  static_assert(OFF_PT + 2 * 4096 <= OFF_VX && OFF_VX + KV_BYTES <= OFF_K,
                "decode buffers overflow the query region");
  static_assert(SMEM <= 232448, "more shared memory than a CTA can have");
};

// One work item as the producer publishes it to the other warps.
struct WorkItem {
  int kind, s, g, qs, q_len, ctx, n_pages;
  int page0, page_end;  // pages of the item: tile t holds pages page0 + 8 (j0 + t) + i
  int j0, n_tiles;      // first KV tile (chunk: absolute) and tiles loaded
  int n_mine[2];        // tiles of query tile / pipeline 0 and 1
  int mp;               // chunk: tile pair
  int n_kv[2], n_kv_max;  // chunk: KV tiles each query tile sees
  int nsplit, slot, first_slot;  // units (pieces) of the pair (segment), this item's slot
};

struct Bars {
  uint64_t q_full[2], q_empty[2], k_full[3], k_empty[3], v_full[3], v_empty[3], s_full[2],
      p_full[2], o_final[2];
  uint64_t k_conv[3], v_conv[3];  // E4M3 cache: a fill widened (256 arrivals)
  uint64_t item_full[kItemSlots], item_empty[kItemSlots];
  uint64_t wg_bar[2];            // softmax warpgroup syncs (128 arrivals)
  uint64_t hand_off, release;    // decode pipelines' merge (128 arrivals each)
  uint64_t mma_done[2];          // each issuer's MMAs drained before TMEM is freed
  uint32_t tmem_base;
  uint32_t mma_lock;             // held by the issuer queueing a batch of MMAs
  int bcast[2];
  float red[2][3][4][8];         // [warpgroup][buffer][warp][row]: block maxima, row sums
  float2 mlx[8];                 // decode pipeline 1's (max, sum) per row
  WorkItem items[kItemSlots];
};
static_assert(sizeof(Bars) <= 2048, "barrier area overflow");

// ---------------------------------------------------------------------------
// Item geometry shared by the plan kernel and the step kernel.

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Context of sequence s clamped to the block table (and to at least q_len).
__device__ __forceinline__ int seq_ctx(const AttnParams &p, int s, int q_len) {
  int ctx = __ldg(p.seq_lens + s);
  const int cap = p.max_pages * kPage;
  if (ctx > cap) ctx = cap;
  if (ctx < q_len) ctx = q_len;  // malformed metadata; never read past the row
  return ctx;
}

// KV tiles seen by query tile m of a chunk (rows m*TM .. m*TM+TM-1).
template <int G>
__device__ __forceinline__ int tile_kv(int ctx, int q_len, int m) {
  constexpr int TM = BM / G;
  return (ctx - q_len + min(m * TM + TM - 1, q_len - 1)) / BN + 1;
}

// Queue entry written by the plan kernel (32 bytes, two 16-byte stores).
struct __align__(16) ItemDesc {
  int s_kind;   // sequence | KIND_DECODE << 30
  int qs, ctx;
  int q_len;    // decode: pieces of the segment
  int g_x;      // kv head | (chunk: tile pair, decode: piece) << 8
  int a, b, c;  // chunk: unit | units << 16, unit index, first unit of the pair
                // decode: first page, end page, slice index
};

// ---------------------------------------------------------------------------
// Plan kernel: block 0 builds the queue; blocks >= 1 append the step's new
// K/V rows into the cache when the append is fused into the call.

// dynamic shared memory of the plan: per sequence its first token, query
// length, context, two exclusive bases and a queue place
inline size_t plan_smem_bytes(int num_seqs) { return sizeof(int) * (6 * (size_t)num_seqs + 2); }

// 16-byte pieces of the plan's side work: the fused append's rows, then (E4M3
// cache with bf16 queries) the queries to convert to binary16.
template <int KVM>
__host__ __device__ __forceinline__ int64_t plan_append_pieces(const AttnParams &p) {
  return p.fused ? (int64_t)p.num_tokens * p.Hkv * (p.D * 2 / 16) : 0;
}
template <int KVM>
__host__ __device__ __forceinline__ int64_t plan_q_pieces(const AttnParams &p) {
  return (KVM == 2 && !p.act_f16) ? (int64_t)p.num_tokens * p.Hq * (p.D * 2 / 16) : 0;
}

template <int KVM, int G>
__global__ void __launch_bounds__(kPlanThreads) attn_plan_kernel(const AttnParams p,
                                                                  const StepWs w) {
  // the step kernel may be scheduled now: it waits in grid_dependency_wait
  // for this whole grid to finish
  ptx::grid_launch_dependents();
  const int tid = threadIdx.x;
  if (blockIdx.x > 0) {
    // the append: every new row into its cache slot, 16 bytes of input per
    // thread (an E4M3 cache stores their 8 codes); then the queries' binary16
    // copy when the MMAs need one
    const int CPR = p.D * 2 / 16;  // 16-byte pieces per input row
    const int64_t na = plan_append_pieces<KVM>(p), total = na + plan_q_pieces<KVM>(p);
    const int64_t stride = (int64_t)(gridDim.x - 1) * blockDim.x;
    const int64_t num_slots = p.num_pages * kPage;
    const uint4 *kin = static_cast<const uint4 *>(p.k_new);
    const uint4 *vin = static_cast<const uint4 *>(p.v_new);
    for (int64_t i = (int64_t)(blockIdx.x - 1) * blockDim.x + tid; i < total; i += stride) {
      if (i >= na) {
        const uint4 x = __ldg(static_cast<const uint4 *>(p.q) + (i - na));
        uint32_t in[4] = {x.x, x.y, x.z, x.w}, o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] = ptx::pack_f16x2(bf16_lo(in[e]), bf16_hi(in[e]));
        static_cast<uint4 *>(p.q16)[i - na] = make_uint4(o[0], o[1], o[2], o[3]);
        continue;
      }
      const int64_t row = i / CPR, t = row / p.Hkv;
      const int g = (int)(row - t * p.Hkv), ch = (int)(i - row * CPR);
      const int64_t sl = __ldg(p.slot_mapping + t);
      if (sl >= num_slots) {
        if (ch == 0) atomicOr(p.status, STATUS_BAD_SLOT);
      } else if (sl >= 0) {
        const int64_t pg = sl / kPage, off = sl - pg * kPage;
        const int64_t dst = ((pg * p.Hkv + g) * kPage + off) * CPR + ch;
        if (KVM == 2) {
          uint2 *kc = static_cast<uint2 *>(const_cast<void *>(p.k_cache));
          uint2 *vc = static_cast<uint2 *>(const_cast<void *>(p.v_cache));
          if (p.act_f16) {
            kc[dst] = ptx::quantise8_e4m3<true>(__ldg(kin + i), p.k_scale);
            vc[dst] = ptx::quantise8_e4m3<true>(__ldg(vin + i), p.v_scale);
          } else {
            kc[dst] = ptx::quantise8_e4m3<false>(__ldg(kin + i), p.k_scale);
            vc[dst] = ptx::quantise8_e4m3<false>(__ldg(vin + i), p.v_scale);
          }
        } else {
          uint4 *kc = static_cast<uint4 *>(const_cast<void *>(p.k_cache));
          uint4 *vc = static_cast<uint4 *>(const_cast<void *>(p.v_cache));
          kc[dst] = __ldg(kin + i);
          vc[dst] = __ldg(vin + i);
        }
      }
    }
    ptx::fence_proxy_async_global();
    return;
  }

  // Block 0: the queue.  Every sequence's metadata is read once (coalesced)
  // into shared memory; totals and per-sequence counts come from block scans;
  // the decode slices are ordered longest first by a count per size bucket
  // (one atomic per sequence); the entries are then written in parallel.
  // Only the first kPlanWorkers threads: a smaller barrier settles faster
  // (the queue is on the step's critical path); they sync on barrier 1.
  if (tid >= kPlanWorkers) return;
  auto sync = [] { asm volatile("bar.sync 1, %0;" ::"n"(kPlanWorkers) : "memory"); };
  extern __shared__ int plan_smem[];
  const int S = p.num_seqs, lane = tid & 31, warp = tid >> 5;
  const int Hkv = p.Hkv;
  int *sq_qs = plan_smem, *sq_len = sq_qs + S, *sq_ctx = sq_len + S;
  int *s_dec = sq_ctx + S;     // [S + 1] exclusive bases of each sequence's slices
  int *s_chk = s_dec + S + 1;  // [S + 1] ... and of its chunk units
  int *s_pos = s_chk + S + 1;  // [S] first place of a decode sequence's slices, by size
  __shared__ long long s_red[kPlanWorkers / 32][3];
  __shared__ int s_wd[kPlanWorkers / 32], s_wc[kPlanWorkers / 32];
  __shared__ int s_hist[kSizeBuckets];
  for (int b = tid; b < kSizeBuckets; b += kPlanWorkers) s_hist[b] = 0;

  // pass 1: metadata, decode pages, chunk tile pairs and their KV tiles
  long long pages = 0, pairs = 0, ctiles = 0;
  for (int s = tid; s < S; s += kPlanWorkers) {
    const int qs = __ldg(p.query_start_loc + s);
    const int q_len = __ldg(p.query_start_loc + s + 1) - qs;
    const int ctx = q_len < 1 ? 0 : seq_ctx(p, s, q_len);
    sq_qs[s] = qs;
    sq_len[s] = q_len;
    sq_ctx[s] = ctx;
    if (q_len == 1) {
      pages += (long long)Hkv * ceil_div(ctx, kPage);
    } else if (q_len > 1) {
      const int mt = ceil_div(q_len * G, BM), npair = (mt + 1) / 2;
      pairs += (long long)Hkv * npair;
      // tiles per pair grow about linearly from the first pair to the last
      ctiles += (long long)Hkv * npair * (tile_kv<G>(ctx, q_len, 1) + tile_kv<G>(ctx, q_len, mt - 1)) / 2;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    pages += __shfl_xor_sync(0xffffffffu, pages, o);
    pairs += __shfl_xor_sync(0xffffffffu, pairs, o);
    ctiles += __shfl_xor_sync(0xffffffffu, ctiles, o);
  }
  if (lane == 0) { s_red[warp][0] = pages; s_red[warp][1] = pairs; s_red[warp][2] = ctiles; }
  sync();
  long long tp = 0, tq = 0, tt = 0;
  for (int i = 0; i < kPlanWorkers / 32; ++i) { tp += s_red[i][0]; tq += s_red[i][1]; tt += s_red[i][2]; }
  const long long grid = w.grid;
  // decode pages per slice: about one slice per CTA, so most segments stay
  // whole (every slice pays a pipeline fill and a finalisation; a segment cut
  // into pieces also pays a merge) while the longest-first order keeps the
  // tail short; at least 16 pages, a multiple of the 8-page block
  const int P = (int)max(16ll, ((tp + grid - 1) / grid + 7) / 8 * 8);
  // Chunk tile pairs are split over several units when they are fewer than
  // the CTAs, so that no unit is longer than three quarters of a CTA's share
  // of the step's work: its chunk KV tiles and decode blocks (both 128-key
  // blocks of attention) over the grid.  Without that, one long unit (a short
  // chunk with a long cached prefix) would set the step's length on its own;
  // with smaller units, each one's partial result, merge and pipeline fill
  // cost more than the balance they buy (measured: at half a share the
  // default hybrid step took 117 us, at three quarters 105 us).
  // At most kMaxStepGrid units in all (the split-unit partials hold that many).
  const int nu = (tq == 0 || tq >= grid) ? 1 : (int)max(1ll, (long long)kMaxStepGrid / tq);
  const int unit_tiles =
      (int)max((long long)kMinUnitTiles, ((tt + (tp + 7) / 8 + grid - 1) / grid * 3 + 3) / 4);
  auto units = [&](int s) {  // chunk units of one kv head of sequence s
    const int mt = ceil_div(sq_len[s] * G, BM), npair = (mt + 1) / 2;
    return npair * min(nu, ceil_div(tile_kv<G>(sq_ctx[s], sq_len[s], mt - 1), unit_tiles));
  };
  auto pieces = [&](int s) { return ceil_div(ceil_div(sq_ctx[s], kPage), P); };
  auto bucket = [&](int s) {  // size class of a decode sequence's pieces, in blocks
    const int n = ceil_div(sq_ctx[s], kPage);
    return min(ceil_div(ceil_div(n, pieces(s)), 8), kSizeBuckets - 1);
  };

  // pass 2: per-sequence counts, block exclusive scan over contiguous ranges;
  // slice counts per size bucket
  const int per = ceil_div(S, kPlanWorkers);
  const int s0 = min(S, tid * per), s1 = min(S, s0 + per);
  int cd = 0, cc = 0;
  for (int s = s0; s < s1; ++s) {
    if (sq_len[s] == 1) {
      const int n = Hkv * pieces(s);
      cd += n;
      atomicAdd(&s_hist[bucket(s)], n);
    } else if (sq_len[s] > 1) {
      cc += Hkv * units(s);
    }
  }
  int id = cd, ic = cc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, id, o), b = __shfl_up_sync(0xffffffffu, ic, o);
    if (lane >= o) { id += a; ic += b; }
  }
  if (lane == 31) { s_wd[warp] = id; s_wc[warp] = ic; }
  sync();
  {
    int rd = 0, rc = 0;
    for (int i = 0; i < warp; ++i) { rd += s_wd[i]; rc += s_wc[i]; }
    rd += id - cd;
    rc += ic - cc;
    for (int s = s0; s < s1; ++s) {
      s_dec[s] = rd;
      s_chk[s] = rc;
      if (sq_len[s] == 1) rd += Hkv * pieces(s);
      else if (sq_len[s] > 1) rc += Hkv * units(s);
    }
    if (tid == kPlanWorkers - 1) { s_dec[S] = rd; s_chk[S] = rc; }
  }
  // bucket bases from the largest size down (one bucket per thread)
  static_assert(kSizeBuckets == kPlanWorkers, "one size bucket per plan thread");
  const int hb = kSizeBuckets - 1 - tid;  // thread 0 holds the largest bucket
  const int hc = s_hist[hb];
  int hi = hc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, hi, o);
    if (lane >= o) hi += v;
  }
  sync();  // s_wd of pass 2 read; s_dec, s_chk complete
  if (lane == 31) s_wd[warp] = hi;
  sync();
  {
    int base = 0;
    for (int i = 0; i < warp; ++i) base += s_wd[i];
    s_hist[hb] = base + hi - hc;
  }
  sync();
  // each decode sequence takes the next places of its bucket
  for (int s = tid; s < S; s += kPlanWorkers)
    if (sq_len[s] == 1) s_pos[s] = atomicAdd(&s_hist[bucket(s)], Hkv * pieces(s));
  sync();
  const int Nd = s_dec[S], Nc = s_chk[S];
  auto search = [&](const int *base, int k) {  // last s with base[s] <= k
    int lo = 0, hi2 = S - 1;
    while (lo < hi2) {
      const int mid = (lo + hi2 + 1) >> 1;
      if (base[mid] <= k) lo = mid; else hi2 = mid - 1;
    }
    return lo;
  };
  // Queue order, longest items first: the chunk units (tile pairs from the
  // last, which see the most keys), then the decode slices by size.  The
  // dynamic queue then fills the SMs the chunk units leave free with decode
  // slices from the start, and ends on the shortest slices.
  ItemDesc *list = reinterpret_cast<ItemDesc *>(w.list);
  for (int k = tid; k < Nc; k += kPlanWorkers) {
    const int s = search(s_chk, k);
    const int q_len = sq_len[s];
    const int mt = ceil_div(q_len * G, BM), npair = (mt + 1) / 2;
    const int nus = units(s) / npair;
    const int local = k - s_chk[s];
    const int pair = local / nus, u = local - pair * nus;
    const int mp = npair - 1 - pair / Hkv, g = pair % Hkv;  // later tiles (more keys) first
    ItemDesc d;
    d.s_kind = s;
    d.qs = sq_qs[s];
    d.ctx = sq_ctx[s];
    d.q_len = q_len;
    d.g_x = g | (mp << 8);
    d.a = u | (nus << 16);
    d.b = k;
    d.c = k - u;
    list[k] = d;
  }
  for (int i = tid; i < Nd; i += kPlanWorkers) {
    const int s = search(s_dec, i);
    const int n = ceil_div(sq_ctx[s], kPage), ks = pieces(s);
    const int local = i - s_dec[s];
    const int g = local / ks, piece = local - g * ks;
    ItemDesc d;
    d.s_kind = s | (KIND_DECODE << 30);
    d.qs = sq_qs[s];
    d.ctx = sq_ctx[s];
    d.q_len = ks;
    d.g_x = g | (piece << 8);
    if (n < 46341) {  // piece * n < 2^31: 32-bit division
      d.a = piece * n / ks;
      d.b = (piece + 1) * n / ks;
    } else {
      d.a = (int)((long long)piece * n / ks);
      d.b = (int)((long long)(piece + 1) * n / ks);
    }
    d.c = i;  // partial slot: the slice's own index, whatever its place
    list[Nc + s_pos[s] + local] = d;
  }
  // merge counters of this step start at zero; so does the queue ticket
  for (int x = tid; x < S * Hkv; x += kPlanWorkers) w.dec_ctr[x] = 0u;
  for (int x = tid; x < 2 * Nc; x += kPlanWorkers) w.chunk_ctr[x] = 0u;
  if (tid == 0) {
    w.hdr[0] = Nc;
    w.hdr[1] = Nd;
    w.hdr[2] = Nc + Nd;
    w.hdr[3] = P;
    w.hdr[4] = 0;  // ticket
  }
}

// ---------------------------------------------------------------------------
// Step kernel.

// Keys at positions >= n of a 32-column chunk become -inf.
__device__ __forceinline__ void mask_chunk(uint32_t (&sr)[32], int n) {
#pragma unroll
  for (int e = 0; e < 32; ++e)
    if (e >= n) sr[e] = __float_as_uint(-INFINITY);
}

// p = exp2(s * scale - m) for 32 columns as 16 bf16 (F16: binary16) pairs in
// `pw`; the fp32 row sum (packed pairs) goes to four independent accumulators.
template <bool F16>
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
    pw[h] = F16 ? ptx::pack_f16x2(p0, p1) : ptx::pack_bf16x2(p0, p1);
  }
}

// Output elements: bf16 or binary16 (mode 2: as the caller's dtype says).
template <int KVM>
__device__ __forceinline__ bool out_f16(const AttnParams &p) {
  return KVM == 1 || (KVM == 2 && p.act_f16);
}
__device__ __forceinline__ uint32_t pack_out2(float a, float b, bool f16) {
  return f16 ? ptx::pack_f16x2(a, b) : ptx::pack_bf16x2(a, b);
}
__device__ __forceinline__ uint16_t cvt_out(float a, bool f16) {
  return f16 ? __half_as_ushort(__float2half_rn(a)) : __bfloat16_as_ushort(__float2bfloat16_rn(a));
}

// One page of E4M3 codes (16 rows x D bytes at `src`, row-major) widened to
// binary16 in the 128-byte-swizzled layout the MMAs read: row rr of panel p at
// dst + p * pstride + rr * 128, its 16-byte chunk c at position c ^ (rr & 7).
// Rows >= zrow (cache slots past the sequence) become zeros.  The codes lie
// inside the page's own destination (the last panel's rows at D = 128, the
// second half of the rows at D = 64): taken a group of rows at a time, in
// order, a group's stores land only on its own codes (read before the
// __syncwarp) or on those of groups already done.
template <int D>
__device__ __forceinline__ void widen_page(const unsigned char *src, unsigned char *dst,
                                           int pstride, int zrow, int lane) {
  constexpr int CPR = D / 16;       // 16-byte chunks of codes per row
  constexpr int N = 16 * CPR / 32;  // groups of 32 / CPR rows: 4 (D = 128) or 2 (D = 64)
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int c = lane + 32 * k, rr = c / CPR, cc = c % CPR;
    const uint4 in = *reinterpret_cast<const uint4 *>(src + c * 16);
    __syncwarp();
    uint32_t w[8];
    ptx::e4m3x4_to_f16x4(in.x, w[0], w[1]);
    ptx::e4m3x4_to_f16x4(in.y, w[2], w[3]);
    ptx::e4m3x4_to_f16x4(in.z, w[4], w[5]);
    ptx::e4m3x4_to_f16x4(in.w, w[6], w[7]);
    if (rr >= zrow) {
#pragma unroll
      for (int e = 0; e < 8; ++e) w[e] = 0u;
    }
    const uint4 lo = make_uint4(w[0], w[1], w[2], w[3]), hi = make_uint4(w[4], w[5], w[6], w[7]);
    const int panel = cc >> 2, s = rr & 7;
    unsigned char *row = dst + panel * pstride + rr * 128;
    // dims 16 cc .. 16 cc + 15 are chunks 2 (cc & 3) and 2 (cc & 3) + 1 of the
    // panel row; lanes of odd panels store their second chunk first, so each
    // quarter warp's stores cover all eight bank groups
    const int odd = panel & 1, j0 = 2 * (cc & 3) + odd;
    *reinterpret_cast<uint4 *>(row + ((j0 ^ s) << 4)) = odd ? hi : lo;
    *reinterpret_cast<uint4 *>(row + (((j0 ^ 1) ^ s) << 4)) = odd ? lo : hi;
  }
}

// Which fill of an item the producer issues f-th (K_0, K_1, V_0, K_2, V_1, ...,
// K_{n-1}, V_{n-2}, V_{n-1}): sets is_v and the tile.
__device__ __forceinline__ void fill_of(int f, int n, bool &is_v, int &t) {
  if (f == 0) { is_v = false; t = 0; }
  else if (f == 2 * n - 1) { is_v = true; t = n - 1; }
  else if (f & 1) { is_v = false; t = (f + 1) >> 1; }
  else { is_v = true; t = (f - 2) >> 1; }
}

// Derive an item's geometry from its queue entry (every lane computes the same).
template <int D, int G>
__device__ __forceinline__ void derive_item(const AttnParams &p, const ItemDesc &d, WorkItem &it) {
  constexpr int TM = BM / G;
  it.s = d.s_kind & 0x3fffffff;
  it.qs = d.qs;
  it.ctx = d.ctx;
  it.g = d.g_x & 0xff;
  it.n_pages = ceil_div(d.ctx, kPage);
  if ((d.s_kind >> 30) == KIND_DECODE) {
    it.kind = KIND_DECODE;
    it.q_len = 1;
    it.nsplit = d.q_len;
    it.page0 = d.a;
    it.page_end = d.b;
    it.slot = d.c;
    it.first_slot = d.c - (d.g_x >> 8);
    it.j0 = 0;
    it.n_tiles = ceil_div(d.b - d.a, 8);
    it.n_mine[0] = (it.n_tiles + 1) / 2;
    it.n_mine[1] = it.n_tiles / 2;
    it.mp = 0;
    it.n_kv[0] = it.n_kv[1] = it.n_kv_max = 0;
  } else {
    it.kind = KIND_CHUNK;
    it.q_len = d.q_len;
    it.mp = d.g_x >> 8;
    const int u = d.a & 0xffff, nu = d.a >> 16;
    const int mt = ceil_div(d.q_len * G, BM);
    const int m0 = 2 * it.mp, m1 = m0 + 1;
    it.n_kv[0] = tile_kv<G>(d.ctx, d.q_len, m0);
    it.n_kv[1] = m1 < mt ? tile_kv<G>(d.ctx, d.q_len, m1) : 0;
    const int nkv = max(it.n_kv[0], it.n_kv[1]);
    it.n_kv_max = nkv;
    const int j0 = u * nkv / nu, j1 = (u + 1) * nkv / nu;
    it.j0 = j0;
    it.n_tiles = j1 - j0;
    it.n_mine[0] = max(0, min(j1, it.n_kv[0]) - j0);
    it.n_mine[1] = max(0, min(j1, it.n_kv[1]) - j0);
    it.page0 = 0;
    it.page_end = it.n_pages;
    it.nsplit = nu;
    it.slot = d.b;
    it.first_slot = d.c;
    (void)TM;
  }
}

// Warpgroup-wide sync on an mbarrier of 128 arrivals (bounded).
__device__ __forceinline__ bool wg_sync(uint64_t *bar, uint32_t &phase) {
  ptx::mbar_arrive(bar);
  const bool ok = ptx::mbar_wait(bar, phase & 1);
  ++phase;
  return __all_sync(0xffffffffu, ok);
}

// The V stages in the order the item's tiles use them.  Chunk items cycle
// through stages 0 and 1, decode items through 0, 1 and 2 (the third lives in
// the query-tile region, which decode items do not fill).  Every role replays
// the same sequence, item by item, so all agree on each tile's stage and on
// how many times that stage was filled before.
struct VRing {
  int next = 0, v0 = 0, nst = 2;
  uint32_t c0 = 0, c1 = 0, c2 = 0;  // fills of each stage before this item
  __device__ __forceinline__ void begin(int kind) {
    nst = kind == KIND_DECODE ? 3 : 2;
    if (next >= nst) next = 0;
    v0 = next;
  }
  // (constant divisors: 2 or 3)
  __device__ __forceinline__ int mod(int x) const { return nst == 2 ? (x & 1) : x - 3 * (x / 3); }
  __device__ __forceinline__ int div(int x) const { return nst == 2 ? (x >> 1) : x / 3; }
  __device__ __forceinline__ int stage(int b) const { return mod(v0 + b); }
  // 0-based fill index of tile b's stage
  __device__ __forceinline__ uint32_t use(int b) const {
    const int st = stage(b);
    return (st == 0 ? c0 : (st == 1 ? c1 : c2)) + (uint32_t)div(b);
  }
  __device__ __forceinline__ void end(int n) {
    auto add = [&](int st) -> uint32_t {
      const int first = mod(st - v0 + nst);
      return (st < nst && first < n) ? (uint32_t)(1 + div(n - 1 - first)) : 0u;
    };
    c0 += add(0);
    c1 += add(1);
    c2 += add(2);
    next = mod(v0 + n);
  }
};

template <int KVM, int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
attn_step_kernel(const AttnParams p, const StepWs w, const __grid_constant__ CUtensorMap tm_q,
                 const __grid_constant__ CUtensorMap tm_qd, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, int kv_rows) {
  using C = StepCfg<D>;
  constexpr int TM = BM / G;  // tokens per chunk tile
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char *sQ = smem + C::OFF_Q;
  unsigned char *sK = smem + C::OFF_K;
  unsigned char *sV = smem + C::OFF_V;
  Bars *bs = reinterpret_cast<Bars *>(smem + C::OFF_BAR);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto v_stage = [&](int st) -> unsigned char * {
    return st < 2 ? sV + st * C::KV_BYTES : smem + C::OFF_VX;
  };

  if (tid == 0) {
    for (int i = 0; i < 3; ++i) {
      ptx::mbar_init(&bs->k_full[i], 1);
      ptx::mbar_init(&bs->k_empty[i], 2);
      ptx::mbar_init(&bs->v_full[i], 1);
      ptx::mbar_init(&bs->v_empty[i], 2);
      ptx::mbar_init(&bs->k_conv[i], 256);
      ptx::mbar_init(&bs->v_conv[i], 256);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bs->q_full[i], 1);
      ptx::mbar_init(&bs->q_empty[i], 2);
      ptx::mbar_init(&bs->s_full[i], 1);
      ptx::mbar_init(&bs->p_full[i], 128);
      ptx::mbar_init(&bs->o_final[i], 1);
      ptx::mbar_init(&bs->wg_bar[i], 128);
    }
    for (int i = 0; i < kItemSlots; ++i) {
      ptx::mbar_init(&bs->item_full[i], 1);
      ptx::mbar_init(&bs->item_empty[i], 10);  // 8 softmax warps + 2 MMA warps
    }
    ptx::mbar_init(&bs->hand_off, 128);
    ptx::mbar_init(&bs->release, 128);
    ptx::mbar_init(&bs->mma_done[0], 1);
    ptx::mbar_init(&bs->mma_done[1], 1);
    ptx::fence_mbar_init();
    bs->mma_lock = 0u;
  }
  if (warp == kMmaWarp) ptx::tmem_alloc(&bs->tmem_base, 512);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bs->tmem_base;  // S_i at columns 128*i, O_i at 256 + 128*i
  // everything below reads what the plan kernel wrote
  ptx::grid_dependency_wait();
  const int n_items = __ldcg(w.hdr + 2);

  if (warp == kProducerWarp) {
    // ------------------------------- producer -------------------------------
    if (lane == 0) {
      ptx::prefetch_tmap(&tm_q);
      ptx::prefetch_tmap(&tm_qd);
      ptx::prefetch_tmap(&tm_k);
      ptx::prefetch_tmap(&tm_v);
    }
    const ItemDesc *list = reinterpret_cast<const ItemDesc *>(w.list);
    // every lane polls; the warp moves on (or gives up) together
    auto uwait = [&](uint64_t *bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity));
    };
    // a CTA's first entry is its block index; later ones come from the ticket
    auto claim = [&]() -> int {
      int t = 0;
      if (lane == 0) t = (int)gridDim.x + atomicAdd(w.hdr + 4, 1);
      return __shfl_sync(0xffffffffu, t, 0);
    };
    auto fetch = [&](int t, ItemDesc &d) -> bool {
      if (t >= n_items) return false;
      const int4 *e = reinterpret_cast<const int4 *>(list + t);
      const int4 x = __ldcg(e), y = __ldcg(e + 1);
      d.s_kind = x.x; d.qs = x.y; d.ctx = x.z; d.q_len = x.w;
      d.g_x = y.x; d.a = y.y; d.b = y.z; d.c = y.w;
      return true;
    };
    uint32_t kvc = 0;  // K/V tiles loaded so far by this CTA
    uint32_t issued_k = 0;
    int64_t vlast0 = -1, vlast1 = -1, vlast2 = -1;  // last fill issued into each V stage
    int qlast = -1;                                  // item of the last query load issued
    VRing vr;
    int prev_kind = KIND_DONE;
    bool ok = true;
    int n = 0;
    // The next item is claimed only once every copy of the current one has
    // been issued: the CTA is then close to free (which keeps the queue's
    // longest-first order dynamic), and the claim's latency hides behind the
    // consumers' last queued tiles.  The first entry needs no claim: CTA b
    // takes entry b, so the step starts without a burst of atomics on the
    // ticket and the longest entries go out in block order.
    ItemDesc dsc;
    bool have;
    {
      // entry b lies within the queue's capacity (at least kMaxStepGrid
      // entries) whatever its size: load it alongside the size
      const int4 *e = reinterpret_cast<const int4 *>(list + blockIdx.x);
      const int4 x = __ldcg(e), y = __ldcg(e + 1);
      have = (int)blockIdx.x < n_items;
      dsc.s_kind = x.x; dsc.qs = x.y; dsc.ctx = x.z; dsc.q_len = x.w;
      dsc.g_x = y.x; dsc.a = y.y; dsc.b = y.z; dsc.c = y.w;
    }
    for (;;) {
      WorkItem it;
      if (have) {
        derive_item<D, G>(p, dsc, it);
        if (it.n_tiles == 0) {  // a unit with no keys in its range
          have = fetch(claim(), dsc);
          continue;
        }
      } else {
        it.kind = KIND_DONE;
      }
      const int slot = n % kItemSlots;
      if (n >= kItemSlots && !uwait(&bs->item_empty[slot], ((n / kItemSlots) - 1) & 1)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        bs->items[slot] = it;
        ptx::mbar_arrive(&bs->item_full[slot]);
      }
      __syncwarp();
      if (it.kind == KIND_DONE) break;
      // Query buffers: item n uses set n & 1.  A decode item's Q^T buffer is
      // free once item n - 2's MMAs completed; a chunk's query tiles cover
      // the whole region, so next to a chunk item n - 1's MMAs must be done too.
      const int qb = n & 1;
      if (n >= 2 && !uwait(&bs->q_empty[qb], ((n - 2) >> 1) & 1)) { ok = false; break; }
      if (n >= 1 && (it.kind == KIND_CHUNK || prev_kind == KIND_CHUNK) &&
          !uwait(&bs->q_empty[qb ^ 1], ((n - 1) >> 1) & 1)) {
        ok = false;
        break;
      }
      prev_kind = it.kind;
      qlast = n;
      vr.begin(it.kind);
      if (lane == 0) {
        if (it.kind == KIND_CHUNK) {
          const int nq = (it.n_mine[0] > 0) + (it.n_mine[1] > 0);
          ptx::mbar_arrive_expect_tx(&bs->q_full[qb], nq * C::Q_BYTES);
          for (int i = 0; i < 2; ++i) {
            if (it.n_mine[i] == 0) continue;
#pragma unroll
            for (int pl = 0; pl < C::PANELS; ++pl)
              ptx::tma_load_3d(sQ + i * C::Q_BYTES + pl * BM * 128, &tm_q, pl * 64, it.g * G,
                               it.qs + (2 * it.mp + i) * TM, &bs->q_full[qb]);
          }
        } else {
          // Q^T: the G query rows of the token, [panel][16 rows][64] (rows
          // G..15 are never read back)
          ptx::mbar_arrive_expect_tx(&bs->q_full[qb], C::PANELS * G * 128);
#pragma unroll
          for (int pl = 0; pl < C::PANELS; ++pl)
            ptx::tma_load_3d(sQ + C::OFF_QT + qb * C::QT_BYTES + pl * kDecN * 128, &tm_qd,
                             pl * 64, it.g * G, it.qs, &bs->q_full[qb]);
        }
      }
      // page ids of the item, 32 at a time in this warp's registers (lane l
      // holds page wb + 32 b + l of window b), the next window prefetched
      const int32_t *bt = p.block_table + (int64_t)it.s * p.max_pages;
      const int wb = it.page0 + 8 * it.j0;
      auto load_window = [&](int b) -> int {
        const int pi = wb + 32 * b + lane;
        if (pi >= it.page_end) return kv_rows;  // past the item: zero fill
        const int page = __ldg(bt + pi);
        if (page < 0 || page >= p.num_pages) {
          atomicOr(p.status, STATUS_BAD_PAGE);
          return kv_rows;
        }
        return (page * p.Hkv + it.g) * kPage;
      };
      // V lags K by one tile, so the window before the current one is kept too
      int win_prev = kv_rows, win_cur = load_window(0), win_next = load_window(1), win = 0;
      auto load_tile = [&](unsigned char *dst, bool is_v, uint64_t *bar, int t) {
        const int b = t >> 2;
        while (win < b) {  // warp-uniform
          win_prev = win_cur;
          win_cur = win_next;
          ++win;
          win_next = load_window(win + 1);
        }
        const int src = (b == win) ? win_cur : win_prev;  // b is win or win - 1
        int rows[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) rows[i] = __shfl_sync(0xffffffffu, src, (t & 3) * 8 + i);
        if (KVM == 2) {
          // pages of E4M3 codes into the upper half of each page's destination
          if (lane == 0) {
            ptx::mbar_arrive_expect_tx(bar, 8 * C::PAGE8);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              ptx::tma_load_2d(dst + (is_v ? i * C::PAGE_BYTES + C::V8_OFF : i * kPage * 128 + C::K8_OFF),
                               is_v ? &tm_v : &tm_k, 0, rows[i], bar);
          }
        } else if (lane == 0) {
          ptx::mbar_arrive_expect_tx(bar, C::KV_BYTES);
          if (is_v) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              ptx::tma_load_3d(dst + i * C::PAGE_BYTES, &tm_v, 0, rows[i], 0, bar);
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
              for (int pl = 0; pl < C::PANELS; ++pl)
                ptx::tma_load_2d(dst + pl * BN * 128 + i * kPage * 128, &tm_k, pl * 64, rows[i], bar);
          }
        }
      };
      // K runs one tile ahead of V: K_t, then V_{t-1}
      for (int t = 0; t <= it.n_tiles; ++t) {
        if (t < it.n_tiles) {
          const uint32_t kc = kvc + t, st = kc % C::KST;
          if (kc >= C::KST && !uwait(&bs->k_empty[st], ((kc / C::KST) - 1) & 1)) {
            ok = false;
            break;
          }
          load_tile(sK + st * C::KV_BYTES, false, &bs->k_full[st], t);
          issued_k = kc + 1;
        }
        if (t >= 1) {
          const int st = vr.stage(t - 1);
          const uint32_t u = vr.use(t - 1);
          if (u >= 1 && !uwait(&bs->v_empty[st], (u - 1) & 1)) {
            ok = false;
            break;
          }
          load_tile(v_stage(st), true, &bs->v_full[st], t - 1);
          if (st == 0) vlast0 = u; else if (st == 1) vlast1 = u; else vlast2 = u;
        }
      }
      if (!ok) break;
      vr.end(it.n_tiles);
      kvc += it.n_tiles;
      ++n;
      have = fetch(claim(), dsc);
    }
    if (!ok) {
      if (lane == 0) {
        atomicOr(p.status, STATUS_TIMEOUT);
        // let the copies still in flight land before the CTA leaves
        for (uint32_t c = issued_k > C::KST ? issued_k - C::KST : 0; c < issued_k; ++c)
          ptx::mbar_wait(&bs->k_full[c % C::KST], (c / C::KST) & 1, 1u << 16);
        if (vlast0 >= 0) ptx::mbar_wait(&bs->v_full[0], (uint32_t)vlast0 & 1, 1u << 16);
        if (vlast1 >= 0) ptx::mbar_wait(&bs->v_full[1], (uint32_t)vlast1 & 1, 1u << 16);
        if (vlast2 >= 0) ptx::mbar_wait(&bs->v_full[2], (uint32_t)vlast2 & 1, 1u << 16);
        if (qlast >= 0) ptx::mbar_wait(&bs->q_full[qlast & 1], (qlast >> 1) & 1, 1u << 16);
      }
      __syncwarp();
    }
  } else if (warp >= kMmaWarp) {
    // ------------------------------ MMA issuers --------------------------------
    // One issuing thread per query tile / decode pipeline (warp 9: 0, warp 10:
    // 1).  A commit tracks the issuing thread's own operations.  The K/V stage
    // and Q release barriers take two arrivals: a stage the other issuer does
    // not read is released twice by this one.  A batch (PV and the next QK)
    // enters the tensor pipe whole, under a lock, so the two issuers' batches
    // do not interleave MMA by MMA.
    const int ti = warp - kMmaWarp;
    auto lock = [&]() -> bool {
      for (uint32_t i = 0; i < (1u << 22); ++i) {
        if (atomicCAS(&bs->mma_lock, 0u, 1u) == 0u) return true;
        __nanosleep(32);
      }
      return false;
    };
    auto unlock = [&]() { atomicExch(&bs->mma_lock, 0u); };
    constexpr bool F16 = KVM != 0;  // binary16 operands
    constexpr uint32_t idesc_qk = ptx::idesc_bf16_f32(BM, BN, false, false, F16);
    constexpr uint32_t idesc_pv = ptx::idesc_bf16_f32(BM, D, false, true, F16);
    constexpr uint32_t idesc_qk_d = ptx::idesc_bf16_f32(BN, kDecN, false, false, F16);
    constexpr uint32_t idesc_pv_d = ptx::idesc_bf16_f32(128, kDecN, true, false, F16);
    // a K/V fill is ready for the MMAs once it has landed, or, for an E4M3
    // cache, once the softmax warps have widened it
    uint64_t *const kready = KVM == 2 ? bs->k_conv : bs->k_full;
    uint64_t *const vready = KVM == 2 ? bs->v_conv : bs->v_full;
    const uint32_t tS = tmem + ti * 128, tO = tmem + 256 + ti * 128;
    constexpr int KS = D / 16, VS = BN / 16;
    uint64_t qdesc[KS], kdesc[C::KST][KS], vdesc[3][VS], qtdesc[2][KS], ptdesc[VS];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int o = (ks >> 2) * BM * 128 + (ks & 3) * 32;  // panel, 16-element step
      qdesc[ks] = ptx::smem_desc_sw128(sQ + ti * C::Q_BYTES + o, 16, 1024);
#pragma unroll
      for (int b = 0; b < 2; ++b)
        qtdesc[b][ks] = ptx::smem_desc_sw128(
            sQ + C::OFF_QT + b * C::QT_BYTES + (ks >> 2) * kDecN * 128 + (ks & 3) * 32, 16, 1024);
#pragma unroll
      for (int st = 0; st < C::KST; ++st)
        kdesc[st][ks] = ptx::smem_desc_sw128(sK + st * C::KV_BYTES + o, 16, 1024);
    }
#pragma unroll
    for (int ks = 0; ks < VS; ++ks) {
#pragma unroll
      for (int st = 0; st < 3; ++st)
        vdesc[st][ks] = ptx::smem_desc_sw128(v_stage(st) + ks * C::PAGE_BYTES, kPage * 128, 1024);
      ptdesc[ks] = ptx::smem_desc_sw128(
          sQ + C::OFF_PT + ti * 4096 + (ks >> 2) * kDecN * 128 + (ks & 3) * 32, 16, 1024);
    }
    uint32_t kvm = 0;   // K/V tiles loaded so far for this CTA (all roles agree)
    uint32_t pcnt = 0;  // P tiles of this slot consumed
    VRing vr;
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int slot = n % kItemSlots;
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bs->item_full[slot], (n / kItemSlots) & 1))) {
        ok = false;
        break;
      }
      const WorkItem it = bs->items[slot];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bs->item_empty[slot]);
      if (it.kind == KIND_DONE) break;
      const int n_mine = (ti ? it.n_mine[1] : it.n_mine[0]), n_other = (ti ? it.n_mine[0] : it.n_mine[1]);
      const int qb = n & 1;
      const bool dec = it.kind == KIND_DECODE;
      vr.begin(it.kind);
      if (lane == 0) {
        // Every K/V fill is observed by both issuers, in tile order: the one
        // that reads it releases it with a commit after its MMAs; the other
        // waits until it has landed and releases it with a plain arrival.
        // So neither ever waits on a stage's barrier for a fill more than one
        // ahead of the last it observed, where the parity could not tell the
        // two apart (consecutive fills of a stage can belong to different
        // issuers: decode blocks alternate between them, and a chunk's later
        // tiles may be read by one query tile only).
        auto ack_k1 = [&](int t) -> bool {  // observe K fill of tile t, release it
          const uint32_t kc = kvm + t;
          if (!ptx::mbar_wait(&kready[kc % C::KST], (kc / C::KST) & 1)) return false;
          ptx::mbar_arrive(&bs->k_empty[kc % C::KST]);
          return true;
        };
        auto ack_v1 = [&](int t) -> bool {  // observe V fill of tile t, release it
          const int st = vr.stage(t);
          if (!ptx::mbar_wait(&vready[st], vr.use(t) & 1)) return false;
          ptx::mbar_arrive(&bs->v_empty[st]);
          return true;
        };
        ok = ptx::mbar_wait(&bs->q_full[qb], (n >> 1) & 1);
        if (!dec) {
          // chunk: this tile reads K/V tiles 0 .. n_mine-1 (the later ones, if
          // any, only the other tile reads)
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
          if (ok && n_mine > 0) {
            ok = ptx::mbar_wait(&kready[kvm % C::KST], (kvm / C::KST) & 1) && lock();
            if (ok) {
              ptx::tc_fence_after();
              issue_qk(kvm);
              unlock();
              ptx::mma_commit(&bs->s_full[ti]);
              ptx::mma_commit(&bs->k_empty[kvm % C::KST]);
            }
          }
          for (int j = 0; ok && j < n_mine; ++j) {
            const uint32_t kv = kvm + j;
            const int vst = vr.stage(j);
            const bool more = j + 1 < n_mine;
            if (!ptx::mbar_wait(&bs->p_full[ti], pcnt & 1) ||
                !ptx::mbar_wait(&vready[vst], vr.use(j) & 1) ||
                (more && !ptx::mbar_wait(&kready[(kv + 1) % C::KST], ((kv + 1) / C::KST) & 1)) ||
                !lock()) {
              ok = false;
              break;
            }
            ++pcnt;
            ptx::tc_fence_after();
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {
              if (vst == s2) {
#pragma unroll
                for (int ks = 0; ks < VS; ++ks)
                  ptx::mma_bf16_ts(tO, tS + ks * 8, vdesc[s2][ks], idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
              }
            }
            if (more) issue_qk(kv + 1);
            unlock();
            if (more) {
              ptx::mma_commit(&bs->s_full[ti]);
              ptx::mma_commit(&bs->k_empty[(kv + 1) % C::KST]);
            } else {
              ptx::mma_commit(&bs->o_final[ti]);
            }
            ptx::mma_commit(&bs->v_empty[vst]);
          }
          // The tiles only the other tile reads, observed and released in the
          // order the producer issues them (K_t before V_{t-1}): it may need
          // one of these releases before it can issue a fill waited on here.
          for (int t = n_mine; ok && t <= it.n_tiles; ++t) {
            if (t < it.n_tiles) ok = ack_k1(t);
            if (ok && t > n_mine) ok = ack_v1(t - 1);
          }
        } else {
          // decode: this pipeline reads blocks ti, ti + 2, ...  The item's
          // fills are observed in the producer's order through a cursor: this
          // pipeline's are released by the commit after the MMA that reads
          // them, the other pipeline's with a plain arrival as soon as they are
          // passed.  While it waits for its softmax's P, the issuer moves the
          // cursor over every fill that has already landed, so the other
          // pipeline's stages are released (and refilled) without waiting for
          // this pipeline's next block.
          const int nt = it.n_tiles;
          int oc = 0;
          auto fill_bars = [&](int f, uint64_t *&rdy, uint64_t *&emp, uint32_t &par) -> bool {
            bool is_v;
            int t;
            fill_of(f, nt, is_v, t);
            if (is_v) {
              const int st = vr.stage(t);
              rdy = &vready[st];
              emp = &bs->v_empty[st];
              par = vr.use(t) & 1;
            } else {
              const uint32_t kc = kvm + t;
              rdy = &kready[kc % C::KST];
              emp = &bs->k_empty[kc % C::KST];
              par = (kc / C::KST) & 1;
            }
            return (t & 1) != ti;  // the other pipeline's fill
          };
          auto observe_through = [&](int last) -> bool {  // waits for each fill
            for (; oc <= last && oc < 2 * nt; ++oc) {
              uint64_t *rdy, *emp;
              uint32_t par;
              const bool other = fill_bars(oc, rdy, emp, par);
              if (!ptx::mbar_wait(rdy, par)) return false;
              if (other) ptx::mbar_arrive(emp);
            }
            return true;
          };
          auto observe_landed = [&]() {  // only the fills already ready
            while (oc < 2 * nt) {
              uint64_t *rdy, *emp;
              uint32_t par;
              const bool other = fill_bars(oc, rdy, emp, par);
              if (!ptx::mbar_test(rdy, par)) break;
              if (other) ptx::mbar_arrive(emp);
              ++oc;
            }
          };
          auto kfill = [&](int t) { return t == 0 ? 0 : 2 * t - 1; };                // fill index of K_t
          auto vfill = [&](int t) { return t == nt - 1 ? 2 * nt - 1 : 2 * t + 2; };  // of V_t
          auto issue_qk = [&](uint32_t kvidx) {
            const uint32_t st = kvidx % C::KST;
#pragma unroll
            for (int s3 = 0; s3 < C::KST; ++s3) {
              if (st == (uint32_t)s3) {
#pragma unroll
                for (int ks = 0; ks < KS; ++ks)
                  ptx::mma_bf16_ss(tS, kdesc[s3][ks], qb ? qtdesc[1][ks] : qtdesc[0][ks], idesc_qk_d,
                                   ks > 0 ? 1u : 0u);
              }
            }
          };
          if (ok && n_mine > 0) {
            const uint32_t kv0 = kvm + ti;
            ok = observe_through(kfill(ti)) && lock();
            if (ok) {
              ptx::tc_fence_after();
              issue_qk(kv0);
              unlock();
              ptx::mma_commit(&bs->s_full[ti]);
              ptx::mma_commit(&bs->k_empty[kv0 % C::KST]);
            }
          }
          for (int j = 0; ok && j < n_mine; ++j) {
            const int t = ti + 2 * j;
            const uint32_t kv = kvm + t;
            const int vst = vr.stage(t);
            const bool more = j + 1 < n_mine;
            // P_t, moving the cursor over landed fills meanwhile; then V_t and
            // K_{t+2} with everything before them in the producer's order
            bool got = false;
            for (uint32_t i = 0; i < (1u << 22) && !got; ++i) {
              got = ptx::mbar_test(&bs->p_full[ti], pcnt & 1);
              if (!got) {
                observe_landed();
                got = ptx::mbar_try_wait(&bs->p_full[ti], pcnt & 1);
              }
            }
            if (!got || !observe_through(more ? kfill(t + 2) : vfill(t)) || !lock()) {
              ok = false;
              break;
            }
            ++pcnt;
            ptx::tc_fence_after();
#pragma unroll
            for (int s2 = 0; s2 < 3; ++s2) {
              if (vst == s2) {
#pragma unroll
                for (int ks = 0; ks < VS; ++ks)
                  ptx::mma_bf16_ss(tO, vdesc[s2][ks], ptdesc[ks], idesc_pv_d,
                                   (j > 0 || ks > 0) ? 1u : 0u);
              }
            }
            if (more) issue_qk(kv + 2);
            unlock();
            if (more) {
              ptx::mma_commit(&bs->s_full[ti]);
              ptx::mma_commit(&bs->k_empty[(kv + 2) % C::KST]);
            } else {
              ptx::mma_commit(&bs->o_final[ti]);
            }
            ptx::mma_commit(&bs->v_empty[vst]);
          }
          // the rest of the item's fills (the other pipeline's last blocks)
          if (ok) ok = observe_through(2 * nt - 1);
        }
        if (ok) {
          if (n_mine > 0) {
            ptx::mma_commit(&bs->q_empty[qb]);
          } else {
            ptx::mbar_arrive(&bs->q_empty[qb]);
          }
        }
        (void)n_other;
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      vr.end(it.n_tiles);
      kvm += it.n_tiles;
    }
    if (lane == 0) {
      if (!ok) atomicOr(p.status, STATUS_TIMEOUT);
      // every MMA this thread issued has completed before TMEM is freed
      ptx::mma_commit(&bs->mma_done[ti]);
      ptx::mbar_wait(&bs->mma_done[ti], 0, 1u << 20);
    }
    __syncwarp();
  } else {
    // ------------------------------- softmax ------------------------------------
    const int ti = warp >> 2;                 // query tile slot / decode pipeline
    const int quarter = warp & 3;             // TMEM lane quarter this warp may access
    const int r = quarter * 32 + lane;        // tile row (chunk) / key of the block (decode)
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t tS = tmem + ti * 128 + lane_off;
    const uint32_t tO = tmem + 256 + ti * 128 + lane_off;
    const float sl2 = p.scale_log2;
    constexpr bool F16 = KVM != 0;
    const bool of16 = out_f16<KVM>(p);
    uint32_t scnt = 0, ocnt = 0, wgp = 0, nfin = 0;
    uint32_t kvs = 0;  // K/V tiles of the items before this one (all roles agree)
    VRing vr;
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int slot = n % kItemSlots;
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bs->item_full[slot], (n / kItemSlots) & 1))) {
        ok = false;
        break;
      }
      const WorkItem it = bs->items[slot];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bs->item_empty[slot]);
      if (it.kind == KIND_DONE) break;
      const int n_mine = (ti ? it.n_mine[1] : it.n_mine[0]);
      const int ctx = it.ctx;
      vr.begin(it.kind);
      // E4M3 cache: widen the item's fills, in the producer's order, up to
      // fill `last` (this warp: page `warp` of each tile).  Every softmax warp
      // takes part in every fill, so each observes every fill of every stage.
      int cf = 0;
      auto widen_through = [&](int last) -> bool {
        const int nf = 2 * it.n_tiles;
        for (; cf <= last && cf < nf; ++cf) {
          bool is_v;
          int t;
          fill_of(cf, it.n_tiles, is_v, t);
          unsigned char *stage;
          uint64_t *full, *conv;
          uint32_t par;
          if (is_v) {
            const int st = vr.stage(t);
            stage = v_stage(st);
            full = &bs->v_full[st];
            conv = &bs->v_conv[st];
            par = vr.use(t) & 1;
          } else {
            const uint32_t kc = kvs + t;
            stage = sK + (kc % C::KST) * C::KV_BYTES;
            full = &bs->k_full[kc % C::KST];
            conv = &bs->k_conv[kc % C::KST];
            par = (kc / C::KST) & 1;
          }
          if (!__all_sync(0xffffffffu, ptx::mbar_wait(full, par))) return false;
          const int key0 = (it.page0 + 8 * (it.j0 + t) + warp) * kPage;  // this page's first key
          if (is_v)
            widen_page<D>(stage + warp * C::PAGE_BYTES + C::V8_OFF, stage + warp * C::PAGE_BYTES,
                          kPage * 128, ctx - key0, lane);
          else
            widen_page<D>(stage + warp * kPage * 128 + C::K8_OFF, stage + warp * kPage * 128,
                          BN * 128, ctx - key0, lane);
          ptx::fence_proxy_async_smem();
          ptx::mbar_arrive(conv);
        }
        return true;
      };
      if (it.kind == KIND_CHUNK) {
        const int q_len = it.q_len;
        const int tok = (2 * it.mp + ti) * TM + r / G;  // index within the chunk
        const bool row_valid = tok < q_len;
        const int last = row_valid ? ctx - q_len + tok : 0;
        float m_run = -INFINITY, l_run = 0.f;
        for (int j = 0; j < n_mine; ++j, ++scnt) {
          // the fills the MMAs after P_j need (V_j, K_{j+1}), before waiting S_j
          if (KVM == 2 && !widen_through(2 * j + 2)) { ok = false; break; }
          if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bs->s_full[ti], scnt & 1))) { ok = false; break; }
          ptx::tc_fence_after();
          const int key0 = (it.j0 + j) * BN;
          const bool diag = key0 + BN - 1 > last;  // tile holds keys past `last`
          const int nvis = last - key0 + 1;        // visible keys of this row in the tile
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
          const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sl2;
          const bool move = tmax > m_run + kRescaleThreshold;
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
            exp_chunk_regs<F16>(sa, sc2, nm2, rs2, w16);
            ptx::tmem_st16(tS + c * 16, w16);
            ptx::tmem_wait_ld_regs(sb);
            if (diag) mask_chunk(sb, nvis - (c + 1) * 32);
            exp_chunk_regs<F16>(sb, sc2, nm2, rs2, w16);
            ptx::tmem_st16(tS + (c + 1) * 16, w16);
          }
          {
            const uint64_t r2 = ptx::fadd2(ptx::fadd2(rs2[0], rs2[1]), ptx::fadd2(rs2[2], rs2[3]));
            float rs0, rs1;
            ptx::unpack2(r2, rs0, rs1);
            l_run += rs0 + rs1;
          }
          // Cache slots at or past ctx in the last page may hold anything (NaN
          // included) and 0 * NaN is NaN inside PV: zero those V rows first
          // (an E4M3 cache: already zeroed by the widening).
          if (KVM != 2 && key0 + BN > ctx) {
            const int vst = vr.stage(j);
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bs->v_full[vst], vr.use(j) & 1))) {
              ok = false;
              break;
            }
            if (r >= ctx - key0 && r < it.n_pages * kPage - key0) {
              unsigned char *vrow = v_stage(vst) + (r / kPage) * C::PAGE_BYTES + (r % kPage) * 128;
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
        // the rest of the item's fills (the other query tile may read them)
        if (KVM == 2 && ok && !widen_through(2 * it.n_tiles - 1)) ok = false;
        vr.end(it.n_tiles);
        kvs += it.n_tiles;
        if (!ok) break;
        if (n_mine == 0) continue;
        // epilogue: O / l, or this unit's partial and, from the last unit of
        // the pair to finish, the merge of all of them
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bs->o_final[ti], ocnt & 1))) { ok = false; break; }
        ++ocnt;
        ptx::tc_fence_after();
        const int64_t orow = ((int64_t)(it.qs + tok) * p.Hq + it.g * G + r % G) * D;
        uint16_t *out = static_cast<uint16_t *>(p.out) + orow;
        if (it.nsplit == 1) {
          const float inv = (KVM == 2 ? p.v_scale : 1.f) / l_run;
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
                  wds[h] = pack_out2(__uint_as_float(o[q4 * 8 + h * 2]) * inv,
                                     __uint_as_float(o[q4 * 8 + h * 2 + 1]) * inv, of16);
                *reinterpret_cast<uint4 *>(out + c * 32 + q4 * 8) =
                    make_uint4(wds[0], wds[1], wds[2], wds[3]);
              }
            }
          }
          ptx::tc_fence_before();
          continue;
        }
        // partial of this unit: [slot][tile][D/4][128 rows] float4, (max, sum)
        {
          float4 *po = reinterpret_cast<float4 *>(w.chunk_o) + ((int64_t)it.slot * 2 + ti) * (D / 4) * 128;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            ptx::tmem_ld32(tO + c * 32, o);
            ptx::tmem_wait_ld_regs(o);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              po[(c * 8 + q4) * 128 + r] =
                  make_float4(__uint_as_float(o[4 * q4]), __uint_as_float(o[4 * q4 + 1]),
                              __uint_as_float(o[4 * q4 + 2]), __uint_as_float(o[4 * q4 + 3]));
          }
          w.chunk_ml[((int64_t)it.slot * 2 + ti) * 128 + r] = make_float2(m_run, l_run);
        }
        ptx::tc_fence_before();
        __threadfence();
        if (!wg_sync(&bs->wg_bar[ti], wgp)) { ok = false; break; }
        if (quarter == 0 && lane == 0)
          bs->bcast[ti] = (int)atomicAdd(w.chunk_ctr + (int64_t)it.first_slot * 2 + ti, 1u);
        if (!wg_sync(&bs->wg_bar[ti], wgp)) { ok = false; break; }
        const int prev = bs->bcast[ti];
        // contributors: the units of the pair whose range holds keys of this tile
        const int nu = it.nsplit, nkv = it.n_kv_max, mine_kv = (ti ? it.n_kv[1] : it.n_kv[0]);
        int ncontrib = 0;
        for (int u = 0; u < nu; ++u) {
          const int a0 = u * nkv / nu, a1 = (u + 1) * nkv / nu;
          ncontrib += (a0 < a1 && a0 < mine_kv);
        }
        if (prev != ncontrib - 1 || !row_valid) continue;
        __threadfence();
        float M = -INFINITY;
        for (int u = 0; u < nu; ++u) {
          const int a0 = u * nkv / nu, a1 = (u + 1) * nkv / nu;
          if (!(a0 < a1 && a0 < mine_kv)) continue;
          M = fmaxf(M, __ldcg(&w.chunk_ml[((int64_t)(it.first_slot + u) * 2 + ti) * 128 + r]).x);
        }
        float L = 0.f;
        for (int u = 0; u < nu; ++u) {
          const int a0 = u * nkv / nu, a1 = (u + 1) * nkv / nu;
          if (!(a0 < a1 && a0 < mine_kv)) continue;
          const float2 ml = __ldcg(&w.chunk_ml[((int64_t)(it.first_slot + u) * 2 + ti) * 128 + r]);
          L = fmaf(ml.y, ml.x == -INFINITY ? 0.f : ptx::ex2(ml.x - M), L);
        }
        const float inv = (KVM == 2 ? p.v_scale : 1.f) / L;
        // 32 output dims at a time over every contributor
#pragma unroll 1
        for (int cg = 0; cg < D / 32; ++cg) {
          float acc[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) acc[e] = 0.f;
          for (int u = 0; u < nu; ++u) {
            const int a0 = u * nkv / nu, a1 = (u + 1) * nkv / nu;
            if (!(a0 < a1 && a0 < mine_kv)) continue;
            const int64_t sl = (int64_t)(it.first_slot + u) * 2 + ti;
            const float2 ml = __ldcg(&w.chunk_ml[sl * 128 + r]);
            const float wgt = ml.x == -INFINITY ? 0.f : ptx::ex2(ml.x - M);
            const float4 *src = reinterpret_cast<const float4 *>(w.chunk_o) + (sl * (D / 4) + cg * 8) * 128 + r;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const float4 v = __ldcg(src + c * 128);
              acc[4 * c] = fmaf(v.x, wgt, acc[4 * c]);
              acc[4 * c + 1] = fmaf(v.y, wgt, acc[4 * c + 1]);
              acc[4 * c + 2] = fmaf(v.z, wgt, acc[4 * c + 2]);
              acc[4 * c + 3] = fmaf(v.w, wgt, acc[4 * c + 3]);
            }
          }
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t wds[4];
#pragma unroll
            for (int h = 0; h < 4; ++h)
              wds[h] = pack_out2(acc[8 * c + 2 * h] * inv, acc[8 * c + 2 * h + 1] * inv, of16);
            *reinterpret_cast<uint4 *>(out + cg * 32 + c * 8) = make_uint4(wds[0], wds[1], wds[2], wds[3]);
          }
        }
      } else {
        // ------------------------------ decode slice ------------------------------
        // thread = key r of each 128-key block; rows = the G query heads
        float m_run[G], l_part[G];
#pragma unroll
        for (int q = 0; q < G; ++q) { m_run[q] = -INFINITY; l_part[q] = 0.f; }
        const int key_lim = min(ctx, it.page_end * kPage);
        unsigned char *pt = smem + C::OFF_PT + ti * 4096;
        for (int j = 0; j < n_mine; ++j, ++scnt) {
          const int blk = ti + 2 * j;
          // the fills the MMAs after P_blk need (up to K_{blk+2}), before
          // waiting S_blk
          if (KVM == 2 && !widen_through(2 * blk + 3)) { ok = false; break; }
          if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bs->s_full[ti], scnt & 1))) { ok = false; break; }
          ptx::tc_fence_after();
          uint32_t sr[G];
          ptx::tmem_ld_cols<G>(tS, sr);
          const int key = (it.page0 + 8 * blk) * kPage + r;
          const bool valid = key < key_lim;
          float sv[G];
#pragma unroll
          for (int q = 0; q < G; ++q) {
            sv[q] = valid ? __uint_as_float(sr[q]) * sl2 : -INFINITY;
            float v = sv[q];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) bs->red[ti][j & 1][quarter][q] = v;
          }
          if (!wg_sync(&bs->wg_bar[ti], wgp)) { ok = false; break; }
          float alpha[G];
          bool any = false;
#pragma unroll
          for (int q = 0; q < G; ++q) {
            const float bm = fmaxf(fmaxf(bs->red[ti][j & 1][0][q], bs->red[ti][j & 1][1][q]),
                                   fmaxf(bs->red[ti][j & 1][2][q], bs->red[ti][j & 1][3][q]));
            const bool move = bm > m_run[q] + kRescaleThreshold;
            alpha[q] = (move && m_run[q] != -INFINITY) ? ptx::ex2(m_run[q] - bm) : 1.f;
            if (move) m_run[q] = bm;
            any |= alpha[q] != 1.f;
          }
          // alpha is the same on every thread: the whole warpgroup rescales O^T
          if (j > 0 && any) {
            uint32_t o[G];
            ptx::tmem_ld_cols<G>(tO, o);
#pragma unroll
            for (int q = 0; q < G; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha[q]);
            ptx::tmem_st_cols<G>(tO, o);
          }
#pragma unroll
          for (int q = 0; q < G; ++q) {
            const float pq = (valid && m_run[q] != -INFINITY) ? ptx::ex2(sv[q] - m_run[q]) : 0.f;
            l_part[q] = l_part[q] * alpha[q] + pq;
            // P^T, K-major: row q, key r; [panel r/64][16 rows][64 keys] swizzled
            const uint32_t off = (r >> 6) * (kDecN * 128) + q * 128 +
                                 ((((r & 63) >> 3) ^ (q & 7)) << 4) + (r & 7) * 2;
            *reinterpret_cast<uint16_t *>(pt + off) = cvt_out(pq, F16);
          }
          // cache slots past ctx in the sequence's last page: zero their V rows
          // (an E4M3 cache: already zeroed by the widening)
          const int key0 = (it.page0 + 8 * blk) * kPage;
          if (KVM != 2 && key0 + BN > ctx && key0 < it.n_pages * kPage) {
            const int vst = vr.stage(blk);
            if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bs->v_full[vst], vr.use(blk) & 1))) {
              ok = false;
              break;
            }
            if (key >= ctx && key < min(it.n_pages, it.page_end) * kPage) {
              unsigned char *vrow = v_stage(vst) + (r / kPage) * C::PAGE_BYTES + (r % kPage) * 128;
#pragma unroll
              for (int pl = 0; pl < C::PANELS; ++pl)
#pragma unroll
                for (int c = 0; c < 8; ++c)
                  *reinterpret_cast<uint4 *>(vrow + pl * kPage * 128 + c * 16) = make_uint4(0, 0, 0, 0);
            }
          }
          ptx::fence_proxy_async_smem();
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          ptx::mbar_arrive(&bs->p_full[ti]);
        }
        // the rest of the item's fills (the other pipeline's last blocks)
        if (KVM == 2 && ok && !widen_through(2 * it.n_tiles - 1)) ok = false;
        vr.end(it.n_tiles);
        kvs += it.n_tiles;
        if (!ok) break;
        if (n_mine > 0) {
          if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bs->o_final[ti], ocnt & 1))) { ok = false; break; }
          ++ocnt;
          ptx::tc_fence_after();
        }
        // the pipeline's row sums over its 128 threads
        float L[G];
#pragma unroll
        for (int q = 0; q < G; ++q) {
          float v = l_part[q];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) bs->red[ti][2][quarter][q] = v;
        }
        if (!wg_sync(&bs->wg_bar[ti], wgp)) { ok = false; break; }
#pragma unroll
        for (int q = 0; q < G; ++q)
          L[q] = (bs->red[ti][2][0][q] + bs->red[ti][2][1][q]) +
                 (bs->red[ti][2][2][q] + bs->red[ti][2][3][q]);
        if (ti == 1) {
          // hand (max, sum) to pipeline 0, which reads this pipeline's O^T
          // from TMEM, and wait until it has
          if (r == 0) {
#pragma unroll
            for (int q = 0; q < G; ++q)
              bs->mlx[q] = n_mine > 0 ? make_float2(m_run[q], L[q]) : make_float2(-INFINITY, 0.f);
          }
          // every thread has read red[1][2] before it is written again
          if (!wg_sync(&bs->wg_bar[ti], wgp)) { ok = false; break; }
          ptx::tc_fence_before();
          ptx::mbar_arrive(&bs->hand_off);
          if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bs->release, nfin & 1))) { ok = false; break; }
          ++nfin;
          continue;
        }
        if (!wg_sync(&bs->wg_bar[ti], wgp)) { ok = false; break; }
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&bs->hand_off, nfin & 1))) { ok = false; break; }
        ++nfin;
        ptx::tc_fence_after();
        const bool other = it.n_mine[1] > 0;
        float a0[G], a1[G], Lt[G], Mt[G];
#pragma unroll
        for (int q = 0; q < G; ++q) {
          const float2 x = bs->mlx[q];
          Mt[q] = fmaxf(m_run[q], x.x);
          a0[q] = m_run[q] == -INFINITY ? 0.f : ptx::ex2(m_run[q] - Mt[q]);
          a1[q] = x.x == -INFINITY ? 0.f : ptx::ex2(x.x - Mt[q]);
          Lt[q] = L[q] * a0[q] + x.y * a1[q];
        }
        uint32_t o0[G], o1[G];
        ptx::tmem_ld_cols<G>(tO, o0);
        if (other) {
          ptx::tmem_ld_cols<G>(tmem + 256 + 128 + lane_off, o1);
        } else {
#pragma unroll
          for (int q = 0; q < G; ++q) o1[q] = 0u;
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(&bs->release);
        float O[G];
#pragma unroll
        for (int q = 0; q < G; ++q)
          O[q] = __uint_as_float(o0[q]) * a0[q] + (other ? __uint_as_float(o1[q]) * a1[q] : 0.f);
        const int d = r;  // O^T lane = head dim
        const int64_t obase = ((int64_t)it.qs * p.Hq + it.g * G) * D;
        uint16_t *out = static_cast<uint16_t *>(p.out) + obase;
        if (it.nsplit == 1) {
          if (d < D) {
#pragma unroll
            for (int q = 0; q < G; ++q)
              out[q * D + d] = cvt_out(KVM == 2 ? O[q] * (p.v_scale / Lt[q]) : O[q] / Lt[q], of16);
          }
          continue;
        }
        // partial of this slice, then the merge by the segment's last slice
        if (d < D) {
#pragma unroll
          for (int q = 0; q < G; ++q) w.dec_o[((int64_t)it.slot * G + q) * D + d] = O[q];
        }
        if (r == 0) {
#pragma unroll
          for (int q = 0; q < G; ++q) w.dec_ml[(int64_t)it.slot * G + q] = make_float2(Mt[q], Lt[q]);
        }
        __threadfence();
        if (!wg_sync(&bs->wg_bar[ti], wgp)) { ok = false; break; }
        if (r == 0) bs->bcast[ti] = (int)atomicAdd(w.dec_ctr + (int64_t)it.s * p.Hkv + it.g, 1u);
        if (!wg_sync(&bs->wg_bar[ti], wgp)) { ok = false; break; }
        if (bs->bcast[ti] != it.nsplit - 1) continue;
        __threadfence();
        float M[G], acc[G], Ls[G];
#pragma unroll
        for (int q = 0; q < G; ++q) { M[q] = -INFINITY; acc[q] = 0.f; Ls[q] = 0.f; }
        for (int c = 0; c < it.nsplit; ++c) {
#pragma unroll
          for (int q = 0; q < G; ++q)
            M[q] = fmaxf(M[q], __ldcg(&w.dec_ml[((int64_t)it.first_slot + c) * G + q]).x);
        }
        for (int c = 0; c < it.nsplit; ++c) {
          const int64_t sl = (int64_t)it.first_slot + c;
#pragma unroll
          for (int q = 0; q < G; ++q) {
            const float2 ml = __ldcg(&w.dec_ml[sl * G + q]);
            const float wgt = ml.x == -INFINITY ? 0.f : ptx::ex2(ml.x - M[q]);
            Ls[q] = fmaf(ml.y, wgt, Ls[q]);
            if (d < D) acc[q] = fmaf(__ldcg(&w.dec_o[(sl * G + q) * D + d]), wgt, acc[q]);
          }
        }
        if (d < D) {
#pragma unroll
          for (int q = 0; q < G; ++q)
            out[q * D + d] = cvt_out(KVM == 2 ? acc[q] * (p.v_scale / Ls[q]) : acc[q] / Ls[q], of16);
        }
      }
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

template <int KVM, int D, int G>
cudaError_t launch_dg(const AttnParams &p, const StepWs &w, cudaStream_t stream) {
  using C = StepCfg<D>;
  auto encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  CUtensorMap tq, tqd, tk, tv;
  // q viewed as [T][Hq][D]: chunk box = 64 dims x G heads x BM/G tokens,
  // decode box = 64 dims x G heads x 1 token.  E4M3 cache: the binary16
  // queries (the caller's, or the plan kernel's copy of bf16 ones).
  {
    const void *qsrc = (KVM == 2 && !p.act_f16) ? p.q16 : p.q;
    const CUtensorMapDataType qt =
        KVM == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.Hq, (cuuint64_t)p.num_tokens};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)p.Hq * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(BM / G)};
    cuuint32_t estr[3] = {1, 1, 1};
    if (encode(&tq, qt, 3, const_cast<void *>(qsrc), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    box[2] = 1;
    if (encode(&tqd, qt, 3, const_cast<void *>(qsrc), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const int64_t rows = p.num_pages * p.Hkv * kPage;
  if (KVM == 2) {
    // E4M3 caches: rows of D one-byte codes, box = one page (16 rows),
    // unswizzled (the widening reads it row-major)
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)D};
    cuuint32_t box[2] = {(cuuint32_t)D, (cuuint32_t)kPage};
    cuuint32_t estr[2] = {1, 1};
    if (encode(&tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(p.k_cache), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if (encode(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(p.v_cache), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  } else {
    const CUtensorMapDataType kt =
        KVM == 0 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    {
      // K: cache rows [rows][D], box = one 64-dim panel of one page (16 rows)
      cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
      cuuint64_t strides[1] = {(cuuint64_t)D * 2};
      cuuint32_t box[2] = {64, (cuuint32_t)kPage};
      cuuint32_t estr[2] = {1, 1};
      if (encode(&tk, kt, 2, const_cast<void *>(p.k_cache), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
    {
      // V: the same rows viewed as (64 dims, row, panel), box = a whole page
      // with its panels outermost, [panel][16 rows][64 dims] in shared memory
      cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)C::PANELS};
      cuuint64_t strides[2] = {(cuuint64_t)D * 2, 128};
      cuuint32_t box[3] = {64, (cuuint32_t)kPage, (cuuint32_t)C::PANELS};
      cuuint32_t estr[3] = {1, 1, 1};
      if (encode(&tv, kt, 3, const_cast<void *>(p.v_cache), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
  }
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_step_kernel<KVM, D, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  // the plan (with its side work: the fused append, the queries' copy) ...
  const int64_t side = plan_append_pieces<KVM>(p) + plan_q_pieces<KVM>(p);
  const int side_ctas = (int)std::min<int64_t>(w.grid, (side + 4 * kPlanThreads - 1) / (4 * kPlanThreads));
  static bool plan_configured = false;
  if (!plan_configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_plan_kernel<KVM, G>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)plan_smem_bytes(kDecodeMaxSeqs));
    if (e != cudaSuccess) return e;
    plan_configured = true;
  }
  attn_plan_kernel<KVM, G><<<1 + side_ctas, kPlanThreads, plan_smem_bytes(p.num_seqs), stream>>>(p, w);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // ... then the step, allowed to start while the plan finishes
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(w.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_step_kernel<KVM, D, G>, p, w, tq, tqd, tk, tv, (int)rows);
}

}  // namespace

template <int KVM>
cudaError_t launch_step(const AttnParams &p, const StepWs &w, cudaStream_t stream) {
  const int G = p.Hq / p.Hkv;
  if (p.D == 128) {
    switch (G) {
      case 1: return launch_dg<KVM, 128, 1>(p, w, stream);
      case 2: return launch_dg<KVM, 128, 2>(p, w, stream);
      case 4: return launch_dg<KVM, 128, 4>(p, w, stream);
      case 8: return launch_dg<KVM, 128, 8>(p, w, stream);
    }
  } else {
    switch (G) {
      case 1: return launch_dg<KVM, 64, 1>(p, w, stream);
      case 2: return launch_dg<KVM, 64, 2>(p, w, stream);
      case 4: return launch_dg<KVM, 64, 4>(p, w, stream);
      case 8: return launch_dg<KVM, 64, 8>(p, w, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace cpa
