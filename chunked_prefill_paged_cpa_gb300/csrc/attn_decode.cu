// Decode attention: the bandwidth-bound part of a hybrid step.
//
// A decode has one query token that reads its sequence's whole KV cache
// ("Chunked Prefill" (deepconcepts.dev), "Why a chunk can be nearly free": a
// decode pass is bandwidth-bound by a wide margin; "How Chunked Prefill Stops
// Decode Starvation", "The stall": decode reads the full KV cache from HBM
// every step).  The kernel is built to stream that cache at HBM speed.
//
// Work decomposition (stream-K over warps).  All decode sequences' pages, for
// every kv head, are laid end to end into one "page stream": segment
// (s, g) = the n_s pages of sequence s seen by kv head g.  A persistent grid of
// one CTA per SM runs 8 warps; every warp is an independent worker that takes
// an equal contiguous slice of the page stream.  A slice may start or end
// inside a segment; a worker that holds a whole segment writes its output
// directly, otherwise it writes a partial (row max, row sum, unnormalised
// output) and the last of the segment's contributors to arrive merges them
// with log-sum-exp weights ("Chunked Prefill 技术深度解析", section 7.2:
// softmax over the visible keys, combined incrementally).  No thread ever
// waits for another CTA.
//
// Per warp: a ring of NST stages in shared memory, each holding one page of K
// and one page of V for one kv head (2 x 4 KB at head_dim 128), filled by
// bulk asynchronous copies (TMA, cp.async.bulk) that lane 0 issues NST pages
// ahead; block-table entries are fetched 32 at a time by the whole warp.
// Compute (GQA: the G query heads of one kv head are done together, so every
// K/V byte is read once): lanes form 4 groups of 8; a group owns 4 of the
// page's 16 keys, a lane owns head_dim/8 dimensions.  QK^T uses packed fp32
// FMAs and a butterfly reduce-scatter inside each 8-lane group; softmax is
// online (log2 domain) per group; PV reads the probabilities through a small
// per-warp shared buffer.
//
// Fused append (cpa_append_attention_forward): a second instantiation copies
// the step's new K/V rows into the cache (the CTAs that start after the chunk
// kernel, else all of them) and takes each decode's own row from the step's
// inputs, so no separate append launch has to finish first.
#include "cpa_internal.cuh"
#include "ptx.cuh"

namespace cpa {
namespace {

constexpr int kWarps = 8;
constexpr int kPage = 16;
constexpr float kLazyRescale = 8.0f;  // log2 units
// Split estimate when part of the grid starts after the chunk kernel: one KV
// tile of a chunk work item at head_dim 128, the fixed cost of an item (Q
// load, first tile, epilogue), and the page rate of one decode CTA beside it.
constexpr double kChunkIterNs = 2200.0;
constexpr double kChunkItemNs = 12000.0;
constexpr double kDecodeBytesPerNs = 34.0;

template <int D>
struct Cfg {
  static constexpr int DL = D / 8;                  // dims per lane
  static constexpr int CH = DL / 8;                 // 16-byte chunks per lane per key row
  static constexpr int PAGE_BYTES = kPage * D * 2;  // one kv head's page, bf16
  static constexpr int STAGE_BYTES = 2 * PAGE_BYTES;
  static constexpr int NST = (192 * 1024) / (kWarps * STAGE_BYTES);  // 192 KB of ring per CTA
};

// Dynamic shared memory: [ring][mbarriers][stage-valid flags][p buffers][seq offsets]
template <int D, int G>
struct Layout {
  static constexpr int RING = kWarps * Cfg<D>::NST * Cfg<D>::STAGE_BYTES;
  static constexpr int BARS = RING;
  static constexpr int FLAGS = BARS + kWarps * Cfg<D>::NST * 8;
  static constexpr int PBUF = (FLAGS + kWarps * Cfg<D>::NST * 4 + 15) / 16 * 16;
  static constexpr int OFFS = PBUF + kWarps * kPage * G * 4;
  static size_t bytes(int num_seqs) { return OFFS + (size_t)(num_seqs + 1) * 4; }
};

__device__ __forceinline__ int seq_decode_pages(const AttnParams &p, int s) {
  const int q_len = __ldg(p.query_start_loc + s + 1) - __ldg(p.query_start_loc + s);
  if (q_len != 1) return 0;
  int ctx = __ldg(p.seq_lens + s);
  const int cap = p.max_pages * kPage;
  if (ctx > cap) ctx = cap;
  if (ctx < 1) return 0;
  return (ctx + kPage - 1) / kPage;
}

// Cursor over the page stream: position -> (sequence, kv head, page index).
struct Cursor {
  int s, g, pi, n;  // n = pages of sequence s
};

__device__ __forceinline__ Cursor locate(const int *off, int num_seqs, int Hkv, int64_t pos) {
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {  // last s with off[s] <= pos
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= pos) lo = mid; else hi = mid - 1;
  }
  Cursor c;
  c.s = lo;
  c.n = (off[lo + 1] - off[lo]) / Hkv;
  const int local = (int)(pos - off[lo]);
  c.g = local / c.n;
  c.pi = local - c.g * c.n;
  return c;
}

__device__ __forceinline__ void advance(Cursor &c, const int *off, int num_seqs, int Hkv) {
  if (++c.pi < c.n) return;
  c.pi = 0;
  if (++c.g < Hkv) return;
  c.g = 0;
  do {
    ++c.s;
  } while (c.s < num_seqs && off[c.s + 1] == off[c.s]);
  if (c.s < num_seqs) c.n = (off[c.s + 1] - off[c.s]) / Hkv;
}

// worker owning stream position p when N positions are split over W workers
__device__ __forceinline__ int owner_worker(int64_t p, int64_t N, int W) {
  return (int)(((p + 1) * (int64_t)W - 1) / N);
}

// The step's new K/V rows [T][Hkv][D] copied into their cache slots (the
// append, when it is fused into the attention call): CTA `cta` of `ncta`
// takes a grid-stride share, four 16-byte pieces in flight per thread.
template <int D>
__device__ __forceinline__ void append_new_rows(const AttnParams &p, int cta, int ncta) {
  constexpr int CPR = D * 2 / 16;  // 16-byte pieces per row
  const int64_t total = (int64_t)p.num_tokens * p.Hkv * CPR;
  const int64_t stride = (int64_t)ncta * blockDim.x;
  const int64_t num_slots = p.num_pages * kPage;
  const uint4 *kin = static_cast<const uint4 *>(p.k_new);
  const uint4 *vin = static_cast<const uint4 *>(p.v_new);
  uint4 *kc = static_cast<uint4 *>(const_cast<void *>(p.k_cache));
  uint4 *vc = static_cast<uint4 *>(const_cast<void *>(p.v_cache));
  for (int64_t i0 = (int64_t)cta * blockDim.x + threadIdx.x; i0 < total; i0 += 4 * stride) {
    uint4 kw[4], vw[4];
    int64_t sl[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < total) {
        sl[u] = __ldg(p.slot_mapping + i / CPR / p.Hkv);
        kw[u] = __ldg(kin + i);
        vw[u] = __ldg(vin + i);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u * stride;
      if (i >= total) continue;
      const int64_t row = i / CPR, t = row / p.Hkv;
      const int g = (int)(row - t * p.Hkv), ch = (int)(i - row * CPR);
      if (sl[u] >= num_slots) {
        if (ch == 0) atomicOr(p.status, STATUS_BAD_SLOT);
      } else if (sl[u] >= 0) {
        const int64_t pg = sl[u] / kPage, off = sl[u] - pg * kPage;
        const int64_t dst = ((pg * p.Hkv + g) * kPage + off) * CPR + ch;
        kc[dst] = kw[u];
        vc[dst] = vw[u];
      }
    }
  }
}

// The last contributor of a (sequence, kv head) merges the nc partials in
// slots base .. base+nc-1 with log-sum-exp weights: one pass for every row's
// maximum (lanes stride the contributors), then U contributors per round with
// every row's (max, sum) and each lane's slice of every row's output in
// flight; each lane owns D/32 output dims of every row.  Out of line: a
// segment in a region of short slices has tens of contributors, and with the
// merge inlined, more loads in flight changed how the page loop was allocated.
template <int D, int G>
__device__ __noinline__ void merge_partials(const float *part_o, const float2 *part_ml,
                                            int64_t base, int nc, __nv_bfloat16 *out, int lane) {
  constexpr int DPL = D / 32;
  constexpr int U = 4;
  float mx[G];
#pragma unroll
  for (int r = 0; r < G; ++r) mx[r] = -INFINITY;
  for (int c = lane; c < nc; c += 32) {
#pragma unroll
    for (int r = 0; r < G; ++r) mx[r] = fmaxf(mx[r], __ldcg(&part_ml[(base + c) * G + r].x));
  }
#pragma unroll
  for (int r = 0; r < G; ++r) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], o));
  }
  float acc[G][DPL], lsum[G];
#pragma unroll
  for (int r = 0; r < G; ++r) {
    lsum[r] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[r][e] = 0.f;
  }
  for (int c0 = 0; c0 < nc; c0 += U) {
    float2 ml[U][G];
    float ov[U][G][DPL];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t slot = base + min(c0 + u, nc - 1);
#pragma unroll
      for (int r = 0; r < G; ++r) {
        ml[u][r] = __ldcg(&part_ml[slot * G + r]);
        const float *src = part_o + (slot * G + r) * D + lane * DPL;
        if constexpr (DPL == 4) {
          const float4 v = __ldcg(reinterpret_cast<const float4 *>(src));
          ov[u][r][0] = v.x; ov[u][r][1] = v.y; ov[u][r][2] = v.z; ov[u][r][3] = v.w;
        } else {
          const float2 v = __ldcg(reinterpret_cast<const float2 *>(src));
          ov[u][r][0] = v.x; ov[u][r][1] = v.y;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int r = 0; r < G; ++r) {
        const float wgt = (c0 + u < nc && ml[u][r].x != -INFINITY)
                              ? ptx::ex2(ml[u][r].x - mx[r]) : 0.f;
        lsum[r] = fmaf(ml[u][r].y, wgt, lsum[r]);
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[r][e] = fmaf(ov[u][r][e], wgt, acc[r][e]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < G; ++r) {
    const float inv = 1.f / lsum[r];
#pragma unroll
    for (int e = 0; e < DPL; e += 2) {
      *reinterpret_cast<__nv_bfloat162 *>(out + r * D + lane * DPL + e) =
          __floats2bfloat162_rn(acc[r][e] * inv, acc[r][e + 1] * inv);
    }
  }
}

// With the append fused in, a decode's own token (position ctx - 1, in the
// last page of its segment) may not be in the cache yet when the page is
// copied in: its K and V rows in the stage are overwritten from the step's
// k/v rows, one 16-byte piece per lane.  Out of line: inlined, its registers
// changed how the page loop was allocated and made it ~10 % slower.
template <int D>
__device__ __noinline__ void patch_last_row(const void *k_new, const void *v_new, int Hkv,
                                            unsigned char *stage_k, int page_bytes, int tok,
                                            int g, int ctx, int lane) {
  constexpr int CPR = D * 2 / 16;
  const int r = (ctx - 1) & (kPage - 1);
  if (lane < 2 * CPR) {
    const bool isv = lane >= CPR;
    const int ch = isv ? lane - CPR : lane;
    const uint4 *src = static_cast<const uint4 *>(isv ? v_new : k_new) +
                       ((int64_t)tok * Hkv + g) * CPR + ch;
    uint4 *dst = reinterpret_cast<uint4 *>(stage_k + (isv ? page_bytes : 0) + r * D * 2) + ch;
    *dst = __ldg(src);
  }
  __syncwarp();
}

template <int D, int G, bool FUSED>
__global__ void __launch_bounds__(kWarps * 32, 1)
attn_decode_kernel(const AttnParams p) {
  using C = Cfg<D>;
  using L = Layout<D, G>;
  constexpr int DL = C::DL, CH = C::CH, NST = C::NST, NP = DL / 2;  // NP: fp32 pairs per row
  constexpr int NV = 4 * G;       // partial dots per lane per page: 4 keys x G rows
  constexpr int HALF = G / 2;     // rows a lane holds after the reduce-scatter

  extern __shared__ __align__(1024) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kg = lane >> 3, dp = lane & 7;
  const int b0 = lane & 1, b1 = (lane >> 1) & 1, b2 = (lane >> 2) & 1;
  // after the reduce-scatter a lane holds key myk of the page, rows r0 .. r0+HALF-1
  const int myk = kg + 4 * (b1 + 2 * b2);
  const int r0 = HALF * b0;

  unsigned char *ring = smem + warp * NST * C::STAGE_BYTES;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BARS) + warp * NST;
  int *valid = reinterpret_cast<int *>(smem + L::FLAGS) + warp * NST;
  float *pbuf = reinterpret_cast<float *>(smem + L::PBUF) + warp * kPage * G;
  int *off = reinterpret_cast<int *>(smem + L::OFFS);

  if constexpr (FUSED) {
    // The append: every new row into its cache slot, for later steps (this
    // step's attention takes its own tokens' rows from k_new/v_new).  The
    // CTAs that start after the chunk kernel do it, or every CTA if none do.
    const int e0 = p.decode_early > 0 ? min(p.decode_early, (int)gridDim.x) : (int)gridDim.x;
    const int first = e0 < (int)gridDim.x ? e0 : 0;
    if ((int)blockIdx.x >= first)
      append_new_rows<D>(p, (int)blockIdx.x - first, (int)gridDim.x - first);
  }

  // ---- page-stream offsets of every sequence (exclusive prefix sum) ----
  const int S = p.num_seqs;
  int c_items = 0, c_ctx = 0;  // chunk work items and longest chunk context (split estimate)
  {
    const int nthr = kWarps * 32;
    const int per = (S + nthr - 1) / nthr;
    const int s0 = threadIdx.x * per, s1 = min(S, s0 + per);
    int local = 0;
    for (int s = s0; s < s1; ++s) {
      local += seq_decode_pages(p, s) * p.Hkv;
      if (p.decode_early > 0) {
        const int ql = __ldg(p.query_start_loc + s + 1) - __ldg(p.query_start_loc + s);
        if (ql > 1) {
          c_items += p.Hkv * ((ql * G + 255) / 256);
          c_ctx = max(c_ctx, __ldg(p.seq_lens + s));
        }
      }
    }
    if (p.decode_early > 0) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        c_items += __shfl_xor_sync(0xffffffffu, c_items, o);
        c_ctx = max(c_ctx, __shfl_xor_sync(0xffffffffu, c_ctx, o));
      }
      __shared__ int chunk_red[2 * kWarps];
      if (lane == 0) { chunk_red[warp] = c_items; chunk_red[kWarps + warp] = c_ctx; }
      __syncthreads();
      c_items = 0;
      c_ctx = 0;
      for (int w = 0; w < kWarps; ++w) {
        c_items += chunk_red[w];
        c_ctx = max(c_ctx, chunk_red[kWarps + w]);
      }
    }
    // block exclusive scan of `local`
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    __shared__ int warp_tot[kWarps];
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += warp_tot[w];
    int run = base + incl - local;
    for (int s = s0; s < s1; ++s) {
      off[s] = run;
      run += seq_decode_pages(p, s) * p.Hkv;
    }
    if (threadIdx.x == nthr - 1) off[S] = base + incl;
    __syncthreads();
  }
  const int64_t N = off[S];
  if (N == 0) return;
  // The page stream [0, N) is [0, NA) for the CTAs that start at once and
  // [NA, N) for those that start as the chunk kernel's CTAs finish (NA = N
  // when every CTA starts at once).  Each group splits its range evenly over
  // its workers, at most one worker per page: with W <= n consecutive slice
  // starts floor(w n / W) strictly increase, so every slice is non-empty and a
  // segment's contributors are exactly the workers owner(start)..owner(end),
  // numbered across both groups (late workers follow the early ones).
  const int early = p.decode_early > 0 ? min(p.decode_early, (int)gridDim.x) : (int)gridDim.x;
  const int late = (int)gridDim.x - early;
  int64_t NA = N;
  if (late > 0) {
    // early CTAs stream for T, late ones for T - t_chunk at the same rate:
    // early * r * T + late * r * (T - t_chunk) = N pages
    const int64_t rounds = (c_items + p.chunk_grid - 1) / max(p.chunk_grid, 1);
    // single precision: the split only has to be close, and every thread
    // computes the same value (fp64 is slow on this part)
    const float t_chunk = (float)rounds * ((float)((c_ctx + 127) / 128) *
                                           (float)(kChunkIterNs * (D / 128.0)) +
                                           (float)kChunkItemNs);
    constexpr float r = (float)(kDecodeBytesPerNs / (2.0 * kPage * D * 2));  // pages/ns/CTA
    const float T = ((float)N * (1.f / r) + (float)late * t_chunk) / (float)gridDim.x;
    NA = (T <= t_chunk) ? N : (int64_t)fminf((float)early * r * T, (float)N);
    if (NA > N) NA = N;
  }
  const int64_t wa = (int64_t)early * kWarps, wb = (int64_t)late * kWarps;
  const int WA = (int)(wa < NA ? wa : NA), WB = (int)(wb < N - NA ? wb : N - NA);
  auto owner = [&](int64_t pos) -> int {
    return pos < NA ? owner_worker(pos, NA, WA) : WA + owner_worker(pos - NA, N - NA, WB);
  };
  int w;  // worker index across both groups
  int64_t a, b;
  if ((int)blockIdx.x < early) {
    const int wl = blockIdx.x * kWarps + warp;
    if (wl >= WA) return;
    w = wl;
    a = (int64_t)wl * NA / WA;
    b = (int64_t)(wl + 1) * NA / WA;
  } else {
    const int wl = ((int)blockIdx.x - early) * kWarps + warp;
    if (wl >= WB) return;
    w = WA + wl;
    a = NA + (int64_t)wl * (N - NA) / WB;
    b = NA + (int64_t)(wl + 1) * (N - NA) / WB;
  }

  if (lane == 0) {
    for (int i = 0; i < NST; ++i) ptx::mbar_init(&bars[i], 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();

  const __nv_bfloat16 *kc = static_cast<const __nv_bfloat16 *>(p.k_cache);
  const __nv_bfloat16 *vc = static_cast<const __nv_bfloat16 *>(p.v_cache);

  // ---- producer state (warp-uniform cursor; lane 0 issues the copies) ----
  Cursor pc = locate(off, S, p.Hkv, a);
  int64_t ppos = a;
  int win_s = -1, win_pi = 0, bt_win = -1;
  bool failed = false;
  int64_t fail_pos = 0;

  auto issue = [&](int stage) {
    if (ppos >= b) return;
    if (pc.s != win_s || pc.pi < win_pi || pc.pi >= win_pi + 32) {
      win_s = pc.s;
      win_pi = pc.pi;
      const int idx = pc.pi + lane;
      bt_win = idx < pc.n ? __ldg(p.block_table + (int64_t)pc.s * p.max_pages + idx) : -1;
    }
    const int page = __shfl_sync(0xffffffffu, bt_win, pc.pi - win_pi);
    if (lane == 0) {
      const bool ok = page >= 0 && page < p.num_pages;
      valid[stage] = ok;
      if (ok) {
        const int64_t row = ((int64_t)page * p.Hkv + pc.g) * kPage * D;
        unsigned char *dst = ring + stage * C::STAGE_BYTES;
        ptx::fence_proxy_async_smem();
        ptx::mbar_arrive_expect_tx(&bars[stage], C::STAGE_BYTES);
        ptx::bulk_g2s(dst, kc + row, C::PAGE_BYTES, &bars[stage]);
        ptx::bulk_g2s(dst + C::PAGE_BYTES, vc + row, C::PAGE_BYTES, &bars[stage]);
      } else {
        atomicOr(p.status, STATUS_BAD_PAGE);
        ptx::mbar_arrive(&bars[stage]);
      }
    }
    advance(pc, off, S, p.Hkv);
    ++ppos;
  };

  for (int i = 0; i < NST; ++i) issue(i);

  // ---- consumer ----
  Cursor cc = locate(off, S, p.Hkv, a);
  uint64_t q2[G][NP], o2[G][NP];
  float m[G], lpart[HALF];
  int tok = 0, ctx = 0;
  bool own_start = false;
  int64_t seg_start = 0;

  for (int64_t pos = a; pos < b; ++pos) {
    const int it = (int)(pos - a);
    const int stage = it % NST;
    const uint32_t parity = (uint32_t)((it / NST) & 1);
    if (pos == a || cc.pi == 0) {
      // a new segment (s, g) begins for this worker
      tok = __ldg(p.query_start_loc + cc.s);
      ctx = min(__ldg(p.seq_lens + cc.s), p.max_pages * kPage);
      own_start = (cc.pi == 0);
      seg_start = pos - cc.pi;
      if constexpr (FUSED) {
        // the decode's own K/V row is patched into the segment's last page
        // from k_new/v_new: start bringing it into L2
        constexpr int LPR = D * 2 / 128;  // 128-byte lines per row
        if (lane < 2 * LPR) {
          const char *src = static_cast<const char *>(lane < LPR ? p.k_new : p.v_new) +
                            ((int64_t)tok * p.Hkv + cc.g) * D * 2 + (lane % LPR) * 128;
          ptx::prefetch_l2(src);
        }
      }
      const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(p.q) +
                               ((int64_t)tok * p.Hq + (int64_t)cc.g * G) * D;
#pragma unroll
      for (int r = 0; r < G; ++r) {
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const uint4 w4 = __ldg(reinterpret_cast<const uint4 *>(q + r * D + (dp + 8 * c) * 8));
          const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float x0 = __uint_as_float(ws[e] << 16) * p.scale_log2;
            float x1 = __uint_as_float(ws[e] & 0xffff0000u) * p.scale_log2;
            q2[r][c * 4 + e] = ptx::pack2(x0, x1);
            o2[r][c * 4 + e] = 0ull;
          }
        }
        m[r] = -INFINITY;
      }
#pragma unroll
      for (int j = 0; j < HALF; ++j) lpart[j] = 0.f;
    }

    if (!ptx::mbar_wait(&bars[stage], parity)) {
      if (lane == 0) atomicOr(p.status, STATUS_TIMEOUT);
      failed = true;
      fail_pos = pos;
      break;
    }
    if (valid[stage]) {
      if constexpr (FUSED) {
        if (cc.pi == cc.n - 1)
          patch_last_row<D>(p.k_new, p.v_new, p.Hkv, ring + stage * C::STAGE_BYTES,
                            C::PAGE_BYTES, tok, cc.g, ctx, lane);
      }
      const unsigned char *ks = ring + stage * C::STAGE_BYTES;
      const unsigned char *vs = ks + C::PAGE_BYTES;
      const int key0 = cc.pi * kPage;
      // ---- S = q K^T (partial over this lane's dims) ----
      float sv[NV];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int k = kg + 4 * kk;
        uint64_t kp[NP];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const uint4 w4 = *reinterpret_cast<const uint4 *>(ks + k * D * 2 + (dp + 8 * c) * 16);
          kp[c * 4 + 0] = ptx::bf16x2_to_f2(w4.x);
          kp[c * 4 + 1] = ptx::bf16x2_to_f2(w4.y);
          kp[c * 4 + 2] = ptx::bf16x2_to_f2(w4.z);
          kp[c * 4 + 3] = ptx::bf16x2_to_f2(w4.w);
        }
#pragma unroll
        for (int r = 0; r < G; ++r) {
          uint64_t acc = ptx::fmul2(q2[r][0], kp[0]);
#pragma unroll
          for (int e = 1; e < NP; ++e) acc = ptx::ffma2(q2[r][e], kp[e], acc);
          float x, y;
          ptx::unpack2(acc, x, y);
          sv[kk * G + r] = x + y;
        }
      }
      // ---- reduce-scatter over the 8 lanes of the group (bits 2, 1, 0) ----
#pragma unroll
      for (int step = 0; step < 3; ++step) {
        const int bit = 4 >> step;
        const int n = NV >> step, h = n >> 1;
        const bool up = (lane & bit) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
          const float send = up ? sv[i] : sv[i + h];
          const float keep = up ? sv[i + h] : sv[i];
          sv[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
        }
      }
      const bool kvalid = key0 + myk < ctx;
      float mine[HALF], theirs[HALF];
#pragma unroll
      for (int j = 0; j < HALF; ++j) {
        if (!kvalid) sv[j] = -INFINITY;
        float v = sv[j];
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
        mine[j] = v;
        theirs[j] = __shfl_xor_sync(0xffffffffu, v, 1);
      }
      // rows [HALF*b0, HALF*b0 + HALF) are "mine", the others the partner's
      float pmax[G];
#pragma unroll
      for (int r = 0; r < G; ++r)
        pmax[r] = ((r / HALF) == b0) ? mine[r % HALF] : theirs[r % HALF];
      // online softmax update (per 8-lane group; all lanes of a group agree).
      // The reference m only moves when the max grew by more than 2^8 (or at
      // the first visible key), so p stays below 2^8 and O is rescaled rarely.
      float alpha[G];
      bool any_rescale = false;
#pragma unroll
      for (int r = 0; r < G; ++r) {
        const bool move = pmax[r] > m[r] + kLazyRescale;  // m = -inf: any visible key
        const float mn = move ? pmax[r] : m[r];
        alpha[r] = (move && m[r] != -INFINITY) ? ptx::ex2(m[r] - mn) : 1.f;
        any_rescale |= (alpha[r] != 1.f);
        m[r] = mn;
      }
#pragma unroll
      for (int j = 0; j < HALF; ++j) {
        const float mj = b0 ? m[HALF + j] : m[j];
        const float aj = b0 ? alpha[HALF + j] : alpha[j];
        const float pj = (mj == -INFINITY) ? 0.f : ptx::ex2(sv[j] - mj);
        lpart[j] = lpart[j] * aj + pj;
        pbuf[myk * G + r0 + j] = pj;
      }
      if (__any_sync(0xffffffffu, any_rescale)) {
#pragma unroll
        for (int r = 0; r < G; ++r) {
          const uint64_t a2 = ptx::pack2(alpha[r], alpha[r]);
#pragma unroll
          for (int e = 0; e < NP; ++e) o2[r][e] = ptx::fmul2(o2[r][e], a2);
        }
      }
      __syncwarp();
      // ---- O += P V ----
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int k = kg + 4 * kk;
        if (key0 + k < ctx) {
          float pr[G];
#pragma unroll
          for (int r = 0; r < G; ++r) pr[r] = pbuf[k * G + r];
          uint64_t vp[NP];
#pragma unroll
          for (int c = 0; c < CH; ++c) {
            const uint4 w4 = *reinterpret_cast<const uint4 *>(vs + k * D * 2 + (dp + 8 * c) * 16);
            vp[c * 4 + 0] = ptx::bf16x2_to_f2(w4.x);
            vp[c * 4 + 1] = ptx::bf16x2_to_f2(w4.y);
            vp[c * 4 + 2] = ptx::bf16x2_to_f2(w4.z);
            vp[c * 4 + 3] = ptx::bf16x2_to_f2(w4.w);
          }
#pragma unroll
          for (int r = 0; r < G; ++r) {
            const uint64_t pp = ptx::pack2(pr[r], pr[r]);
#pragma unroll
            for (int e = 0; e < NP; ++e) o2[r][e] = ptx::ffma2(vp[e], pp, o2[r][e]);
          }
        }
      }
    }
    __syncwarp();
    issue(stage);  // refill this stage NST positions ahead

    // ---- end of this worker's part of the segment? ----
    const bool seg_end = (cc.pi == cc.n - 1);
    if (seg_end || pos == b - 1) {
      // group row sums, then all rows on all lanes of the group
      float lmine[HALF], ltheirs[HALF];
#pragma unroll
      for (int j = 0; j < HALF; ++j) {
        float v = lpart[j];
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        lmine[j] = v;
        ltheirs[j] = __shfl_xor_sync(0xffffffffu, v, 1);
      }
      float lg[G];
#pragma unroll
      for (int r = 0; r < G; ++r)
        lg[r] = ((r / HALF) == b0) ? lmine[r % HALF] : ltheirs[r % HALF];
      // combine the 4 groups (lanes xor 8, 16)
      float M[G], Lr[G];
#pragma unroll
      for (int r = 0; r < G; ++r) {
        float mx = m[r];
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float sc = (m[r] == -INFINITY) ? 0.f : ptx::ex2(m[r] - mx);
        float l = lg[r] * sc;
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        M[r] = mx;
        Lr[r] = l;
        const uint64_t s2 = ptx::pack2(sc, sc);
#pragma unroll
        for (int e = 0; e < NP; ++e) {
          uint64_t v = ptx::fmul2(o2[r][e], s2);
          float x, y;
          ptx::unpack2(v, x, y);
          x += __shfl_xor_sync(0xffffffffu, x, 8);
          y += __shfl_xor_sync(0xffffffffu, y, 8);
          x += __shfl_xor_sync(0xffffffffu, x, 16);
          y += __shfl_xor_sync(0xffffffffu, y, 16);
          o2[r][e] = ptx::pack2(x, y);
        }
      }
      const int sg = cc.s * p.Hkv + cc.g;
      const bool own_end = seg_end;
      if (own_start && own_end) {
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(p.out) +
                             ((int64_t)tok * p.Hq + (int64_t)cc.g * G) * D;
#pragma unroll
        for (int r = 0; r < G; ++r) {
          if ((r & 3) != kg) continue;
          const float inv = 1.f / Lr[r];
#pragma unroll
          for (int c = 0; c < CH; ++c) {
            uint32_t wds[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float x, y;
              ptx::unpack2(o2[r][c * 4 + e], x, y);
              __nv_bfloat162 h2 = __floats2bfloat162_rn(x * inv, y * inv);
              wds[e] = *reinterpret_cast<uint32_t *>(&h2);
            }
            *reinterpret_cast<uint4 *>(out + r * D + (dp + 8 * c) * 8) =
                make_uint4(wds[0], wds[1], wds[2], wds[3]);
          }
        }
      } else {
        const int64_t slot = (int64_t)sg + w;
        float *po = p.part_o + slot * G * D;
#pragma unroll
        for (int r = 0; r < G; ++r) {
          if ((r & 3) != kg) continue;
#pragma unroll
          for (int c = 0; c < CH; ++c) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) ptx::unpack2(o2[r][c * 4 + e], f[2 * e], f[2 * e + 1]);
            float4 *dst = reinterpret_cast<float4 *>(po + r * D + (dp + 8 * c) * 8);
            dst[0] = make_float4(f[0], f[1], f[2], f[3]);
            dst[1] = make_float4(f[4], f[5], f[6], f[7]);
          }
          if (dp == 0) p.part_ml[slot * G + r] = make_float2(M[r], Lr[r]);
        }
        __threadfence();
        __syncwarp();
        const int64_t seg_last = seg_start + cc.n - 1;
        const int wf = owner(seg_start);
        const int wl = owner(seg_last);
        unsigned prev = 0;
        if (lane == 0) prev = atomicAdd(p.counters + sg, 1u);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == (unsigned)(wl - wf)) {
          // last contributor: merge every contributor's partial
          __threadfence();
          merge_partials<D, G>(p.part_o, p.part_ml, (int64_t)sg + wf, wl - wf + 1,
                               static_cast<__nv_bfloat16 *>(p.out) +
                                   ((int64_t)tok * p.Hq + (int64_t)cc.g * G) * D,
                               lane);
          if (lane == 0) p.counters[sg] = 0u;
        }
      }
    }
    advance(cc, off, S, p.Hkv);
  }

  if (failed) {
    // drain this warp's copies still in flight (bounded), then leave
    if (lane == 0) {
      for (int64_t q = fail_pos; q < ppos; ++q) {
        const int it = (int)(q - a);
        ptx::mbar_wait(&bars[it % NST], (uint32_t)((it / NST) & 1), 1u << 16);
      }
    }
    __syncwarp();
  }
}

template <int D, int G, bool FUSED>
cudaError_t launch_dgf(const AttnParams &p, int grid, cudaStream_t stream) {
  const size_t smem = Layout<D, G>::bytes(p.num_seqs);
  static bool configured = false;  // per instantiation; attribute is per function
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<D, G, FUSED>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Layout<D, G>::bytes(kDecodeMaxSeqs));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  attn_decode_kernel<D, G, FUSED><<<grid, kWarps * 32, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int D, int G>
cudaError_t launch_dg(const AttnParams &p, int grid, cudaStream_t stream) {
  return p.fused ? launch_dgf<D, G, true>(p, grid, stream)
                 : launch_dgf<D, G, false>(p, grid, stream);
}

}  // namespace

bool decode_fast_path(int dtype, int D, int G) {
  if (dtype != CPA_BF16) return false;
  if (D != 64 && D != 128) return false;
  if (G != 2 && G != 4 && G != 8) return false;
  return G * D <= 512;
}

cudaError_t launch_attention_decode(const AttnParams &p, int grid, cudaStream_t stream) {
  const int G = p.Hq / p.Hkv;
  if (p.D == 128) {
    if (G == 2) return launch_dg<128, 2>(p, grid, stream);
    if (G == 4) return launch_dg<128, 4>(p, grid, stream);
  } else {
    if (G == 2) return launch_dg<64, 2>(p, grid, stream);
    if (G == 4) return launch_dg<64, 4>(p, grid, stream);
    if (G == 8) return launch_dg<64, 8>(p, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace cpa
