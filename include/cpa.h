/*
 * cpa.h -- C ABI of libcpa: one chunked-prefill attention step over a paged
 * KV cache, on one NVIDIA GB300 (sm_103a).
 *
 * The step ("vllm-learning-book 05. Chunked Prefill", sections 3 and 4):
 * a packed hybrid batch of S sequences whose scheduled tokens are concatenated
 * on one token axis with no padding.  Sequence s owns packed tokens
 * query_start_loc[s] .. query_start_loc[s+1]-1 (q_len of them) and holds
 * seq_lens[s] tokens in the cache once this step's K/V are appended.  A
 * prefill chunk has q_len > 1; a decode has q_len == 1.  Query row i of
 * sequence s attends to cache positions 0 .. seq_lens[s]-q_len+i: every
 * earlier chunk's K/V plus a causal mask inside the chunk (same page, Q&A of
 * section 8; "Chunked Prefill 技术深度解析", section 4.1).
 *
 * Conventions shared by every call
 *  - All pointers are device pointers unless a comment says otherwise.  The
 *    caller owns and allocates every buffer; the library never allocates
 *    device memory, never synchronises the stream, and keeps no state
 *    between calls besides the workspace the caller passes in.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously.
 *  - Arguments are validated on the host before anything is launched; an
 *    invalid argument returns a negative cpa_status and launches nothing.
 *  - Layouts (row-major, contiguous):
 *      q, out            [num_tokens][num_q_heads][head_dim]
 *      k, v (new tokens) [num_tokens][num_kv_heads][head_dim]
 *      k_cache, v_cache  [num_pages][num_kv_heads][page_size][head_dim]
 *      block_table       int32 [num_seqs][max_pages_per_seq]
 *      query_start_loc   int32 [num_seqs + 1], query_start_loc[0] == 0
 *      seq_lens          int32 [num_seqs]
 *      slot_mapping      int64 [num_tokens]
 *    Element type of q, k, v and out: `dtype` (fp32, bf16 or fp16).  The
 *    caches hold `dtype` too, or, with desc->kv_dtype = CPA_KV_E4M3 (16-bit
 *    dtypes only), one OCP FP8 E4M3 code per element (see cpa_kv_dtype).
 *  - GQA: query head h reads kv head h / (num_q_heads / num_kv_heads).
 *  - Supported: head_dim 64 or 128, page_size 16, num_q_heads a multiple of
 *    num_kv_heads with a group of 1, 2, 4 or 8 heads.
 */
#ifndef CPA_H
#define CPA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CPA_OK = 0,
  CPA_ERR_ARG = -1,          /* malformed argument (null pointer, bad size)    */
  CPA_ERR_UNSUPPORTED = -2,  /* valid but not supported (e.g. head_dim 96)     */
  CPA_ERR_WORKSPACE = -3,    /* workspace missing, misaligned or too small     */
  CPA_ERR_CUDA = -4,         /* a CUDA runtime call or launch failed           */
  CPA_ERR_DEVICE = -5        /* a kernel found an out-of-range index or gave
                                up a bounded wait (status word, read back with
                                cpa_read_device_status)                       */
} cpa_status;

/* After CPA_ERR_DEVICE.  The word collects, since its last read, bit 1: a
 * block_table entry outside [0, num_pages) (that page was skipped), bit 2: a
 * slot_mapping entry past the cache (that row was not written), bit 4: a
 * bounded wait in the step kernel gave up (after 2^22 polls of its barrier,
 * on the order of a second; the CTA drained its copies and left, so some output rows of that call were
 * not written).  The output of every call since the last read is then
 * unreliable and must be recomputed; the cache rows the calls appended are
 * still valid unless bit 2 is set.  Nothing else needs resetting: the read
 * clears the word, and the next call rebuilds its work queue and zeroes its
 * counters itself.  Bits 1 and 2 mean the metadata is wrong; fix it before
 * re-running.  Bit 4 alone means the GPU did not run the kernel's CTAs to
 * completion in time (for instance a stream starved for longer than the wait
 * limit by other work); the same call can simply be issued again. */

typedef enum { CPA_F32 = 0, CPA_BF16 = 1, CPA_F16 = 2 } cpa_dtype;

/* Storage of the paged caches.
 *  CPA_KV_SAME  the caches hold `dtype` elements, bit for bit what was
 *               appended.
 *  CPA_KV_E4M3  the caches hold one byte per element: the OCP 8-bit floating
 *               point (OFP8) E4M3 code of the value divided by a per-tensor
 *               scale (desc->k_scale for K, desc->v_scale for V); the cached
 *               K is k_scale * E4M3 value, V likewise.  The append computes
 *               x / scale as one correctly rounded binary32 division, then
 *               rounds to the nearest E4M3 value (ties to even), saturating
 *               at +-448 (infinities included); NaN gives a NaN code.  The
 *               attention reads the codes exactly: the tensor cores multiply
 *               their exact binary16 values, q rounded to binary16 (exact for
 *               bf16 or fp16 inputs of magnitude 2^-17 .. 65504; larger
 *               magnitudes overflow), the softmax weights in binary16, with
 *               fp32 accumulation; k_scale is folded into the softmax scale
 *               and v_scale into the output.  Halves the cache bytes a step
 *               reads.  The pages do not cover an 8-bit cache: a library
 *               extension. */
typedef enum { CPA_KV_SAME = 0, CPA_KV_E4M3 = 1 } cpa_kv_dtype;

/* Problem description shared by the calls.  Sizes are host values. */
typedef struct cpa_desc {
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int64_t num_pages;          /* pages in each of k_cache / v_cache           */
  int32_t max_pages_per_seq;  /* row stride of block_table; also bounds
                                 seq_lens[s] <= max_pages_per_seq * page_size */
  int32_t dtype;              /* cpa_dtype                                    */
  int64_t num_tokens;         /* packed tokens this step (query_start_loc[S]) */
  void *workspace;            /* device scratch, >= cpa_workspace_bytes(),
                                 256-byte aligned.  Only its first 4 bytes (the
                                 device status word) must be zero before the
                                 first call; every call resets the rest of the
                                 state it uses (work queue, merge counters),
                                 whatever an earlier call left there          */
  size_t workspace_bytes;
  int32_t kv_dtype;           /* cpa_kv_dtype; 0 = caches of `dtype`          */
  float k_scale, v_scale;     /* CPA_KV_E4M3: positive finite per-tensor
                                 scales; ignored otherwise                    */
} cpa_desc;

/* Human-readable name of a cpa_status value (static string, never NULL). */
const char *cpa_status_string(int status);

/* Bytes of workspace cpa_attention_forward needs for steps of at most
 * `num_seqs` sequences and desc->num_tokens packed tokens.  Pure host
 * arithmetic; returns 0 if the description is invalid.  The workspace holds
 * the step's work queue, the split-KV partial results (o, running max, running
 * sum) of decode segments and of chunk tiles split over several CTAs, their
 * arrival counters (zeroed by every call before use, never carried over from
 * an earlier call), and a device status
 * word.  It is sized for a GPU of up to 256 SMs. */
size_t cpa_workspace_bytes(const cpa_desc *desc, int32_t num_seqs);

/* KV append: for every packed token t with slot = slot_mapping[t] >= 0, copy
 * k[t][g][:] to k_cache[slot / page_size][g][slot % page_size][:] and likewise
 * v, for all kv heads g.  A negative slot skips the token.  The copy is
 * bit-exact (an E4M3 cache stores the codes of k / k_scale and v / v_scale,
 * see cpa_kv_dtype).  ("Chunked Prefill on an M5 Max", section "Wiring it into the
 * loop": a chunk extends the cache instead of rebuilding it; "Chunked Prefill
 * 技术深度解析", section 4.2: 16-token pages.)
 * Slots >= num_pages * page_size are skipped and raise the device status word
 * when a workspace is given in desc.  Tokens must map to distinct slots.
 * Only desc->num_kv_heads, head_dim, page_size, num_pages, dtype, num_tokens,
 * kv_dtype (with k_scale, v_scale) and (optionally) workspace are read. */
int cpa_kv_append(const void *k, const void *v, const int64_t *slot_mapping,
                  void *k_cache, void *v_cache, const cpa_desc *desc,
                  void *stream);

/* Attention forward of the whole hybrid batch in one call: out[t][h][:] =
 * softmax(scale * q[t][h] . K_j) . V_j over the visible cache positions j of
 * t's sequence (see the top of this file).  K/V are read through
 * block_table; the step's own new K/V must already be in the cache
 * (cpa_kv_append first).  Requires 1 <= q_len <= seq_lens[s] for every
 * sequence and seq_lens[s] <= max_pages_per_seq * page_size; entries of
 * block_table outside [0, num_pages) are not read and raise the device status
 * word.  Decodes with long contexts are split over the KV axis and merged in
 * the same launch with log-sum-exp weights ("Chunked Prefill 技术深度解析",
 * section 7.2: softmax normalised over the visible keys and combined
 * incrementally).  fp32 accumulation throughout; out has q's dtype.  With
 * fp32 activations the tensor cores round the chunk rows' MMA inputs to tf32
 * (10 mantissa bits); decode rows are computed in fp32 on CUDA cores. */
int cpa_attention_forward(const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *block_table,
                          const int32_t *query_start_loc, const int32_t *seq_lens,
                          int32_t num_seqs, float scale, void *out, void *stream,
                          const cpa_desc *desc);

/* KV append and attention forward of one step in one call: the same results
 * as cpa_kv_append(k, v, slot_mapping, k_cache, v_cache, desc, stream)
 * followed by cpa_attention_forward(...) on the same stream -- the cache holds
 * the same bytes afterwards and out the same values -- without a separate
 * append launch ("Chunked Prefill on an M5 Max", section "Wiring it into the
 * loop": appending is part of each chunk's fixed cost).
 *  - Arguments: those of the two calls; k, v [num_tokens][Hkv][D] in the
 *    cache dtype and 16-byte aligned, slot_mapping int64 [num_tokens] and
 *    8-byte aligned.  slot_mapping[t] must be the cache slot of token t's
 *    position in its sequence (block_table[s][pos / 16] * 16 + pos % 16);
 *    tokens with a negative slot are not written, and no query may attend to
 *    them.
 *  - Where the step kernel takes the shape (bf16, head_dim 64 or 128, GQA
 *    group 1, 2, 4 or 8), the step's planning kernel copies the new rows into
 *    the cache while the attention kernel sets up, and the attention reads
 *    them from the cache once that copy is complete: a sequence may appear
 *    more than once in the batch (a chunk and a decode of the same sequence
 *    in one step).  Otherwise the call launches the append and then the
 *    attention on `stream`.
 *  - Errors: those of the two calls; slots >= num_pages * page_size raise the
 *    device status word and are not written. */
int cpa_append_attention_forward(const void *q, const void *k, const void *v,
                                 const int64_t *slot_mapping, void *k_cache, void *v_cache,
                                 const int32_t *block_table, const int32_t *query_start_loc,
                                 const int32_t *seq_lens, int32_t num_seqs, float scale,
                                 void *out, void *stream, const cpa_desc *desc);

/* Size of the scratch array built into the library for
 * cpa_attention_forward_noalloc: 64 MiB of device memory on every GPU that
 * loads the library, held until the process exits. */
#define CPA_NOALLOC_SCRATCH_BYTES (64u << 20)

/* CPA_NOALLOC_SCRATCH_BYTES as the library was built with it (for bindings
 * that cannot read the macro). */
size_t cpa_noalloc_scratch_bytes(void);

/* Attention forward for callers that may not allocate device memory.  The
 * pages have no counterpart to this call: it is a library convenience.
 * Callers in this position include plugins inside a host runtime that owns
 * all device memory and passes in only inputs and outputs, and serving loops
 * that forbid cudaMalloc/cudaFree after start-up because those calls can
 * synchronise the device and can fail under memory pressure mid-step.
 *
 * Same computation, arguments and layouts as cpa_attention_forward, except
 * that desc->workspace and desc->workspace_bytes are ignored: the scratch
 * lives in a fixed array compiled into the library.  The call allocates
 * nothing (no cudaMalloc, no cudaFree, no allocating library routine).
 *  - Limit: the workspace this step would need, cpa_workspace_bytes(desc,
 *    num_seqs), must not exceed CPA_NOALLOC_SCRATCH_BYTES; larger steps are
 *    rejected with CPA_ERR_WORKSPACE before anything is launched.
 *  - Set-up: every call looks up the array's device address in the current
 *    context with cudaGetSymbolAddress (host-side; nothing is allocated).
 *    The first call in a context may load the library's device code, so make
 *    it before any stream capture.  CPA_ERR_CUDA if the lookup fails.
 *  - Sharing: every call on a device uses the same array, which keeps what the
 *    last call left in it.  Once a call has passed its argument checks it
 *    clears the array's status word on `stream`, right before its first
 *    launch (the call resets its work queue and merge counters itself); a
 *    rejected or empty call touches nothing.
 *    Calls whose work overlaps on the GPU (different streams, or different
 *    host threads) race on the array: serialise them.
 *  - Errors: those of cpa_attention_forward; out-of-range indices met by the
 *    kernels are reported by cpa_noalloc_read_device_status. */
int cpa_attention_forward_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *block_table,
                                  const int32_t *query_start_loc, const int32_t *seq_lens,
                                  int32_t num_seqs, float scale, void *out, void *stream,
                                  const cpa_desc *desc);

/* Synchronously read (and clear) the device status word of the no-alloc
 * scratch array on the current device: CPA_OK, or CPA_ERR_DEVICE if the last
 * cpa_attention_forward_noalloc call on this device met an out-of-range page
 * index or gave up a bounded wait (its output is then incomplete).  Waits for
 * `stream`; allocates nothing.  Test/debug helper, not meant for the hot
 * path.  Returns CPA_ERR_ARG for a null status_out, CPA_ERR_CUDA if a CUDA
 * call fails. */
int cpa_noalloc_read_device_status(void *stream, int32_t *status_out);

/* Synchronously read (and clear) the device status word held in the
 * workspace: CPA_OK, or CPA_ERR_DEVICE if a kernel since the last read met an
 * out-of-range page or slot index.  Waits for `stream`.  Test/debug helper,
 * not meant for the hot path. */
int cpa_read_device_status(const cpa_desc *desc, void *stream, int32_t *status_out);

#ifdef __cplusplus
}
#endif

#endif /* CPA_H */
