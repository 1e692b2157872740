"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bars (bf16 in, fp32 accumulate): attention within max-abs 2e-2 and mean-abs
2e-3 of the oracle; KV append and page addressing bit-exact.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from chunked_prefill_paged_cpa_gb300 import ops, workloads
from chunked_prefill_paged_cpa_gb300.batch import pages_for
from support import oracle_append, make_step, oracle_state_for, to_np64

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3


def assert_close(got, want, what=""):
    if isinstance(got, torch.Tensor):
        got = got.detach().to("cpu", torch.float64).numpy()
    if isinstance(want, torch.Tensor):
        want = want.detach().to("cpu", torch.float64).numpy()
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - want)
    assert err.max() <= MAX_ABS, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean abs err {err.mean():.3e}"


def bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def gpu_step(k_cache, v_cache, inp, scale, Hq, workspace=None):
    m = inp["meta"]
    ops.kv_append(inp["k"], inp["v"], m.slot_mapping, k_cache, v_cache)
    if workspace is None:
        workspace = ops.workspace_for(k_cache, Hq, m.block_table.shape[1], m.num_seqs, m.num_tokens)
    out = ops.attention_forward(inp["q"], k_cache, v_cache, m.block_table,
                                m.query_start_loc, m.seq_lens, scale, workspace)
    return out, workspace


def test_tiny_all_steps_match_oracle_and_cache_is_bitexact(cuda_device):
    sc = workloads.scenario("tiny")
    ws = workloads.WorkloadState(sc, device=cuda_device)
    oc = oracle_state_for(ws)
    sh = sc.shape
    # the prefix fill must already agree bit for bit
    assert torch.equal(bits(ws.k_cache.cpu()), bits(oc.k))
    for k in range(len(sc.plans)):
        inp = ws.step(k)
        m = inp["meta"]
        out, wsp = gpu_step(ws.k_cache, ws.v_cache, inp, sh.scale, sh.num_q_heads)
        oc.append(m.block_table.cpu(), m.q_lens, m.seq_lens_list, inp["k"].cpu(),
                  inp["v"].cpu())
        assert torch.equal(bits(ws.k_cache.cpu()), bits(oc.k)), f"step {k}: K cache"
        assert torch.equal(bits(ws.v_cache.cpu()), bits(oc.v)), f"step {k}: V cache"
        want = oracle.attention(inp["q"], oc.k, oc.v, m.block_table, m.query_start_loc,
                                m.seq_lens, sh.scale)
        assert_close(out.cpu(), want, f"tiny step {k + 1}")
        assert ops.device_status(ws.k_cache, sh.num_q_heads, m.block_table.shape[1], wsp) == 0


def test_tiny_chunked_equals_oneshot_on_gpu(cuda_device):
    """A's three 32-token chunks (steps 1-3) equal A's one-shot 96-token
    prefill, and A's step-4 decode equals row 96 of a one-shot 97-token
    prefill."""
    sc = workloads.scenario("tiny")
    ws = workloads.WorkloadState(sc, device=cuda_device)
    sh = sc.shape
    rows = []
    for k in range(4):
        inp = ws.step(k)
        out, _ = gpu_step(ws.k_cache, ws.v_cache, inp, sh.scale, sh.num_q_heads)
        qsl = inp["meta"].query_start_loc.cpu().tolist()
        rids = [s.rid for s in inp["plan"].seqs]
        a = rids.index("A")
        rows.append(out[qsl[a]:qsl[a + 1]].cpu())
    chunked = torch.cat(rows)                                   # positions 0..96
    ws2 = workloads.WorkloadState(sc, device=cuda_device)
    pl = ws2.paged.ensure("A", 97)
    from chunked_prefill_paged_cpa_gb300.batch import build_metadata, write_positions
    pos = torch.arange(97)
    kk, vv = ws2.kv_rows("A", pos)
    write_positions(ws2.k_cache, ws2.v_cache, pl, pos, kk, vv)
    meta = build_metadata([97], [97], [pl], 16, ws2.num_pages).to(cuda_device)
    wsp = ops.workspace_for(ws2.k_cache, sh.num_q_heads, meta.block_table.shape[1], 1, meta.num_tokens)
    one = ops.attention_forward(ws2.q_rows("A", pos).to(cuda_device).contiguous(),
                                ws2.k_cache, ws2.v_cache, meta.block_table,
                                meta.query_start_loc, meta.seq_lens, sh.scale, wsp)
    assert_close(chunked, one.cpu().double(), "chunked vs one-shot (GPU both)")


SMALL_CASES = [
    # (q_lens, seq_lens, Hq, Hkv, D, dtype)
    ([1, 1, 1], [1, 17, 600], 8, 8, 128, torch.bfloat16),
    ([33, 1, 129, 1], [50, 1100, 129, 3], 32, 8, 128, torch.bfloat16),
    ([200], [1300], 16, 2, 128, torch.bfloat16),
    ([5, 1, 64], [5, 2049, 100], 4, 2, 64, torch.float32),
    ([1, 70, 1], [513, 70, 1025], 16, 2, 64, torch.bfloat16),
    ([300, 1], [310, 4000], 8, 1, 128, torch.float32),
]


@pytest.mark.parametrize("case", range(len(SMALL_CASES)))
def test_small_hybrid_batches(cuda_device, case):
    q_lens, seq_lens, Hq, Hkv, D, dtype = SMALL_CASES[case]
    st = make_step(q_lens, seq_lens, Hq, Hkv, D, dtype, seed=100 + case)
    m, oc = st["meta"], st["oracle_cache"]
    dev = cuda_device
    k_cache, v_cache = oc.k.to(dev), oc.v.to(dev)   # prefix state (input), pre-append
    inp = {"meta": m.to(dev), "q": st["q"].to(dev), "k": st["k_new"].to(dev),
           "v": st["v_new"].to(dev)}
    scale = 1 / math.sqrt(D)
    out, _ = gpu_step(k_cache, v_cache, inp, scale, Hq)
    slots = oracle.slot_mapping(m.block_table, m.query_start_loc, m.seq_lens, 16)
    assert torch.equal(slots, m.slot_mapping)
    oracle.kv_append(oc.k, oc.v, st["k_new"], st["v_new"], slots)
    assert torch.equal(bits(k_cache.cpu()), bits(oc.k))
    assert torch.equal(bits(v_cache.cpu()), bits(oc.v))
    want = oracle.attention(st["q"], oc.k, oc.v, m.block_table, m.query_start_loc,
                            m.seq_lens, scale)
    assert_close(out.cpu(), want, f"case {case}")


def _planted_logit_jumps(q, k_seqs, v_seqs):
    """Sequence 0 (a chunk): every query row is one direction u per kv-head
    group; the first key tile is near-orthogonal (logits ~0), keys 128..191
    are 1.0 u (a jump of ~16 in log2 units: the running max moves) and keys
    384..447 are 5.0 u (a jump of ~80: past the lazy bound, the tile is
    recomputed against its own max)."""
    q, k0 = q.clone(), k_seqs[0].clone()
    T0 = k0.shape[0]
    q_len0 = 100
    Hq, D = q.shape[1], q.shape[2]
    Hkv = k0.shape[1]
    G = Hq // Hkv
    gen = torch.Generator().manual_seed(4242)
    u = torch.randn(Hkv, D, generator=gen)
    q[:q_len0] = u.repeat_interleave(G, dim=0).to(q.dtype)[None]
    k0 = (k0.float() * 0.05).to(k0.dtype)
    k0[128:192] = u.to(k0.dtype)[None]
    k0[384:448] = (5.0 * u).to(k0.dtype)[None]
    assert T0 > 448
    return q, [k0] + list(k_seqs[1:]), v_seqs


def test_large_logit_jumps_rescale_and_redo(cuda_device):
    q_lens, seq_lens = [100, 1], [800, 900]
    Hq, Hkv, D = 32, 8, 128
    st = make_step(q_lens, seq_lens, Hq, Hkv, D, torch.bfloat16, seed=77,
                   transform=_planted_logit_jumps)
    m, oc = st["meta"], st["oracle_cache"]
    dev = cuda_device
    k_cache, v_cache = oc.k.to(dev), oc.v.to(dev)
    inp = {"meta": m.to(dev), "q": st["q"].to(dev), "k": st["k_new"].to(dev),
           "v": st["v_new"].to(dev)}
    scale = 1 / math.sqrt(D)
    out, _ = gpu_step(k_cache, v_cache, inp, scale, Hq)
    oracle_append(st)
    want = oracle.attention(st["q"], oc.k, oc.v, m.block_table, m.query_start_loc,
                            m.seq_lens, scale)
    # the planted keys dominate: the output is close to the mean of their V rows
    assert np.isfinite(out.float().cpu().numpy()).all()
    assert_close(out.cpu(), want, "planted logit jumps")


def _jumps_inside_tiles(q, k_seqs, v_seqs):
    """Sequence 0 (a chunk of 60 tokens after 340 cached): every query row is
    one direction u per kv-head group, the other keys near-orthogonal; keys
    40..47 are 1.0 u (a jump of ~16 log2 units in the second 32-key chunk of
    the first 128-key tile), keys 200..203 are 3.0 u (~48, third chunk of the
    second tile) and key 360 is 5.0 u (~80, fourth chunk of the third tile,
    one of the chunk's own new rows): each moves the running maximum after
    chunks of its tile were written."""
    q, k0 = q.clone(), k_seqs[0].clone()
    Hq, D = q.shape[1], q.shape[2]
    Hkv = k0.shape[1]
    G = Hq // Hkv
    gen = torch.Generator().manual_seed(4343)
    u = torch.randn(Hkv, D, generator=gen)
    q[:60] = u.repeat_interleave(G, dim=0).to(q.dtype)[None]
    k0 = (k0.float() * 0.05).to(k0.dtype)
    k0[40:48] = u.to(k0.dtype)[None]
    k0[200:204] = (3.0 * u).to(k0.dtype)[None]
    k0[360] = (5.0 * u).to(k0.dtype)
    return q, [k0] + list(k_seqs[1:]), v_seqs


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_logit_jumps_inside_a_tile_rescale_written_chunks(cuda_device, dtype):
    q_lens, seq_lens = [60, 1], [400, 500]
    Hq, Hkv, D = 8, 2, 128
    st = make_step(q_lens, seq_lens, Hq, Hkv, D, dtype, seed=78,
                   transform=_jumps_inside_tiles)
    m, oc = st["meta"], st["oracle_cache"]
    dev = cuda_device
    k_cache, v_cache = oc.k.to(dev), oc.v.to(dev)
    inp = {"meta": m.to(dev), "q": st["q"].to(dev), "k": st["k_new"].to(dev),
           "v": st["v_new"].to(dev)}
    scale = 1 / math.sqrt(D)
    out, _ = gpu_step(k_cache, v_cache, inp, scale, Hq)
    oracle_append(st)
    want = oracle.attention(st["q"], oc.k, oc.v, m.block_table, m.query_start_loc,
                            m.seq_lens, scale)
    assert np.isfinite(out.float().cpu().numpy()).all()
    assert_close(out.cpu(), want, f"jumps inside tiles ({dtype})")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_every_chunk_kernel_shape(cuda_device, D, G):
    """Every (head_dim, GQA group) instantiation of the chunk-tile kernel, in a
    hybrid batch: a chunk with a cached prefix, one without, and decodes."""
    Hkv = 2
    Hq = G * Hkv
    q_lens, seq_lens = [1, 150, 1, 37], [300, 350, 2000, 37]
    st = make_step(q_lens, seq_lens, Hq, Hkv, D, torch.bfloat16, seed=900 + 10 * G + D)
    m, oc = st["meta"], st["oracle_cache"]
    dev = cuda_device
    k_cache, v_cache = oc.k.to(dev), oc.v.to(dev)
    inp = {"meta": m.to(dev), "q": st["q"].to(dev), "k": st["k_new"].to(dev),
           "v": st["v_new"].to(dev)}
    scale = 1 / math.sqrt(D)
    out, wsp = gpu_step(k_cache, v_cache, inp, scale, Hq)
    oracle_append(st)
    assert torch.equal(bits(k_cache.cpu()), bits(oc.k))
    want = oracle.attention(st["q"], oc.k, oc.v, m.block_table, m.query_start_loc,
                            m.seq_lens, scale)
    assert_close(out.cpu(), want, f"D {D} G {G}")
    assert ops.device_status(k_cache, Hq, m.block_table.shape[1], wsp) == 0


DECODE_CASES = [
    # (num decodes, ctx range, Hq, Hkv, D) -- decode kernel shapes and fallbacks
    (3, (1, 40), 8, 4, 128),       # fewer pages than workers, ragged pages
    (40, (1, 700), 32, 8, 128),
    (17, (100, 3000), 16, 8, 128),  # G = 2
    (9, (1, 2000), 32, 4, 64),      # G = 8, D = 64
    (25, (30, 1500), 16, 4, 64),    # G = 4, D = 64
    (11, (500, 900), 8, 4, 64),     # G = 2, D = 64
    (7, (1, 1000), 64, 8, 128),     # G = 8, D = 128: row kernel
    (5, (1, 600), 8, 8, 128),       # G = 1: row kernel
]


@pytest.mark.parametrize("case", range(len(DECODE_CASES)))
def test_decode_batches(cuda_device, case):
    n, (lo, hi), Hq, Hkv, D = DECODE_CASES[case]
    g = torch.Generator().manual_seed(500 + case)
    seq_lens = torch.randint(lo, hi + 1, (n,), generator=g).tolist()
    # one chunk too, so both roles run in the same call
    q_lens = [1] * n + [37]
    seq_lens = seq_lens + [37 + 50]
    st = make_step(q_lens, seq_lens, Hq, Hkv, D, torch.bfloat16, seed=600 + case)
    m, oc = st["meta"], st["oracle_cache"]
    dev = cuda_device
    k_cache, v_cache = oc.k.to(dev), oc.v.to(dev)
    inp = {"meta": m.to(dev), "q": st["q"].to(dev), "k": st["k_new"].to(dev),
           "v": st["v_new"].to(dev)}
    scale = 1 / math.sqrt(D)
    out, wsp = gpu_step(k_cache, v_cache, inp, scale, Hq)
    oracle_append(st)
    want = oracle.attention(st["q"], oc.k, oc.v, m.block_table, m.query_start_loc,
                            m.seq_lens, scale)
    assert_close(out.cpu(), want, f"decode case {case}")
    assert ops.device_status(k_cache, Hq, m.block_table.shape[1], wsp) == 0
    # a second call on the same workspace (counters were reset) gives the same bits
    out2 = ops.attention_forward(inp["q"], k_cache, v_cache, inp["meta"].block_table,
                                 inp["meta"].query_start_loc, inp["meta"].seq_lens, scale, wsp)
    assert torch.equal(bits(out), bits(out2))


MULTI_CHUNK_CASES = [
    # (decode contexts, [(chunk q_len, cached prefix)]) -- Llama-3-8B shape, bf16
    ([600, 33, 1500, 17] * 10, [(100, 37), (100, 500)]),      # concurrent kernels
    ([2000, 90, 4100, 700, 1], [(1000, 0), (1000, 333), (1000, 2000)]),  # items > CTAs
    ([], [(64, 0), (65, 15), (129, 16), (2, 5000)]),          # chunks only, tiny tiles
    ([5000] * 3, [(257, 4096)]),                             # page-aligned prefix, ragged tile
]


@pytest.mark.parametrize("case", range(len(MULTI_CHUNK_CASES)))
def test_multiple_chunks_per_step(cuda_device, case):
    """Several prefill chunks (with cached prefixes that need not be
    page-aligned) beside decodes in one step."""
    dec, chunks = MULTI_CHUNK_CASES[case]
    q_lens = [1] * len(dec) + [c for c, _ in chunks]
    seq_lens = list(dec) + [c + pre for c, pre in chunks]
    st = make_step(q_lens, seq_lens, 32, 8, 128, torch.bfloat16, seed=900 + case)
    m, oc = st["meta"], st["oracle_cache"]
    dev = cuda_device
    k_cache, v_cache = oc.k.to(dev), oc.v.to(dev)
    inp = {"meta": m.to(dev), "q": st["q"].to(dev), "k": st["k_new"].to(dev),
           "v": st["v_new"].to(dev)}
    scale = 1 / math.sqrt(128)
    out, wsp = gpu_step(k_cache, v_cache, inp, scale, 32)
    oracle_append(st)
    want = oracle.attention(st["q"], oc.k, oc.v, m.block_table, m.query_start_loc,
                            m.seq_lens, scale)
    assert_close(out.cpu(), want, f"multi-chunk case {case}")
    assert ops.device_status(k_cache, 32, m.block_table.shape[1], wsp) == 0


def test_ones_values_give_ones_and_onehot_values_give_probabilities(cuda_device):
    """V == 1 makes every output 1 (softmax rows sum to 1, including across
    merged splits); V_j = e_j (ctx <= D) makes the output row the probability
    row, compared with the oracle's probabilities."""
    dev = cuda_device
    q_lens, seq_lens, Hq, Hkv, D = [1, 20, 1], [1500, 60, 64], 8, 2, 64
    st = make_step(q_lens, seq_lens, Hq, Hkv, D, torch.bfloat16, seed=7)
    m, oc = st["meta"], st["oracle_cache"]
    oracle_append(st)
    ones = torch.ones_like(oc.v).to(dev)
    k_cache = oc.k.to(dev)
    wsp = ops.workspace_for(k_cache, Hq, m.block_table.shape[1], m.num_seqs, m.num_tokens)
    md = m.to(dev)
    out = ops.attention_forward(st["q"].to(dev), k_cache, ones, md.block_table,
                                md.query_start_loc, md.seq_lens, 0.125, wsp)
    assert (out.float() - 1).abs().max().item() <= 2 ** -7
    # one-hot values over the 64-token sequence (third sequence: a decode)
    vh = torch.zeros_like(oc.v)
    pl = m.block_table[2].tolist()
    for j in range(64):
        vh[pl[j // 16], :, j % 16, j] = 1.0
    out = ops.attention_forward(st["q"].to(dev), k_cache, vh.to(dev), md.block_table,
                                md.query_start_loc, md.seq_lens, 0.125, wsp)
    t = int(m.query_start_loc[2])
    for h in range(Hq):
        p, _ = oracle.probs(st["q"], oc.k, vh, m.block_table, m.query_start_loc,
                            m.seq_lens, 0.125, t, h)
        got = out[t, h, :64].float().cpu().numpy()
        assert np.abs(got - p).max() <= 4e-3, h


def test_workspace_reuse_gives_identical_results(cuda_device):
    sc = workloads.scenario("page1_default")
    ws = workloads.WorkloadState(sc, device=cuda_device)
    inp = ws.step(0)
    out1, wsp = gpu_step(ws.k_cache, ws.v_cache, inp, sc.shape.scale, 32)
    m = inp["meta"]
    out2 = ops.attention_forward(inp["q"], ws.k_cache, ws.v_cache, m.block_table,
                                 m.query_start_loc, m.seq_lens, sc.shape.scale, wsp)
    assert torch.equal(bits(out1), bits(out2))


def test_out_of_range_page_sets_status_without_fault(cuda_device):
    dev = cuda_device
    st = make_step([1, 4], [40, 20], 4, 2, 64, torch.float32, seed=3)
    m, oc = st["meta"], st["oracle_cache"]
    k_cache, v_cache = oc.k.to(dev), oc.v.to(dev)
    md = m.to(dev)
    bt = md.block_table.clone()
    bt[0, 1] = 10 ** 6                     # not a page of the pool
    wsp = ops.workspace_for(k_cache, 4, bt.shape[1], 2, md.num_tokens)
    ops.attention_forward(st["q"].to(dev), k_cache, v_cache, bt, md.query_start_loc,
                          md.seq_lens, 0.125, wsp)
    assert ops.device_status(k_cache, 4, bt.shape[1], wsp) == ops.CPA_ERR_DEVICE
    assert ops.device_status(k_cache, 4, bt.shape[1], wsp) == ops.CPA_OK   # cleared
    slots = md.slot_mapping.clone()
    slots[0] = k_cache.shape[0] * 16 + 5   # past the pool
    ops.kv_append(st["k_new"].to(dev), st["v_new"].to(dev), slots, k_cache, v_cache, wsp)
    assert ops.device_status(k_cache, 4, bt.shape[1], wsp) == ops.CPA_ERR_DEVICE


# ---- full-size workloads: every row, per-sequence oracle -------------------

def oracle_rows_for_seq(ws, rid, seq_len, q_len, rows=None):
    """fp64 oracle output of rows ``rows`` (indices within the sequence's
    q_len new tokens; all of them when None) computed from the generator's
    per-position tensors in a fresh identity-paged host cache built by the
    oracle itself (its own slots, its own append)."""
    sh = ws.sc.shape
    n = pages_for(seq_len, sh.page_size)
    kc = torch.full((n, sh.num_kv_heads, sh.page_size, sh.head_dim), float("nan"),
                    dtype=sh.dtype)
    vc = kc.clone()
    bt = torch.arange(n, dtype=torch.int32).view(1, n)
    allq = torch.tensor([0, seq_len], dtype=torch.int32)
    sl = torch.tensor([seq_len], dtype=torch.int32)
    pos = torch.arange(seq_len)
    kk, vv = ws.kv_rows(rid, pos)
    oracle.kv_append(kc, vc, kk.cpu(), vv.cpu(), oracle.slot_mapping(bt, allq, sl, sh.page_size))
    q = ws.q_rows(rid, torch.arange(seq_len - q_len, seq_len)).cpu()
    qsl = torch.tensor([0, q_len], dtype=torch.int32)
    return oracle.attention(q, kc, vc, bt, qsl, sl, sh.scale, rows=rows)


def oracle_step(ws, inp):
    """fp64 oracle output of every query row of one step, [T, Hq, D]."""
    m = inp["meta"]
    sh = ws.sc.shape
    qsl = m.query_start_loc.cpu().tolist()
    want = np.empty((m.num_tokens, sh.num_q_heads, sh.head_dim), dtype=np.float64)
    for i, s in enumerate(inp["plan"].seqs):
        want[qsl[i]:qsl[i + 1]] = oracle_rows_for_seq(ws, s.rid, s.seq_len, s.q_len)
    return want


def check_step_against_oracle(name, ws, inp, out):
    """Every row and head of a step's GPU output against the oracle: each
    sequence on its own (max-abs and mean-abs), then the whole step."""
    want = oracle_step(ws, inp)
    got = out.float().cpu().numpy()
    qsl = inp["meta"].query_start_loc.cpu().tolist()
    for i, s in enumerate(inp["plan"].seqs):
        assert_close(got[qsl[i]:qsl[i + 1]], want[qsl[i]:qsl[i + 1]],
                     f"{name} seq {s.rid} ({s.kind}, q_len {s.q_len}, ctx {s.seq_len})")
    assert_close(got, want, name)
    return want


def check_full_config(name, cuda_device, fused=False):
    sc = workloads.scenario(name)
    ws = workloads.WorkloadState(sc, device=cuda_device)
    inp = ws.step(0)
    m = inp["meta"]
    if fused:
        wsp = ops.workspace_for(ws.k_cache, sc.shape.num_q_heads, m.block_table.shape[1],
                                m.num_seqs, m.num_tokens)
        out = ops.append_attention_forward(inp["q"], inp["k"], inp["v"], m.slot_mapping,
                                           ws.k_cache, ws.v_cache, m.block_table,
                                           m.query_start_loc, m.seq_lens, sc.shape.scale, wsp)
    else:
        out, wsp = gpu_step(ws.k_cache, ws.v_cache, inp, sc.shape.scale, sc.shape.num_q_heads)
    torch.cuda.synchronize()
    assert ops.device_status(ws.k_cache, sc.shape.num_q_heads, m.block_table.shape[1],
                             wsp) == 0
    # paging bit-exact: the package's slots equal the oracle's, and the cache
    # holds the new rows at exactly those slots
    mc = m.to("cpu")
    slots = oracle.slot_mapping(mc.block_table, mc.query_start_loc, mc.seq_lens, 16)
    assert torch.equal(slots, mc.slot_mapping)
    sd = slots.to(cuda_device)
    got_k = ws.k_cache[sd // 16, :, sd % 16, :]
    got_v = ws.v_cache[sd // 16, :, sd % 16, :]
    assert torch.equal(bits(got_k), bits(inp["k"])) and torch.equal(bits(got_v), bits(inp["v"]))
    # pages never handed out are still poisoned
    used = torch.zeros(ws.num_pages, dtype=torch.bool)
    for pl in ws.paged.pages.values():
        used[pl] = True
    unused = (~used).nonzero().flatten().to(cuda_device)
    if unused.numel():
        assert torch.isnan(ws.k_cache[unused].float()).all()
    # every row of every sequence against the oracle
    check_step_against_oracle(name, ws, inp, out)


@pytest.mark.parametrize("name", ["page1_default", "large_budget", "long_context",
                                  "decode_only", "oneshot_8192"])
def test_full_size_config(name, cuda_device):
    check_full_config(name, cuda_device)


def test_chunked_prefill_equals_oneshot_at_full_size(cuda_device):
    """The 8192-token prompt of the large-budget configuration prefilled as
    four 2048-token chunks beside 4 decodes (four fused steps, each chunk
    attending to the earlier chunks through the paged cache) equals the
    one-shot 8192-token prefill of the same prompt: on the GPU, both within
    tolerance of each other, and each, every row and head, within tolerance of
    the fp64 oracle ("vllm-learning-book 05. Chunked Prefill", section 3;
    "Chunked Prefill 技术深度解析", section 7.2).  The decodes of every step
    are checked against the oracle too."""
    from chunked_prefill_paged_cpa_gb300.batch import build_metadata
    sc = workloads.scenario("large_budget_chunked")
    ws = workloads.WorkloadState(sc, device=cuda_device)
    sh = sc.shape
    chunk_rows = []
    for k in range(len(sc.plans)):
        inp = ws.step(k)
        m = inp["meta"]
        assert sorted(m.q_lens) == [1, 1, 1, 1, 2048]
        wsp = ops.workspace_for(ws.k_cache, sh.num_q_heads, m.block_table.shape[1],
                                m.num_seqs, m.num_tokens)
        out = ops.append_attention_forward(inp["q"], inp["k"], inp["v"], m.slot_mapping,
                                           ws.k_cache, ws.v_cache, m.block_table,
                                           m.query_start_loc, m.seq_lens, sh.scale, wsp)
        torch.cuda.synchronize()
        qsl = m.query_start_loc.cpu().tolist()
        for i, s in enumerate(inp["plan"].seqs):
            if s.kind == "decode":
                want = oracle_rows_for_seq(ws, s.rid, s.seq_len, 1)
                assert_close(out[qsl[i]:qsl[i + 1]].float().cpu(), want,
                             f"step {k + 1} decode {s.rid}")
            else:
                assert s.rid == "P" and s.seq_len == 2048 * (k + 1)
                chunk_rows.append(out[qsl[i]:qsl[i + 1]].clone())
    chunked = torch.cat(chunk_rows)                       # prompt positions 0..8191
    # the same prompt in one shot: its rows are already in the cache (the
    # append writes the same bytes again), one 8192-token prefill entry
    pos = torch.arange(8192)
    meta = build_metadata([8192], [8192], [ws.paged.pages["P"]], 16,
                          ws.num_pages).to(cuda_device)
    kk, vv = ws.kv_rows("P", pos)
    q = ws.q_rows("P", pos).to(cuda_device).contiguous()
    wsp = ops.workspace_for(ws.k_cache, sh.num_q_heads, meta.block_table.shape[1], 1, meta.num_tokens)
    one = ops.append_attention_forward(q, kk.to(cuda_device).contiguous(),
                                       vv.to(cuda_device).contiguous(), meta.slot_mapping,
                                       ws.k_cache, ws.v_cache, meta.block_table,
                                       meta.query_start_loc, meta.seq_lens, sh.scale, wsp)
    torch.cuda.synchronize()
    assert_close(chunked.float().cpu(), one.float().cpu().double(),
                 "chunked vs one-shot (GPU both)")
    want = oracle_rows_for_seq(ws, "P", 8192, 8192)
    assert_close(chunked.float().cpu(), want, "chunked prefill vs oracle")
    assert_close(one.float().cpu(), want, "one-shot prefill vs oracle")


def test_tiny_alternative_reading_sequence_twice_in_one_step(cuda_device):
    """The tiny configuration's other reading: in step 3, A appears twice --
    its last 32-token chunk (seq_len 96) and, in the same step, the decode of
    its first generated token (position 96, seq_len 97), over the same block
    table ("vllm-learning-book 05. Chunked Prefill", section 2: the first
    output token is produced in the pass that finishes the prompt).  Run
    through the separate calls, which allow a sequence more than once (the
    fused call does not: its header requires each sequence at most once).
    Checked against the oracle on every row, and A's decode against the last
    row of a one-shot 97-token prefill."""
    from chunked_prefill_paged_cpa_gb300.batch import build_metadata
    sc = workloads.scenario("tiny")
    ws = workloads.WorkloadState(sc, device=cuda_device)
    oc = oracle_state_for(ws)
    sh = sc.shape
    for k in range(2):                                    # steps 1 and 2 as planned
        inp = ws.step(k)
        m = inp["meta"]
        gpu_step(ws.k_cache, ws.v_cache, inp, sh.scale, sh.num_q_heads)
        oc.append(m.block_table.cpu(), m.q_lens, m.seq_lens_list, inp["k"].cpu(),
                  inp["v"].cpu())
    # step 3, alternative reading: B decodes position 42; A's chunk 64..95 and
    # A's decode at 96
    pa = ws.paged.ensure("A", 97)
    pb = ws.paged.ensure("B", 43)
    q_lens, seq_lens = [1, 32, 1], [43, 96, 97]
    meta = build_metadata(q_lens, seq_lens, [pb, pa, pa], 16, ws.num_pages)
    qb = ws.q_rows("B", torch.tensor([42]))
    qa = ws.q_rows("A", torch.arange(64, 97))
    kb, vb = ws.kv_rows("B", torch.tensor([42]))
    ka, va = ws.kv_rows("A", torch.arange(64, 97))
    q = torch.cat([qb, qa]).to(cuda_device).contiguous()
    k_new = torch.cat([kb, ka]).to(cuda_device).contiguous()
    v_new = torch.cat([vb, va]).to(cuda_device).contiguous()
    inp = {"meta": meta.to(cuda_device), "q": q, "k": k_new, "v": v_new}
    out, wsp = gpu_step(ws.k_cache, ws.v_cache, inp, sh.scale, sh.num_q_heads)
    torch.cuda.synchronize()
    slots = oc.append(meta.block_table, q_lens, seq_lens, k_new.cpu(), v_new.cpu())
    assert torch.equal(slots, meta.slot_mapping)
    assert torch.equal(bits(ws.k_cache.cpu()), bits(oc.k))
    assert torch.equal(bits(ws.v_cache.cpu()), bits(oc.v))
    want = oracle.attention(q.cpu(), oc.k, oc.v, meta.block_table, meta.query_start_loc,
                            meta.seq_lens, sh.scale)
    assert_close(out.cpu(), want, "tiny step 3, A twice")
    assert ops.device_status(ws.k_cache, sh.num_q_heads, meta.block_table.shape[1], wsp) == 0
    # A's decode equals the last row of A's one-shot 97-token prefill
    one = oracle_rows_for_seq(ws, "A", 97, 97, rows=[96])
    assert_close(out[33:34].cpu(), one, "A's decode vs one-shot last row")
