"""The 8-bit (OCP FP8 E4M3) cache and binary16 activations on the GPU, against
the fp64 oracle.

* The quantising append (separate and fused into the attention call) stores,
  bit for bit, the oracle's codes of x / scale at the oracle's slots, planted
  rounding ties, saturation, infinities and signed zeros included.
* Attention over an E4M3 cache matches the oracle run on the same codes (the
  oracle widens them exactly and multiplies by the scales) on every head_dim /
  GQA group shape, with bf16 and binary16 queries, several scales, chunks over
  cached prefixes beside decodes, and at full size on the default hybrid step
  (every row) and the decode-only step (every row of every 8th decode).
* binary16 queries with a binary16 cache match the oracle too.

Bars as for bf16: max-abs 2e-2 and mean-abs 2e-3 against the oracle; cache
bytes bit-exact.  The oracle's E4M3 arithmetic is pinned on the CPU
(tests/test_oracle_fp8.py).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from chunked_prefill_paged_cpa_gb300 import ops, workloads
from support import make_step
from test_gpu_parity import assert_close

pytestmark = pytest.mark.gpu

POISON = 0x7f  # the NaN code: a read of an unused slot would show up as NaN


def fp8_step(q_lens, seq_lens, Hq, Hkv, D, act, seed, ks, vs, transform=None):
    """A one-step problem whose caches hold E4M3 codes: the prefix written by
    the oracle's quantising append at the oracle's own slots."""
    st = make_step(q_lens, seq_lens, Hq, Hkv, D, act, seed, transform=transform)
    m = st["meta"]
    shape = (st["pool"], Hkv, 16, D)
    kc = torch.full(shape, POISON, dtype=torch.uint8)
    vc = kc.clone()
    pre = [L - q for q, L in zip(q_lens, seq_lens)]
    idx = [i for i, p in enumerate(pre) if p > 0]
    if idx:
        bt = m.block_table[idx]
        qsl = torch.zeros(len(idx) + 1, dtype=torch.int32)
        qsl[1:] = torch.cumsum(torch.tensor([pre[i] for i in idx], dtype=torch.int32), 0)
        sl = torch.tensor([pre[i] for i in idx], dtype=torch.int32)
        slots = oracle.slot_mapping(bt, qsl, sl, 16)
        oracle.kv_append_e4m3(kc, vc, torch.cat([st["k_seqs"][i][:pre[i]] for i in idx]),
                              torch.cat([st["v_seqs"][i][:pre[i]] for i in idx]), slots, ks, vs)
    st["kc8"], st["vc8"] = kc, vc
    return st


def oracle_fp8(st, ks, vs, scale):
    """Oracle append of the step's new rows, then attention on the codes."""
    m = st["meta"]
    slots = oracle.slot_mapping(m.block_table, m.query_start_loc, m.seq_lens, 16)
    assert torch.equal(slots, m.slot_mapping.cpu())
    oracle.kv_append_e4m3(st["kc8"], st["vc8"], st["k_new"], st["v_new"], slots, ks, vs)
    return oracle.attention(st["q"], st["kc8"], st["vc8"], m.block_table, m.query_start_loc,
                            m.seq_lens, scale, k_scale=ks, v_scale=vs)


def _specials(act, scale):
    """Values whose codes exercise every corner of the quantiser at a
    power-of-two scale (so each x / scale below is exact)."""
    base = [0.0, -0.0, 1.0625, -1.1875, 15.5, 2.0 ** -10, 3 * 2.0 ** -11, 448.0, 460.0,
            1.0e6, float("inf"), float("-inf"), 2.0 ** -9, 7 * 2.0 ** -9, -3.0]
    return torch.tensor([b * scale for b in base], dtype=torch.float32).to(act)


@pytest.mark.parametrize("act", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("fused", [False, True])
def test_quantising_append_is_bitexact(cuda_device, act, fused):
    ks, vs = 2.0 ** -4, 0.037  # one power of two (exact ties), one not
    q_lens, seq_lens = [1, 45, 1, 3], [70, 300, 16, 3]

    def plant(q, k_seqs, v_seqs):
        sk, sv = _specials(act, ks), _specials(act, vs)
        for k, v in zip(k_seqs, v_seqs):  # the last (new) row of every sequence
            k[-1, 0, :sk.numel()] = sk
            v[-1, 1, :sv.numel()] = sv
        return q, k_seqs, v_seqs

    st = fp8_step(q_lens, seq_lens, 16, 4, 128, act, 5100 + fused, ks, vs, transform=plant)
    dev = cuda_device
    m = st["meta"].to(dev)
    kc, vc = st["kc8"].to(dev), st["vc8"].to(dev)
    q, k, v = st["q"].to(dev), st["k_new"].to(dev), st["v_new"].to(dev)
    wsp = ops.workspace_for(kc, 16, m.block_table.shape[1], m.num_seqs, m.num_tokens, act)
    if fused:
        ops.append_attention_forward(q, k, v, m.slot_mapping, kc, vc, m.block_table,
                                     m.query_start_loc, m.seq_lens, 0.1, wsp,
                                     k_scale=ks, v_scale=vs)
    else:
        ops.kv_append(k, v, m.slot_mapping, kc, vc, wsp, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert ops.device_status(kc, 16, m.block_table.shape[1], wsp) == 0
    oracle_fp8(st, ks, vs, 0.1)
    assert torch.equal(kc.cpu(), st["kc8"]), "K codes differ from the oracle's"
    assert torch.equal(vc.cpu(), st["vc8"]), "V codes differ from the oracle's"


SHAPES = [(D, G) for D in (64, 128) for G in (1, 2, 4, 8)]


@pytest.mark.parametrize("D,G", SHAPES)
@pytest.mark.parametrize("act", [torch.bfloat16, torch.float16])
def test_e4m3_attention_matches_oracle(cuda_device, D, G, act):
    Hkv = 8 // G if G < 8 else 2
    Hq = Hkv * G
    # decodes (one past a page end, one inside the first page), a chunk over an
    # unaligned cached prefix, a chunk from scratch, long decodes split into slices
    q_lens = [1, 37, 1, 200, 1, 1]
    seq_lens = [301, 537, 9, 200, 2600, 1800]
    ks, vs = (0.013, 0.029) if act == torch.bfloat16 else (2.0 ** -6, 0.5)
    st = fp8_step(q_lens, seq_lens, Hq, Hkv, D, act, 5200 + 10 * D + G, ks, vs)
    dev = cuda_device
    m = st["meta"].to(dev)
    q, k, v = st["q"].to(dev), st["k_new"].to(dev), st["v_new"].to(dev)
    scale = 1 / math.sqrt(D)
    # separate calls
    kc1, vc1 = st["kc8"].to(dev), st["vc8"].to(dev)
    wsp = ops.workspace_for(kc1, Hq, m.block_table.shape[1], m.num_seqs, m.num_tokens, act)
    ops.kv_append(k, v, m.slot_mapping, kc1, vc1, wsp, k_scale=ks, v_scale=vs)
    out1 = ops.attention_forward(q, kc1, vc1, m.block_table, m.query_start_loc, m.seq_lens,
                                 scale, wsp, k_scale=ks, v_scale=vs)
    # the fused call on a second copy
    kc2, vc2 = st["kc8"].to(dev), st["vc8"].to(dev)
    out2 = ops.append_attention_forward(q, k, v, m.slot_mapping, kc2, vc2, m.block_table,
                                        m.query_start_loc, m.seq_lens, scale, wsp,
                                        k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert out1.dtype == act
    assert ops.device_status(kc1, Hq, m.block_table.shape[1], wsp) == 0
    assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    want = oracle_fp8(st, ks, vs, scale)
    assert torch.equal(kc1.cpu(), st["kc8"])
    assert_close(out1.cpu(), want, f"E4M3 cache D={D} G={G} {act}")


@pytest.mark.parametrize("D,G", [(128, 4), (64, 8), (128, 1)])
def test_binary16_activations_and_cache_match_oracle(cuda_device, D, G):
    Hkv = 8 // G if G < 8 else 2
    Hq = Hkv * G
    q_lens = [1, 64, 1, 130]
    seq_lens = [777, 64 + 1000, 40, 130]
    st = make_step(q_lens, seq_lens, Hq, Hkv, D, torch.float16, 5300 + D + G)
    dev = cuda_device
    m = st["meta"].to(dev)
    q, k, v = st["q"].to(dev), st["k_new"].to(dev), st["v_new"].to(dev)
    kc, vc = st["oracle_cache"].k.to(dev), st["oracle_cache"].v.to(dev)
    wsp = ops.workspace_for(kc, Hq, m.block_table.shape[1], m.num_seqs, m.num_tokens)
    out = ops.append_attention_forward(q, k, v, m.slot_mapping, kc, vc, m.block_table,
                                       m.query_start_loc, m.seq_lens, 1 / math.sqrt(D), wsp)
    torch.cuda.synchronize()
    assert out.dtype == torch.float16
    assert ops.device_status(kc, Hq, m.block_table.shape[1], wsp) == 0
    mc = st["meta"]
    slots = oracle.slot_mapping(mc.block_table, mc.query_start_loc, mc.seq_lens, 16)
    oracle.kv_append(st["oracle_cache"].k, st["oracle_cache"].v, st["k_new"], st["v_new"], slots)
    assert torch.equal(kc.cpu().view(torch.int16), st["oracle_cache"].k.view(torch.int16))
    want = oracle.attention(st["q"], st["oracle_cache"].k, st["oracle_cache"].v, mc.block_table,
                            mc.query_start_loc, mc.seq_lens, 1 / math.sqrt(D))
    assert_close(out.cpu(), want, f"binary16 D={D} G={G}")


def oracle_rows_e4m3(ws, rid, seq_len, q_len, ks, vs):
    """Oracle output of a sequence's new rows over an identity-paged 8-bit
    cache built by the oracle's own quantising append."""
    sh = ws.sc.shape
    n = -(-seq_len // 16)
    kc = torch.full((n, sh.num_kv_heads, 16, sh.head_dim), POISON, dtype=torch.uint8)
    vc = kc.clone()
    bt = torch.arange(n, dtype=torch.int32).view(1, n)
    allq = torch.tensor([0, seq_len], dtype=torch.int32)
    sl = torch.tensor([seq_len], dtype=torch.int32)
    kk, vv = ws.kv_rows(rid, torch.arange(seq_len))
    oracle.kv_append_e4m3(kc, vc, kk.cpu(), vv.cpu(), oracle.slot_mapping(bt, allq, sl, 16), ks, vs)
    q = ws.q_rows(rid, torch.arange(seq_len - q_len, seq_len)).cpu()
    qsl = torch.tensor([0, q_len], dtype=torch.int32)
    return oracle.attention(q, kc, vc, bt, qsl, sl, sh.scale, k_scale=ks, v_scale=vs)


@pytest.mark.parametrize("name,every", [("decode_only", 8), ("page1_default", 1)])
def test_full_size_e4m3(cuda_device, name, every):
    """Full-size steps through the fused call: every row of page1_default and
    every row of every 8th decode of decode_only (the oracle quantises each
    checked sequence's whole context itself, about 10 M codes a second)."""
    ks, vs = workloads.E4M3_SCALES
    sc = workloads.scenario(name)
    ws = workloads.WorkloadState(sc, device=cuda_device, kv_e4m3=(ks, vs))
    inp = ws.step(0)
    m = inp["meta"]
    sh = sc.shape
    wsp = ops.workspace_for(ws.k_cache, sh.num_q_heads, m.block_table.shape[1], m.num_seqs,
                            m.num_tokens, sh.dtype)
    out = ops.append_attention_forward(inp["q"], inp["k"], inp["v"], m.slot_mapping,
                                       ws.k_cache, ws.v_cache, m.block_table, m.query_start_loc,
                                       m.seq_lens, sh.scale, wsp, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert ops.device_status(ws.k_cache, sh.num_q_heads, m.block_table.shape[1], wsp) == 0
    got = out.float().cpu().numpy()
    qsl = m.query_start_loc.cpu().tolist()
    want = np.empty_like(got, dtype=np.float64)
    checked = []
    for i, s in enumerate(inp["plan"].seqs):
        if i % every:
            continue
        want[qsl[i]:qsl[i + 1]] = oracle_rows_e4m3(ws, s.rid, s.seq_len, s.q_len, ks, vs)
        assert_close(got[qsl[i]:qsl[i + 1]], want[qsl[i]:qsl[i + 1]],
                     f"{name} E4M3 seq {s.rid} ({s.kind}, ctx {s.seq_len})")
        checked += list(range(qsl[i], qsl[i + 1]))
    assert_close(got[checked], want[checked], f"{name} E4M3")
    # the new rows' codes are the oracle's
    sd = m.slot_mapping
    want_k = oracle.e4m3_encode(inp["k"].cpu(), ks)
    assert torch.equal(ws.k_cache[sd // 16, :, sd % 16, :].cpu(), want_k)


@pytest.mark.parametrize("mode", ["bf16", "f16", "e4m3_bf16", "e4m3_f16"])
def test_long_decode_slices_every_cache_mode(cuda_device, mode):
    """Decode slices long enough for every pipeline to run its look-ahead
    (several 128-key blocks per slice, slice lengths of every residue mod 4,
    so the last fills of a slice meet the widening window in every position)
    beside a chunk, in every cache mode."""
    act = torch.float16 if mode.endswith("f16") else torch.bfloat16
    e4m3 = mode.startswith("e4m3")
    n = 12
    q_lens = [1] * n + [48]
    seq_lens = [6000 + 130 * i for i in range(n)] + [48 + 700]
    ks, vs = 0.021, 0.043
    D, Hq, Hkv = 128, 32, 8
    scale = 1 / math.sqrt(D)
    dev = cuda_device
    if e4m3:
        st = fp8_step(q_lens, seq_lens, Hq, Hkv, D, act, 5400, ks, vs)
        kc, vc = st["kc8"].to(dev), st["vc8"].to(dev)
    else:
        st = make_step(q_lens, seq_lens, Hq, Hkv, D, act, 5400)
        kc, vc = st["oracle_cache"].k.to(dev), st["oracle_cache"].v.to(dev)
    m = st["meta"].to(dev)
    q, k, v = st["q"].to(dev), st["k_new"].to(dev), st["v_new"].to(dev)
    wsp = ops.workspace_for(kc, Hq, m.block_table.shape[1], m.num_seqs, m.num_tokens, act)
    kw = dict(k_scale=ks, v_scale=vs) if e4m3 else {}
    out = ops.append_attention_forward(q, k, v, m.slot_mapping, kc, vc, m.block_table,
                                       m.query_start_loc, m.seq_lens, scale, wsp, **kw)
    torch.cuda.synchronize()
    assert ops.device_status(kc, Hq, m.block_table.shape[1], wsp) == 0
    if e4m3:
        want = oracle_fp8(st, ks, vs, scale)
    else:
        mc = st["meta"]
        slots = oracle.slot_mapping(mc.block_table, mc.query_start_loc, mc.seq_lens, 16)
        oracle.kv_append(st["oracle_cache"].k, st["oracle_cache"].v, st["k_new"], st["v_new"], slots)
        want = oracle.attention(st["q"], st["oracle_cache"].k, st["oracle_cache"].v,
                                mc.block_table, mc.query_start_loc, mc.seq_lens, scale)
    assert_close(out.cpu(), want, f"long decode slices, {mode}")
