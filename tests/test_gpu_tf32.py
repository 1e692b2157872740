"""fp32 steps: the chunk rows on the tensor cores (tcgen05.mma kind::tf32),
the decode rows on the row kernel, both against the fp64 oracle.

The tensor core rounds the products' inputs to tf32 (10 mantissa bits); the
bar is the one for every attention output here, max-abs 2e-2 and mean-abs
2e-3 of the oracle.  Chunk rows follow "vllm-learning-book 05. Chunked
Prefill", section 3: row i of a chunk of q_len tokens among ctx keys sees keys
0 .. ctx - q_len + i.  Cases cover head_dim 64 and 128, every GQA group,
chunks from an empty prefix, an unaligned prefix and a prefix ending one key
short of a page, chunks of several 128-row tiles with a partial last one,
several 64-key KV tiles, and decodes in the same step.
"""
import math

import pytest
import torch

import oracle
from chunked_prefill_paged_cpa_gb300 import ops
from support import make_step, oracle_append

from test_gpu_parity import assert_close, bits, gpu_step

pytestmark = pytest.mark.gpu


def _cases():
    out = []
    for D in (64, 128):
        for G in (1, 2, 4, 8):
            full = 2 * (128 // G) + 1  # two full 128-row tiles and one row
            out.append((D, G, [40, 1, 97, 1, full, 2], [40, 300, 247, 64, full + 130, 513]))
    return out


CASES = _cases()


@pytest.mark.parametrize("case", range(len(CASES)),
                         ids=[f"D{c[0]}-G{c[1]}" for c in CASES])
def test_fp32_chunk_rows_on_tf32_match_oracle(cuda_device, case):
    D, G, q_lens, seq_lens = CASES[case]
    Hkv = 2
    Hq = Hkv * G
    st = make_step(q_lens, seq_lens, Hq, Hkv, D, torch.float32, seed=700 + case)
    m, oc = st["meta"], st["oracle_cache"]
    dev = cuda_device
    k_cache, v_cache = oc.k.to(dev), oc.v.to(dev)
    inp = {"meta": m.to(dev), "q": st["q"].to(dev), "k": st["k_new"].to(dev),
           "v": st["v_new"].to(dev)}
    scale = 1 / math.sqrt(D)
    out, wsp = gpu_step(k_cache, v_cache, inp, scale, Hq)
    assert ops.device_status(k_cache, Hq, m.block_table.shape[1], wsp) == ops.CPA_OK
    oracle_append(st)
    assert torch.equal(bits(k_cache.cpu()), bits(oc.k))
    want = oracle.attention(st["q"], oc.k, oc.v, m.block_table, m.query_start_loc,
                            m.seq_lens, scale)
    got = out.cpu()
    qsl = m.query_start_loc.tolist()
    for s, ql in enumerate(q_lens):
        rows = slice(qsl[s], qsl[s + 1])
        assert_close(got[rows], want[rows], f"D{D} G{G} seq {s} (q_len {ql})")


def test_fp32_fused_call_matches_separate_calls(cuda_device):
    """The fused call on an fp32 step runs the append, the tf32 chunk kernel
    and the row kernel; the cache and the output equal the separate calls'."""
    q_lens, seq_lens = [70, 1, 33], [70 + 45, 200, 33]
    st = make_step(q_lens, seq_lens, 8, 2, 64, torch.float32, seed=790)
    m, oc = st["meta"], st["oracle_cache"]
    dev = cuda_device
    md = m.to(dev)
    q, k, v = st["q"].to(dev), st["k_new"].to(dev), st["v_new"].to(dev)
    kc1, vc1 = oc.k.to(dev), oc.v.to(dev)
    kc2, vc2 = kc1.clone(), vc1.clone()
    wsp = ops.workspace_for(kc1, 8, md.block_table.shape[1], md.num_seqs, md.num_tokens)
    ops.kv_append(k, v, md.slot_mapping, kc1, vc1)
    sep = ops.attention_forward(q, kc1, vc1, md.block_table, md.query_start_loc, md.seq_lens,
                                0.125, wsp)
    fused = ops.append_attention_forward(q, k, v, md.slot_mapping, kc2, vc2, md.block_table,
                                         md.query_start_loc, md.seq_lens, 0.125, wsp)
    torch.cuda.synchronize()
    assert torch.equal(bits(kc1), bits(kc2)) and torch.equal(bits(vc1), bits(vc2))
    assert torch.equal(bits(sep), bits(fused))


def test_fp32_chunk_with_bad_page_sets_status_without_fault(cuda_device):
    dev = cuda_device
    st = make_step([40], [80], 4, 2, 64, torch.float32, seed=791)
    m, oc = st["meta"], st["oracle_cache"]
    k_cache, v_cache = oc.k.to(dev), oc.v.to(dev)
    md = m.to(dev)
    ops.kv_append(st["k_new"].to(dev), st["v_new"].to(dev), md.slot_mapping, k_cache, v_cache)
    bt = md.block_table.clone()
    bt[0, 1] = 10 ** 6  # keys 16..31 of the chunk's prefix: not a page of the pool
    wsp = ops.workspace_for(k_cache, 4, bt.shape[1], 1, md.num_tokens)
    out = ops.attention_forward(st["q"].to(dev), k_cache, v_cache, bt, md.query_start_loc,
                                md.seq_lens, 0.125, wsp)
    assert ops.device_status(k_cache, 4, bt.shape[1], wsp) == ops.CPA_ERR_DEVICE
    assert torch.isfinite(out).all()   # the page reads as zeros
