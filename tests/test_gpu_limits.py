"""Edges of the supported sizes, on the GPU.

The plan kernel holds each sequence's metadata (lengths, item counts, queue
offsets) in shared memory, up to 4096 sequences per call; a larger batch is
refused on the host (CPA_ERR_UNSUPPORTED) before anything is launched.  The largest batch is
checked against the oracle through both the separate calls and the fused
append + attention call."""
import math

import pytest
import torch

import oracle
from chunked_prefill_paged_cpa_gb300 import ops
from support import oracle_append, make_step
from test_gpu_parity import assert_close, bits, gpu_step

pytestmark = pytest.mark.gpu

MAX_DECODE_SEQS = 4096


def test_largest_decode_batch_separate_and_fused(cuda_device):
    g = torch.Generator().manual_seed(1700)
    seq_lens = torch.randint(1, 40, (MAX_DECODE_SEQS,), generator=g).tolist()
    q_lens = [1] * MAX_DECODE_SEQS
    st = make_step(q_lens, seq_lens, 32, 8, 128, torch.bfloat16, seed=1701)
    dev = cuda_device
    m, oc = st["meta"], st["oracle_cache"]
    md = m.to(dev)
    q, k, v = st["q"].to(dev), st["k_new"].to(dev), st["v_new"].to(dev)
    scale = 1 / math.sqrt(128)
    kc1, vc1 = oc.k.to(dev), oc.v.to(dev)
    kc2, vc2 = kc1.clone(), vc1.clone()
    out1, wsp1 = gpu_step(kc1, vc1, {"meta": md, "q": q, "k": k, "v": v}, scale, 32)
    wsp2 = ops.workspace_for(kc2, 32, md.block_table.shape[1], md.num_seqs, md.num_tokens)
    out2 = ops.append_attention_forward(q, k, v, md.slot_mapping, kc2, vc2, md.block_table,
                                        md.query_start_loc, md.seq_lens, scale, wsp2)
    torch.cuda.synchronize()
    assert torch.equal(bits(kc2), bits(kc1)) and torch.equal(bits(vc2), bits(vc1))
    assert torch.equal(bits(out2), bits(out1))
    oracle_append(st)
    assert torch.equal(bits(kc1.cpu()), bits(oc.k))
    want = oracle.attention(st["q"], oc.k, oc.v, m.block_table, m.query_start_loc,
                            m.seq_lens, scale)
    assert_close(out1.cpu(), want, "4096 decodes")
    for wsp, kc in ((wsp1, kc1), (wsp2, kc2)):
        assert ops.device_status(kc, 32, md.block_table.shape[1], wsp) == 0


def test_one_more_sequence_than_supported_is_refused(cuda_device):
    n = MAX_DECODE_SEQS + 1
    st = make_step([1] * n, [3] * n, 32, 8, 128, torch.bfloat16, seed=1702)
    dev = cuda_device
    m, oc = st["meta"].to(dev), st["oracle_cache"]
    kc, vc = oc.k.to(dev), oc.v.to(dev)
    wsp = ops.workspace_for(kc, 32, m.block_table.shape[1], m.num_seqs, m.num_tokens)
    q, k, v = st["q"].to(dev), st["k_new"].to(dev), st["v_new"].to(dev)
    before_k, before_v = kc.clone(), vc.clone()
    with pytest.raises(ops.CpaError) as e:
        ops.attention_forward(q, kc, vc, m.block_table, m.query_start_loc, m.seq_lens,
                              1 / math.sqrt(128), wsp)
    assert e.value.status == ops.CPA_ERR_UNSUPPORTED
    with pytest.raises(ops.CpaError) as e:
        ops.append_attention_forward(q, k, v, m.slot_mapping, kc, vc, m.block_table,
                                     m.query_start_loc, m.seq_lens, 1 / math.sqrt(128), wsp)
    assert e.value.status == ops.CPA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    # refused before any launch: the cache is untouched
    assert torch.equal(bits(kc), bits(before_k)) and torch.equal(bits(vc), bits(before_v))
