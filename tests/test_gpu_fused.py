"""The append fused into the attention call (cpa_append_attention_forward).

The fused call must leave the cache holding the same bytes as cpa_kv_append
followed by cpa_attention_forward, and give the same output bits: the same
values reach shared memory by another route (the step's own rows are read
from k/v instead of the cache).  Both are also checked against the oracle.
Shapes cover page-aligned and unaligned chunk starts (a page holding cached
and new rows), decode-only steps, several chunks, the decode kernel's shapes,
and shapes the fused kernels do not take (the call then launches the append
ahead of the attention)."""
import math

import pytest
import torch

import oracle
from chunked_prefill_paged_cpa_gb300 import ops, workloads
from support import oracle_append, make_step
from test_gpu_parity import assert_close, bits, check_full_config, gpu_step

pytestmark = pytest.mark.gpu

BF16, F32 = torch.bfloat16, torch.float32

FUSED_CASES = [
    # (q_lens, seq_lens, Hq, Hkv, D, dtype)
    # page-aligned chunk start (3840 cached) beside decodes: Llama-3-8B shape
    ([1] * 6 + [480], [600, 33, 1500, 17, 4096, 2, 480 + 3840], 32, 8, 128, BF16),
    # chunk starts inside a page (17 and 7 cached tokens) and a chunk with none
    ([33, 1, 129, 1, 40], [50, 1100, 136, 3, 40], 32, 8, 128, BF16),
    # two chunks beside decodes, prefixes 37 and 500 (both unaligned)
    ([1, 1, 1, 100, 100], [600, 1500, 17, 137, 600], 32, 8, 128, BF16),
    # decode-only steps, G = 4 and G = 2
    ([1] * 5, [1, 17, 600, 3000, 16], 32, 8, 128, BF16),
    ([1] * 9, [5, 300, 31, 32, 33, 1200, 2, 7, 999], 16, 8, 128, BF16),
    # head_dim 64: G = 8, G = 4, G = 2 (chunk without prefix, chunk at 1100)
    ([1, 70, 1], [513, 70, 1025], 16, 2, 64, BF16),
    ([200, 1, 1], [1300, 900, 48], 16, 4, 64, BF16),
    ([1, 64, 1], [77, 64 + 160, 3000], 8, 4, 64, BF16),
    # shapes the fused kernels do not take: the call appends first
    ([5, 1, 64], [5, 2049, 100], 4, 2, 64, F32),     # fp32
    ([300, 1], [310, 4000], 8, 1, 128, BF16),        # G = 8 at head_dim 128
    ([40, 1], [40, 50], 8, 8, 128, BF16),            # G = 1
    # a chunk only, no decodes (chunk start inside a page)
    ([129], [129 + 21], 32, 8, 128, BF16),
]


def _run_both(st, Hq, D, dev):
    """The separate calls and the fused call on copies of the same prefix
    cache; returns (separate out, fused out, caches of both, workspace)."""
    m, oc = st["meta"], st["oracle_cache"]
    md = m.to(dev)
    q, k, v = st["q"].to(dev), st["k_new"].to(dev), st["v_new"].to(dev)
    scale = 1 / math.sqrt(D)
    kc1, vc1 = oc.k.to(dev), oc.v.to(dev)
    kc2, vc2 = kc1.clone(), vc1.clone()
    out1, _ = gpu_step(kc1, vc1, {"meta": md, "q": q, "k": k, "v": v}, scale, Hq)
    wsp = ops.workspace_for(kc2, Hq, md.block_table.shape[1], md.num_seqs, md.num_tokens)
    out2 = ops.append_attention_forward(q, k, v, md.slot_mapping, kc2, vc2, md.block_table,
                                        md.query_start_loc, md.seq_lens, scale, wsp)
    torch.cuda.synchronize()
    return out1, out2, (kc1, vc1, kc2, vc2), wsp, (q, k, v, md, scale)


@pytest.mark.parametrize("case", range(len(FUSED_CASES)))
def test_fused_call_equals_separate_calls_and_oracle(cuda_device, case):
    q_lens, seq_lens, Hq, Hkv, D, dtype = FUSED_CASES[case]
    st = make_step(q_lens, seq_lens, Hq, Hkv, D, dtype, seed=1300 + case)
    out1, out2, (kc1, vc1, kc2, vc2), wsp, (q, k, v, md, scale) = _run_both(st, Hq, D,
                                                                            cuda_device)
    # the same cache bytes and the same output bits as the separate calls
    assert torch.equal(bits(kc2), bits(kc1)), "K cache"
    assert torch.equal(bits(vc2), bits(vc1)), "V cache"
    assert torch.equal(bits(out2), bits(out1)), "output"
    # and against the oracle: its own append, then the definition
    m, oc = st["meta"], st["oracle_cache"]
    oracle_append(st)
    assert torch.equal(bits(kc2.cpu()), bits(oc.k)) and torch.equal(bits(vc2.cpu()), bits(oc.v))
    want = oracle.attention(st["q"], oc.k, oc.v, m.block_table, m.query_start_loc,
                            m.seq_lens, scale)
    assert_close(out2.cpu(), want, f"fused case {case}")
    assert ops.device_status(kc2, Hq, md.block_table.shape[1], wsp) == 0
    # a second fused call on the same workspace and cache: the append writes the
    # same bytes again and the output repeats bit for bit
    out3 = ops.append_attention_forward(q, k, v, md.slot_mapping, kc2, vc2, md.block_table,
                                        md.query_start_loc, md.seq_lens, scale, wsp)
    torch.cuda.synchronize()
    assert torch.equal(bits(out3), bits(out2))
    assert torch.equal(bits(kc2), bits(kc1)) and torch.equal(bits(vc2), bits(vc1))


def test_fused_out_of_range_slot_sets_status_without_fault(cuda_device):
    """A slot past the cache is neither written nor read: the status word
    reports it, in the fused path as in the separate append."""
    q_lens, seq_lens = [1, 1, 50], [300, 40, 50 + 32]
    st = make_step(q_lens, seq_lens, 32, 8, 128, BF16, seed=1401)
    dev = cuda_device
    m, oc = st["meta"].to(dev), st["oracle_cache"]
    kc, vc = oc.k.to(dev), oc.v.to(dev)
    slots = m.slot_mapping.clone()
    slots[0] = kc.shape[0] * 16 + 5            # the first decode's token: out of range
    wsp = ops.workspace_for(kc, 32, m.block_table.shape[1], m.num_seqs, m.num_tokens)
    ops.append_attention_forward(st["q"].to(dev), st["k_new"].to(dev), st["v_new"].to(dev),
                                 slots, kc, vc, m.block_table, m.query_start_loc, m.seq_lens,
                                 1 / math.sqrt(128), wsp)
    torch.cuda.synchronize()
    assert ops.device_status(kc, 32, m.block_table.shape[1], wsp) != 0


@pytest.mark.parametrize("name", ["page1_default", "long_context"])
def test_full_size_config_fused(name, cuda_device):
    """The full-size workloads through the fused call, in the launch
    configuration the benchmark times, against sampled oracle rows."""
    check_full_config(name, cuda_device, fused=True)
