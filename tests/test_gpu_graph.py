"""The step (append + attention) captured in a CUDA graph and replayed.

The attention call is two launches on the caller's stream (the plan kernel,
then the persistent step kernel as its programmatic dependent), launches
nothing that synchronises, and rebuilds its work queue and counters itself, so
a captured step replays to the same bits as the eager call on the same inputs
-- and again on a second replay."""
import math

import pytest
import torch

from chunked_prefill_paged_cpa_gb300 import ops
from support import make_step

pytestmark = pytest.mark.gpu


def bits(t):
    return t.contiguous().view(torch.int16) if t.dtype == torch.bfloat16 else t


def test_captured_step_replays_bit_for_bit(cuda_device):
    # two chunks (one with a cached prefix) beside four decodes: chunk tiles and
    # decode slices share the step kernel's work queue
    q_lens = [33, 1, 129, 1, 1, 1]
    seq_lens = [50, 1100, 429, 3, 700, 2000]
    Hq, Hkv, D = 32, 8, 128
    st = make_step(q_lens, seq_lens, Hq, Hkv, D, torch.bfloat16, seed=321)
    dev = cuda_device
    m = st["meta"].to(dev)
    q, k, v = st["q"].to(dev), st["k_new"].to(dev), st["v_new"].to(dev)
    k0, v0 = st["oracle_cache"].k.to(dev), st["oracle_cache"].v.to(dev)
    scale = 1 / math.sqrt(D)
    max_pages = m.block_table.shape[1]

    # eager reference
    kc, vc = k0.clone(), v0.clone()
    ws_e = ops.workspace_for(kc, Hq, max_pages, m.num_seqs, m.num_tokens)
    ops.kv_append(k, v, m.slot_mapping, kc, vc)
    out_e = ops.attention_forward(q, kc, vc, m.block_table, m.query_start_loc, m.seq_lens,
                                  scale, ws_e)
    torch.cuda.synchronize()

    # capture on static buffers (warm-up first, as graph capture requires)
    kg, vg = k0.clone(), v0.clone()
    ws_g = ops.workspace_for(kg, Hq, max_pages, m.num_seqs, m.num_tokens)
    out_g = torch.empty_like(out_e)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ops.kv_append(k, v, m.slot_mapping, kg, vg)
        ops.attention_forward(q, kg, vg, m.block_table, m.query_start_loc, m.seq_lens,
                              scale, ws_g, out=out_g)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ops.kv_append(k, v, m.slot_mapping, kg, vg)
        ops.attention_forward(q, kg, vg, m.block_table, m.query_start_loc, m.seq_lens,
                              scale, ws_g, out=out_g)

    for replay in range(2):
        kg.copy_(k0)
        vg.copy_(v0)
        out_g.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(bits(kg), bits(kc)), f"replay {replay}: K cache"
        assert torch.equal(bits(vg), bits(vc)), f"replay {replay}: V cache"
        assert torch.equal(bits(out_g), bits(out_e)), f"replay {replay}: attention output"
    assert ops.device_status(kg, Hq, max_pages, ws_g) == 0


def test_captured_fused_call_replays_bit_for_bit(cuda_device):
    """cpa_append_attention_forward (the append fused into the attention
    kernels) captured in a CUDA graph: every replay leaves the same cache bytes
    and output bits as the eager call."""
    q_lens = [33, 1, 129, 1, 1, 1]
    seq_lens = [50, 1100, 429, 3, 700, 2000]
    Hq, Hkv, D = 32, 8, 128
    st = make_step(q_lens, seq_lens, Hq, Hkv, D, torch.bfloat16, seed=322)
    dev = cuda_device
    m = st["meta"].to(dev)
    q, k, v = st["q"].to(dev), st["k_new"].to(dev), st["v_new"].to(dev)
    k0, v0 = st["oracle_cache"].k.to(dev), st["oracle_cache"].v.to(dev)
    scale = 1 / math.sqrt(D)
    max_pages = m.block_table.shape[1]

    kc, vc = k0.clone(), v0.clone()
    ws_e = ops.workspace_for(kc, Hq, max_pages, m.num_seqs, m.num_tokens)
    out_e = ops.append_attention_forward(q, k, v, m.slot_mapping, kc, vc, m.block_table,
                                         m.query_start_loc, m.seq_lens, scale, ws_e)
    torch.cuda.synchronize()

    kg, vg = k0.clone(), v0.clone()
    ws_g = ops.workspace_for(kg, Hq, max_pages, m.num_seqs, m.num_tokens)
    out_g = torch.empty_like(out_e)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ops.append_attention_forward(q, k, v, m.slot_mapping, kg, vg, m.block_table,
                                     m.query_start_loc, m.seq_lens, scale, ws_g, out=out_g)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ops.append_attention_forward(q, k, v, m.slot_mapping, kg, vg, m.block_table,
                                     m.query_start_loc, m.seq_lens, scale, ws_g, out=out_g)
    for replay in range(2):
        kg.copy_(k0)
        vg.copy_(v0)
        out_g.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(bits(kg), bits(kc)), f"replay {replay}: K cache"
        assert torch.equal(bits(vg), bits(vc)), f"replay {replay}: V cache"
        assert torch.equal(bits(out_g), bits(out_e)), f"replay {replay}: attention output"
    assert ops.device_status(kg, Hq, max_pages, ws_g) == 0
