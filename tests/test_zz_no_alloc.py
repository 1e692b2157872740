"""The allocation-free attention entry point, for callers that may not call
cudaMalloc (e.g. a plugin inside a runtime that owns all device memory, or a
serving loop that forbids allocation after start-up).  It keeps its scratch in
a fixed array inside the library; its results must match the regular entry
point (which takes a caller workspace) within the parity tolerance, on two
calls in a row.  Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from chunked_prefill_paged_cpa_gb300 import ops, workloads

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _check(got, want):
    err = (got.double() - want.double()).abs()
    assert torch.isfinite(got.double()).all()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS


@pytest.mark.parametrize("name", ["tiny", "page1_default"])
def test_noalloc_matches_workspace_entry_point_twice(cuda_device, name):
    sc = workloads.scenario(name)
    ws = workloads.WorkloadState(sc, device=cuda_device)
    inp = ws.step(0)
    m = inp["meta"]
    sh = sc.shape
    ops.kv_append(inp["k"], inp["v"], m.slot_mapping, ws.k_cache, ws.v_cache)
    wsp = ops.workspace_for(ws.k_cache, sh.num_q_heads, m.block_table.shape[1], m.num_seqs)
    assert wsp.numel() <= ops.CPA_NOALLOC_SCRATCH_BYTES
    ref = ops.attention_forward(inp["q"], ws.k_cache, ws.v_cache, m.block_table,
                                m.query_start_loc, m.seq_lens, sh.scale, wsp)
    desc = ops.make_desc(ws.k_cache, sh.num_q_heads, m.num_tokens, m.block_table.shape[1])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    outs = []
    for _ in range(2):
        out = torch.full_like(inp["q"], float("nan"))
        rc = ops.cpa_attention_forward_noalloc(
            _ptr(inp["q"]), _ptr(ws.k_cache), _ptr(ws.v_cache), _ptr(m.block_table),
            _ptr(m.query_start_loc), _ptr(m.seq_lens), m.num_seqs, sh.scale, _ptr(out),
            stream, desc)
        assert rc == ops.CPA_OK, ops.cpa_status_string(rc)
        torch.cuda.synchronize()
        _check(out, ref)
        outs.append(out)
    _check(outs[1], outs[0])


def test_noalloc_rejects_steps_beyond_its_scratch(cuda_device):
    # 1024 sequences need more split-KV scratch than the fixed array holds
    k_cache = torch.empty(4, 8, 16, 128, dtype=torch.bfloat16, device=cuda_device)
    desc = ops.make_desc(k_cache, 32, 1024, 512)
    assert ops.cpa_workspace_bytes(desc, 1024) > ops.CPA_NOALLOC_SCRATCH_BYTES
    P = ctypes.c_void_p(k_cache.data_ptr())
    rc = ops.cpa_attention_forward_noalloc(P, P, P, P, P, P, 1024, 0.1, P, None, desc)
    assert rc == ops.CPA_ERR_WORKSPACE
