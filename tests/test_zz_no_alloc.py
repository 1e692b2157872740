"""The allocation-free attention entry point, for callers that may not call
cudaMalloc: a plugin inside a runtime that owns all device memory and hands it
only its inputs and outputs, or a serving loop that forbids allocation after
start-up (cudaMalloc/cudaFree can synchronise the device and can fail under
memory pressure in the middle of a step).  It keeps its scratch in a fixed
array inside the library.  It runs the same kernels with the same scratch
layout as the regular entry point, so its output must equal that entry
point's bit for bit, on two calls in a row and after a larger step has left
its state in the array.  Collected last on purpose."""
import ctypes

import pytest
import torch

from chunked_prefill_paged_cpa_gb300 import ops, workloads

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def _prepare(name, device, kv_e4m3=None):
    """A workload's first step with its new K/V already appended, and the
    regular entry point's output on a zero-filled caller workspace
    (``kv_e4m3`` = (k_scale, v_scale): an E4M3 cache)."""
    sc = workloads.scenario(name)
    ws = workloads.WorkloadState(sc, device=device, kv_e4m3=kv_e4m3)
    inp = ws.step(0)
    m = inp["meta"]
    sh = sc.shape
    kw = dict(k_scale=kv_e4m3[0], v_scale=kv_e4m3[1]) if kv_e4m3 else {}
    ops.kv_append(inp["k"], inp["v"], m.slot_mapping, ws.k_cache, ws.v_cache, **kw)
    wsp = ops.workspace_for(ws.k_cache, sh.num_q_heads, m.block_table.shape[1], m.num_seqs,
                            m.num_tokens, inp["q"].dtype)
    assert wsp.numel() <= ops.cpa_noalloc_scratch_bytes()
    ref = ops.attention_forward(inp["q"], ws.k_cache, ws.v_cache, m.block_table,
                                m.query_start_loc, m.seq_lens, sh.scale, wsp, **kw)
    torch.cuda.synchronize()
    return sc, ws, inp, ref


def _noalloc(sc, ws, inp):
    m = inp["meta"]
    sh = sc.shape
    scales = ws.kv_e4m3 or (1.0, 1.0)
    desc = ops.make_desc(ws.k_cache, sh.num_q_heads, m.num_tokens, m.block_table.shape[1],
                         act_dtype=inp["q"].dtype, k_scale=scales[0], v_scale=scales[1])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    out = torch.full_like(inp["q"], float("nan"))
    rc = ops.cpa_attention_forward_noalloc(
        _ptr(inp["q"]), _ptr(ws.k_cache), _ptr(ws.v_cache), _ptr(m.block_table),
        _ptr(m.query_start_loc), _ptr(m.seq_lens), m.num_seqs, sh.scale, _ptr(out),
        stream, desc)
    assert rc == ops.CPA_OK, ops.cpa_status_string(rc)
    torch.cuda.synchronize()
    assert ops.cpa_noalloc_read_device_status(stream) == ops.CPA_OK
    return out


@pytest.mark.parametrize("name", ["tiny", "page1_default", "long_context", "decode_only"])
def test_noalloc_equals_workspace_entry_point_twice(cuda_device, name):
    sc, ws, inp, ref = _prepare(name, cuda_device)
    for _ in range(2):
        out = _noalloc(sc, ws, inp)
        assert torch.equal(_bits(out), _bits(ref))


@pytest.mark.parametrize("name", ["page1_default", "decode_only"])
def test_noalloc_e4m3_cache_equals_workspace_entry_point(cuda_device, name):
    """With an E4M3 cache and bf16 queries the step also keeps the queries'
    binary16 copy in its scratch."""
    sc, ws, inp, ref = _prepare(name, cuda_device, workloads.E4M3_SCALES)
    for _ in range(2):
        out = _noalloc(sc, ws, inp)
        assert torch.equal(_bits(out), _bits(ref))


def test_noalloc_after_a_larger_step(cuda_device):
    """A 256-sequence step leaves its partials and counters in the array; the
    33-sequence step after it must not see them."""
    big = _prepare("decode_only", cuda_device)
    small = _prepare("page1_default", cuda_device)
    out_big = _noalloc(*big[:3])
    out_small = _noalloc(*small[:3])
    assert torch.equal(_bits(out_big), _bits(big[3]))
    assert torch.equal(_bits(out_small), _bits(small[3]))


def test_noalloc_rejects_steps_beyond_its_scratch(cuda_device):
    # 4096 sequences need more split-KV scratch than the fixed array holds
    k_cache = torch.empty(4, 8, 16, 128, dtype=torch.bfloat16, device=cuda_device)
    desc = ops.make_desc(k_cache, 32, 4096, 512)
    assert ops.cpa_workspace_bytes(desc, 4096) > ops.cpa_noalloc_scratch_bytes()
    P = ctypes.c_void_p(k_cache.data_ptr())
    rc = ops.cpa_attention_forward_noalloc(P, P, P, P, P, P, 4096, 0.1, P, None, desc)
    assert rc == ops.CPA_ERR_WORKSPACE
