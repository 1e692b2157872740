"""A workspace in an unknown state gives the same answer as a fresh one.

Every call rebuilds its work queue and zeroes the split-merge counters it
uses, so whatever an earlier call left in the workspace -- a call that gave up
a bounded wait, a caller's stray write -- cannot leak into the next step.  The
test fills the whole workspace (all but the status word) with random bytes
from the host before each call and checks the result bit for bit against a
call on a zero-filled workspace, and against the fp64 oracle.  The steps are
chosen so that decode sequences and chunk tile pairs are split over several
CTAs (the counters and partial buffers are live), on the tensor-core step
path (bf16) and on the row path (fp32, split over 512-key ranges).
"""
import math

import pytest
import torch

import oracle
from chunked_prefill_paged_cpa_gb300 import ops
from support import oracle_append, make_step
from test_gpu_parity import assert_close, bits

pytestmark = pytest.mark.gpu

CASES = {
    # two chunks over long cached prefixes beside long decodes (split units)
    "bf16 hybrid": ([256, 1, 1, 97, 1, 1], [2256, 3000, 5000, 1400, 700, 9000],
                    torch.bfloat16),
    # long decodes alone: many page slices per sequence, merged by counters
    "bf16 decodes": ([1] * 12, [4000 + 900 * i for i in range(12)], torch.bfloat16),
    # fp32 steps run the row kernel, whose splits merge through counters too
    "f32 hybrid": ([40, 1, 1], [1500, 2100, 700], torch.float32),
}


def _garbage_fill(ws, seed):
    g = torch.Generator().manual_seed(seed)
    junk = torch.randint(0, 256, (ws.numel(),), generator=g, dtype=torch.int32).to(torch.uint8)
    junk[:4] = 0  # the status word: nonzero would (correctly) read as an error
    ws.copy_(junk.to(ws.device))


@pytest.mark.parametrize("name", list(CASES))
def test_garbage_workspace_matches_fresh(cuda_device, name):
    q_lens, seq_lens, dtype = CASES[name]
    Hq, Hkv, D = 32, 8, 128
    st = make_step(q_lens, seq_lens, Hq, Hkv, D, dtype, seed=4100 + len(name))
    dev = cuda_device
    m = st["meta"].to(dev)
    q, k, v = st["q"].to(dev), st["k_new"].to(dev), st["v_new"].to(dev)
    k0, v0 = st["oracle_cache"].k.to(dev), st["oracle_cache"].v.to(dev)
    scale = 1 / math.sqrt(D)
    max_pages = m.block_table.shape[1]

    # reference: fresh zeroed workspace, separate append + attention
    kc, vc = k0.clone(), v0.clone()
    ops.kv_append(k, v, m.slot_mapping, kc, vc)
    ws_ref = ops.workspace_for(kc, Hq, max_pages, m.num_seqs, m.num_tokens)
    ref = ops.attention_forward(q, kc, vc, m.block_table, m.query_start_loc, m.seq_lens,
                                scale, ws_ref)

    # the same calls on a workspace full of random bytes, twice in a row
    ws = ops.workspace_for(kc, Hq, max_pages, m.num_seqs, m.num_tokens)
    for rep in range(2):
        _garbage_fill(ws, 4200 + rep)
        out = ops.attention_forward(q, kc, vc, m.block_table, m.query_start_loc, m.seq_lens,
                                    scale, ws)
        torch.cuda.synchronize()
        assert ops.device_status(kc, Hq, max_pages, ws) == 0
        assert torch.equal(bits(out), bits(ref)), f"{name}: call {rep} differs from fresh"

    # the fused call on a garbage workspace (fresh cache copy)
    kc2, vc2 = k0.clone(), v0.clone()
    _garbage_fill(ws, 4300)
    out2 = ops.append_attention_forward(q, k, v, m.slot_mapping, kc2, vc2, m.block_table,
                                        m.query_start_loc, m.seq_lens, scale, ws)
    torch.cuda.synchronize()
    assert ops.device_status(kc2, Hq, max_pages, ws) == 0
    assert torch.equal(bits(kc2), bits(kc)) and torch.equal(bits(vc2), bits(vc))

    oracle_append(st)
    want = oracle.attention(st["q"], st["oracle_cache"].k, st["oracle_cache"].v,
                            st["meta"].block_table, st["meta"].query_start_loc,
                            st["meta"].seq_lens, scale)
    assert_close(ref.cpu(), want, f"{name}, fresh workspace")
    assert_close(out2.cpu(), want, f"{name}, fused call on a garbage workspace")
