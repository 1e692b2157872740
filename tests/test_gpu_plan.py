"""The device work queue the plan kernel builds for the step kernel.

After a call the workspace still holds the step's queue, so the schedule can
be checked directly: every decode (sequence, kv head) segment is cut into
slices that cover its pages exactly once, every chunk tile pair is cut into
units with every unit present once, the chunk units come first and the decode
slices follow longest first, and the queue ticket shows that every CTA
claimed until the queue ran dry.  Parity of the outputs is checked elsewhere;
this pins the scheduling itself ("vllm-learning-book 05. Chunked Prefill",
section 4: one packed batch, no padding, work handed out from one list).

Queue entry (8 int32): s | kind << 30, query start, context, q_len (decode:
slices of the segment), kv head | (pair or slice index) << 8, then for chunk
units (unit | units << 16, own index, first unit of the pair) and for decode
slices (first page, end page, slice index).  Header at byte 64: chunk units,
decode slices, entries, pages per slice, ticket.  Entries from byte 256.
"""
import math

import pytest
import torch

from chunked_prefill_paged_cpa_gb300 import ops, workloads

pytestmark = pytest.mark.gpu


def _run(name, cuda_device):
    sc = workloads.free_ride(int(name.split("_")[-1])) if name.startswith("free_ride_") \
        else workloads.scenario(name)
    ws = workloads.WorkloadState(sc, device=cuda_device)
    inp = ws.step(0)
    m = inp["meta"]
    sh = sc.shape
    wsp = ops.workspace_for(ws.k_cache, sh.num_q_heads, m.block_table.shape[1], m.num_seqs,
                            m.num_tokens)
    ops.append_attention_forward(inp["q"], inp["k"], inp["v"], m.slot_mapping, ws.k_cache,
                                 ws.v_cache, m.block_table, m.query_start_loc, m.seq_lens,
                                 sh.scale, wsp)
    torch.cuda.synchronize()
    assert ops.device_status(ws.k_cache, sh.num_q_heads, m.block_table.shape[1], wsp) == 0
    return sc, m, wsp.cpu()


@pytest.mark.parametrize("name", ["page1_default", "large_budget", "long_context",
                                  "decode_only", "free_ride_64", "oneshot_8192"])
def test_queue_covers_every_page_and_tile_once(cuda_device, name):
    sc, m, wsp = _run(name, cuda_device)
    sh = sc.shape
    G, Hkv = sh.num_q_heads // sh.num_kv_heads, sh.num_kv_heads
    hdr = wsp[64:84].view(torch.int32).tolist()
    n_chunk, n_dec, n_items, P, ticket = hdr
    assert n_items == n_chunk + n_dec
    # each CTA claimed until the queue ran dry: one claim per entry past the
    # grid plus one failed claim per CTA that had work
    assert ticket == n_items
    q = wsp[256:256 + 32 * n_items].view(torch.int32).view(n_items, 8).tolist()
    qsl = m.query_start_loc.cpu().tolist()
    ctxs = m.seq_lens.cpu().tolist()

    chunk, dec = q[:n_chunk], q[n_chunk:]
    assert all((e[0] >> 30) == 0 for e in chunk) and all((e[0] >> 30) == 1 for e in dec)

    # decode slices: per (sequence, head) the slices partition its pages
    seen = {}
    for e in dec:
        s, g, piece = e[0] & 0x3fffffff, e[4] & 0xff, e[4] >> 8
        assert e[1] == qsl[s] and e[2] == ctxs[s] and qsl[s + 1] - qsl[s] == 1
        seen.setdefault((s, g), {})[piece] = (e[5], e[6], e[3])
    dec_seqs = [s for s in range(len(ctxs)) if qsl[s + 1] - qsl[s] == 1]
    assert set(seen) == {(s, g) for s in dec_seqs for g in range(Hkv)}
    for (s, g), pieces in seen.items():
        k = next(iter(pieces.values()))[2]
        assert sorted(pieces) == list(range(k))
        edges = [pieces[i][:2] for i in range(k)]
        assert edges[0][0] == 0 and edges[-1][1] == math.ceil(ctxs[s] / 16)
        assert all(edges[i][1] == edges[i + 1][0] for i in range(k - 1))
        assert all(b > a for a, b in edges)
    # longest first: the size class of a segment's slices (its longest slice
    # in 8-page blocks) never grows along the queue, and no slice is longer
    # than the step's pages per slice
    def size_class(e):
        n = math.ceil(e[2] / 16)
        return min(math.ceil(math.ceil(n / e[3]) / 8), 255)
    classes = [size_class(e) for e in dec]
    assert all(classes[i] >= classes[i + 1] for i in range(len(classes) - 1))
    assert all(0 < e[6] - e[5] <= P for e in dec) and P >= 16 and P % 8 == 0

    # chunk units: every unit of every tile pair of every head, once
    units = {}
    for k_, e in enumerate(chunk):
        s, g, mp = e[0] & 0x3fffffff, e[4] & 0xff, e[4] >> 8
        u, nu = e[5] & 0xffff, e[5] >> 16
        assert e[6] == k_ and e[7] == k_ - u
        assert e[1] == qsl[s] and e[2] == ctxs[s] and e[3] == qsl[s + 1] - qsl[s]
        units.setdefault((s, g, mp), []).append((u, nu))
    pairs = {(s, g, mp) for s in range(len(ctxs)) if qsl[s + 1] - qsl[s] > 1
             for g in range(Hkv)
             for mp in range((math.ceil((qsl[s + 1] - qsl[s]) * G / 128) + 1) // 2)}
    assert set(units) == pairs
    for us in units.values():
        nu = us[0][1]
        assert all(n == nu for _, n in us) and sorted(u for u, _ in us) == list(range(nu))
    # later tile pairs (more keys) come first
    mps = [e[4] >> 8 for e in chunk]
    assert all(mps[i] >= mps[i + 1] for i in range(len(mps) - 1) if chunk[i][0] == chunk[i + 1][0])
