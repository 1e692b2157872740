"""Test helpers: small hand-made steps and the oracle-side paged cache.

The oracle side never uses the package's slot arithmetic: it computes its own
slots (``oracle.slot_mapping``) from the block table and appends with
``oracle.kv_append``.  Inputs (per-position Q/K/V, page order, block table)
come from the shared seeded generator and page allocator.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from chunked_prefill_paged_cpa_gb300 import synth
from chunked_prefill_paged_cpa_gb300.batch import (PageAllocator, PagedSeqs,
                                                    build_metadata, pages_for)


class OracleCache:
    """Host paged caches built by the oracle's own append."""

    def __init__(self, num_pages, Hkv, page_size, D, dtype):
        shape = (num_pages, Hkv, page_size, D)
        self.k = torch.full(shape, float("nan"), dtype=dtype)
        self.v = torch.full(shape, float("nan"), dtype=dtype)
        self.page_size = page_size

    def append(self, block_table, q_lens, seq_lens, k_rows, v_rows):
        """Append rows for positions seq_len-q_len .. seq_len-1 of each seq."""
        qsl = torch.zeros(len(q_lens) + 1, dtype=torch.int32)
        qsl[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int32), 0)
        sl = torch.tensor(seq_lens, dtype=torch.int32)
        slots = oracle.slot_mapping(block_table, qsl, sl, self.page_size)
        oracle.kv_append(self.k, self.v, k_rows, v_rows, slots)
        return slots


def oracle_append(st, meta=None):
    """Append a ``make_step`` problem's new rows to its oracle cache through
    the oracle's own slots (``oracle.slot_mapping`` on the block table),
    checking on the way that the package's slot_mapping is the same bit for
    bit.  Returns the oracle's slots."""
    m = st["meta"] if meta is None else meta
    slots = oracle.slot_mapping(m.block_table, m.query_start_loc, m.seq_lens,
                                st["oracle_cache"].page_size)
    assert torch.equal(slots, m.slot_mapping.cpu()), "package slots differ from the oracle's"
    oracle.kv_append(st["oracle_cache"].k, st["oracle_cache"].v, st["k_new"], st["v_new"],
                     slots)
    return slots


def oracle_state_for(ws):
    """Oracle cache holding each sequence's prefix as ``ws`` (a
    WorkloadState) has it before its first step."""
    sh = ws.sc.shape
    oc = OracleCache(ws.num_pages, sh.num_kv_heads, sh.page_size, sh.head_dim, sh.dtype)
    seen = set()
    for k, plan in enumerate(ws.sc.plans):
        for s in plan.seqs:
            if s.rid in seen:
                continue
            seen.add(s.rid)
            pre = s.seq_len - s.q_len
            if pre == 0:
                continue
            pl = ws.paged.pages[s.rid]
            bt = torch.tensor([pl], dtype=torch.int32)
            kk, vv = ws.kv_rows(s.rid, torch.arange(pre))
            oc.append(bt, [pre], [pre], kk.cpu(), vv.cpu())
    return oc


def make_step(q_lens, seq_lens, Hq, Hkv, D, dtype, seed, page_size=16,
              pool_factor=1.5, device="cpu", transform=None):
    """A one-step problem on CPU: per-position Q/K/V from the generator, pages
    from a random permutation, the package's metadata, and the logical
    (unpaged) K/V of each sequence for the dense oracle.  ``transform(q,
    k_seqs, v_seqs)`` may return edited tensors before anything is derived
    from them (planted structure for special cases)."""
    st = synth.draw_sequences(seq_lens, [s - q for q, s in zip(q_lens, seq_lens)],
                              Hq, Hkv, D, dtype, seed)
    need = sum(pages_for(s, page_size) for s in seq_lens)
    pool = max(1, math.ceil(need * pool_factor))
    alloc = PageAllocator(synth.permutation(pool, seed + 7))
    paged = PagedSeqs(alloc, page_size)
    lists = [paged.ensure(i, s) for i, s in enumerate(seq_lens)]
    meta = build_metadata(q_lens, seq_lens, lists, page_size, pool)
    k_seqs = [st.k[o:o + L] for o, L in zip(st.kv_offsets, seq_lens)]
    v_seqs = [st.v[o:o + L] for o, L in zip(st.kv_offsets, seq_lens)]
    q = st.q
    if transform is not None:
        q, k_seqs, v_seqs = transform(q, k_seqs, v_seqs)
    new_k = torch.cat([ks[L - ql:] for ks, L, ql in zip(k_seqs, seq_lens, q_lens)])
    new_v = torch.cat([vs[L - ql:] for vs, L, ql in zip(v_seqs, seq_lens, q_lens)])
    # oracle-side cache: prefix via the oracle's own slots, then the new rows
    oc = OracleCache(pool, Hkv, page_size, D, dtype)
    pre = [L - ql for L, ql in zip(seq_lens, q_lens)]
    idx = [i for i, p in enumerate(pre) if p > 0]
    if idx:
        bt = meta.block_table[idx]
        oc.append(bt, [pre[i] for i in idx], [pre[i] for i in idx],
                  torch.cat([k_seqs[i][:pre[i]] for i in idx]),
                  torch.cat([v_seqs[i][:pre[i]] for i in idx]))
    return dict(q=q, k_new=new_k, v_new=new_v, meta=meta, k_seqs=k_seqs,
                v_seqs=v_seqs, oracle_cache=oc, pool=pool)


def to_np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()
