"""Packed metadata, page allocation and slot addressing (host side)."""
import json
import os

import pytest
import torch

import oracle
from chunked_prefill_paged_cpa_gb300 import synth
from chunked_prefill_paged_cpa_gb300.batch import (PageAllocator, PagedSeqs,
                                                    build_metadata, pages_for)

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_page_count_example():
    with open(os.path.join(GOLD, "page_count.json")) as f:
        g = json.load(f)
    assert pages_for(g["tokens"], g["page_size"]) == g["pages"]
    alloc = PageAllocator(torch.arange(1000))
    seqs = PagedSeqs(alloc, g["page_size"])
    # chunked allocation: 1024-token chunks only ever append pages
    got = []
    for end in (1024, 2048, 2500):
        got.append(len(seqs.ensure("r", end)))
    assert got == [64, 128, g["pages"]]


def test_allocator_exhaustion():
    alloc = PageAllocator(torch.arange(3))
    alloc.allocate(2)
    with pytest.raises(MemoryError):
        alloc.allocate(2)


@pytest.mark.parametrize("seed", range(5))
def test_metadata_layout_and_slots_match_oracle(seed):
    g = torch.Generator().manual_seed(seed)
    S = int(torch.randint(1, 9, (1,), generator=g))
    q_lens, seq_lens = [], []
    for _ in range(S):
        ql = int(torch.randint(1, 70, (1,), generator=g))
        pre = int(torch.randint(0, 90, (1,), generator=g))
        q_lens.append(ql)
        seq_lens.append(ql + pre)
    need = sum(pages_for(s, 16) for s in seq_lens)
    alloc = PageAllocator(synth.permutation(need + 5, seed))
    paged = PagedSeqs(alloc, 16)
    lists = [paged.ensure(i, s) for i, s in enumerate(seq_lens)]
    meta = build_metadata(q_lens, seq_lens, lists, 16, need + 5)
    assert meta.query_start_loc.dtype == torch.int32
    assert meta.query_start_loc[0] == 0
    assert meta.query_start_loc.tolist()[1:] == torch.cumsum(torch.tensor(q_lens), 0).tolist()
    assert meta.seq_lens.tolist() == seq_lens
    assert meta.slot_mapping.dtype == torch.int64
    ref = oracle.slot_mapping(meta.block_table, meta.query_start_loc, meta.seq_lens, 16)
    assert torch.equal(meta.slot_mapping, ref)
    # every slot distinct and inside the pool
    assert len(set(meta.slot_mapping.tolist())) == meta.num_tokens
    assert int(meta.slot_mapping.max()) < (need + 5) * 16


def test_metadata_rejects_bad_lengths():
    with pytest.raises(ValueError):
        build_metadata([3], [2], [[0]], 16, 4)
    with pytest.raises(ValueError):
        build_metadata([0], [2], [[0]], 16, 4)
