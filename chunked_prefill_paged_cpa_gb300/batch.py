"""Packed-batch metadata and the page allocator (host side).

* Packed 1-D token layout ("vllm-learning-book 05. Chunked Prefill", section
  4): every scheduled sequence's tokens are concatenated into one [T] axis with
  no padding; ``query_start_loc`` (int32 [S+1], prefix sum of q_len) and
  ``seq_lens`` (int32 [S], tokens in the cache once this step's K/V are
  appended) tell the sequences apart.
* Paged cache ("Chunked Prefill 技术深度解析", section 4.2): pages of 16 tokens;
  a request holds a list of pages (``block_table`` row) and a chunk only
  appends pages, ``ceil(len / 16)`` in total.
* ``slot_mapping`` (int64 [T]): cache slot page * page_size + offset of each
  new token, consumed by ``cpa_kv_append``.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


def pages_for(num_tokens: int, page_size: int) -> int:
    return -(-int(num_tokens) // page_size)


class PageAllocator:
    """Hands out physical pages in a given (normally random) order.  The pool
    holds ``len(order)`` pages; pages are never freed within a workload."""

    def __init__(self, order: torch.Tensor):
        self.order = [int(x) for x in order.tolist()]
        self.next = 0

    @property
    def num_pages(self) -> int:
        return len(self.order)

    def allocate(self, n: int) -> list[int]:
        if self.next + n > len(self.order):
            raise MemoryError(f"page pool exhausted ({len(self.order)} pages)")
        out = self.order[self.next:self.next + n]
        self.next += n
        return out


class PagedSeqs:
    """Page lists of a set of sequences, grown as their contexts grow."""

    def __init__(self, allocator: PageAllocator, page_size: int = 16):
        self.alloc = allocator
        self.page_size = page_size
        self.pages: dict[object, list[int]] = {}

    def ensure(self, key, num_tokens: int) -> list[int]:
        have = self.pages.setdefault(key, [])
        need = pages_for(num_tokens, self.page_size) - len(have)
        if need > 0:
            have.extend(self.alloc.allocate(need))
        return have


@dataclass
class StepMetadata:
    q_lens: list[int]
    seq_lens_list: list[int]
    query_start_loc: torch.Tensor   # int32 [S+1]
    seq_lens: torch.Tensor          # int32 [S]
    block_table: torch.Tensor       # int32 [S, max_pages]
    slot_mapping: torch.Tensor      # int64 [T]
    page_size: int
    num_pages: int

    @property
    def num_seqs(self) -> int:
        return len(self.q_lens)

    @property
    def num_tokens(self) -> int:
        return int(sum(self.q_lens))

    def to(self, device) -> "StepMetadata":
        return StepMetadata(self.q_lens, self.seq_lens_list,
                            self.query_start_loc.to(device), self.seq_lens.to(device),
                            self.block_table.to(device), self.slot_mapping.to(device),
                            self.page_size, self.num_pages)


def build_metadata(q_lens, seq_lens, page_lists, page_size: int, num_pages: int,
                   max_pages: int | None = None) -> StepMetadata:
    """Host metadata of one step.  ``page_lists[s]`` is sequence s's page list
    (at least ceil(seq_lens[s] / page_size) pages)."""
    S = len(q_lens)
    if S != len(seq_lens) or S != len(page_lists):
        raise ValueError("q_lens, seq_lens and page_lists differ in length")
    for ql, sl, pl in zip(q_lens, seq_lens, page_lists):
        if ql < 1 or sl < ql:
            raise ValueError(f"need seq_len >= q_len >= 1, got q_len={ql}, seq_len={sl}")
        if len(pl) < pages_for(sl, page_size):
            raise ValueError("page list shorter than the context")
    need = max(pages_for(sl, page_size) for sl in seq_lens)
    if max_pages is None:
        max_pages = need
    if max_pages < need:
        raise ValueError("max_pages below the longest context")
    qsl = torch.zeros(S + 1, dtype=torch.int32)
    qsl[1:] = torch.cumsum(torch.tensor(q_lens, dtype=torch.int32), 0)
    bt = torch.zeros(S, max_pages, dtype=torch.int32)
    slots = []
    for s, (ql, sl, pl) in enumerate(zip(q_lens, seq_lens, page_lists)):
        n = pages_for(sl, page_size)
        bt[s, :n] = torch.tensor(pl[:n], dtype=torch.int32)
        pos = torch.arange(sl - ql, sl, dtype=torch.int64)
        pages = torch.tensor(pl[:n], dtype=torch.int64)[pos // page_size]
        slots.append(pages * page_size + pos % page_size)
    return StepMetadata(list(map(int, q_lens)), list(map(int, seq_lens)), qsl,
                        torch.tensor(seq_lens, dtype=torch.int32), bt,
                        torch.cat(slots), page_size, num_pages)


def position_slots(page_list, positions: torch.Tensor, page_size: int):
    """(page, offset) of logical positions of one sequence."""
    pages = torch.tensor(page_list, dtype=torch.int64)[positions // page_size]
    return pages, positions % page_size


def write_positions(k_cache: torch.Tensor, v_cache: torch.Tensor, page_list,
                    positions: torch.Tensor, k_rows: torch.Tensor,
                    v_rows: torch.Tensor) -> None:
    """Place already-computed K/V rows of one sequence at their cache positions
    (state preparation: the prefix a step finds in the cache).  Caches are
    [num_pages, Hkv, page_size, D]; rows are [n, Hkv, D]."""
    page_size = k_cache.shape[2]
    pages, offs = position_slots(page_list, positions.cpu(), page_size)
    pages, offs = pages.to(k_cache.device), offs.to(k_cache.device)
    k_cache[pages, :, offs, :] = k_rows.to(k_cache.device, k_cache.dtype)
    v_cache[pages, :, offs, :] = v_rows.to(v_cache.device, v_cache.dtype)
