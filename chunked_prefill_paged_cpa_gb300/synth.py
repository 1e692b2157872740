"""Seeded synthetic inputs.

This module only draws random numbers.  It holds none of the attention or
paging arithmetic, imports neither the CUDA binding nor the oracle, and is the
one source of inputs that both sides of a parity test read.

Distributions follow the workloads being modelled: Q/K/V entries ~ N(0, 1)
(stored in the step's dtype), context lengths ~ U[lo, hi] integers, physical
pages in a uniformly random order.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


def uniform_lengths(n: int, lo: int, hi: int, seed: int) -> list[int]:
    """n integers drawn uniformly from [lo, hi] (inclusive)."""
    g = torch.Generator("cpu").manual_seed(seed)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


def permutation(n: int, seed: int) -> torch.Tensor:
    """A uniformly random permutation of 0..n-1 (int64, CPU)."""
    g = torch.Generator("cpu").manual_seed(seed)
    return torch.randperm(n, generator=g)


@dataclass
class SequenceTensors:
    """Per-position Q/K/V of a set of sequences, packed sequence after sequence.

    Sequence s owns K/V rows kv_offsets[s] .. kv_offsets[s] + lengths[s] - 1
    (one row per token position) and Q rows for positions q_from[s] ..
    lengths[s] - 1 starting at q_offsets[s] (queries are only drawn where some
    step will need them)."""
    lengths: list[int]
    q_from: list[int]
    q: torch.Tensor          # [sum(lengths - q_from), Hq, D]
    k: torch.Tensor          # [sum(lengths), Hkv, D]
    v: torch.Tensor          # [sum(lengths), Hkv, D]
    q_offsets: list[int]
    kv_offsets: list[int]


def draw_sequences(lengths, q_from, num_q_heads: int, num_kv_heads: int,
                   head_dim: int, dtype: torch.dtype, seed: int,
                   device="cpu") -> SequenceTensors:
    """Draw N(0,1) Q/K/V for every needed position, in a fixed order (K, V, Q)
    from one generator on ``device``, then round to ``dtype``."""
    lengths = [int(x) for x in lengths]
    q_from = [int(x) for x in q_from]
    n_kv = sum(lengths)
    n_q = sum(L - f for L, f in zip(lengths, q_from))
    g = torch.Generator(device).manual_seed(seed)

    def draw(rows, heads):
        return torch.randn(rows, heads, head_dim, generator=g, device=device,
                           dtype=torch.float32).to(dtype)

    k = draw(n_kv, num_kv_heads)
    v = draw(n_kv, num_kv_heads)
    q = draw(n_q, num_q_heads)
    kv_off, q_off, a, b = [], [], 0, 0
    for L, f in zip(lengths, q_from):
        kv_off.append(a)
        q_off.append(b)
        a += L
        b += L - f
    return SequenceTensors(lengths, q_from, q, k, v, q_off, kv_off)
