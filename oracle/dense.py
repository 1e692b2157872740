"""Brute-force dense oracle (test infrastructure; see the package docstring).

It never reads a page.  Each sequence's K/V are given as one contiguous
[ctx, Hkv, D] array in logical order; the visibility of query row i to key j
is written out as an explicit [q_len, ctx] boolean matrix, and the softmax is
scipy's.  It is meant for small inputs only.

Visibility ("vllm-learning-book 05. Chunked Prefill", section 3; "Chunked
Prefill 技术深度解析", section 4.1): the q_len new tokens are the last q_len
positions of the ctx-token sequence, so row i sits at position ctx-q_len+i and
sees every key at a position not after its own.
"""
from __future__ import annotations

import numpy as np
from scipy.special import softmax


def visibility(q_len: int, ctx: int) -> np.ndarray:
    """[q_len, ctx] matrix: True where query row i may attend to key j."""
    pos_q = np.arange(ctx - q_len, ctx)[:, None]   # absolute position of row i
    pos_k = np.arange(ctx)[None, :]
    return pos_k <= pos_q


def attention_dense(q: np.ndarray, k_seqs: list, v_seqs: list, q_lens: list,
                    scale: float) -> np.ndarray:
    """q: [T, Hq, D] (packed, sequences in order); k_seqs[s], v_seqs[s]:
    [ctx_s, Hkv, D].  Returns [T, Hq, D] float64."""
    q = np.asarray(q, dtype=np.float64)
    T, Hq, D = q.shape
    out = np.zeros((T, Hq, D), dtype=np.float64)
    start = 0
    for s, q_len in enumerate(q_lens):
        K = np.asarray(k_seqs[s], dtype=np.float64)
        V = np.asarray(v_seqs[s], dtype=np.float64)
        ctx, Hkv, _ = K.shape
        group = Hq // Hkv
        mask = visibility(q_len, ctx)
        for h in range(Hq):
            g = h // group
            Qh = q[start:start + q_len, h, :]                  # [q_len, D]
            logits = scale * (Qh @ K[:, g, :].T)               # [q_len, ctx]
            logits = np.where(mask, logits, -np.inf)
            P = softmax(logits, axis=1)
            out[start:start + q_len, h, :] = P @ V[:, g, :]
        start += q_len
    return out
