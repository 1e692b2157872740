"""Pins of the fp64 oracle to things other than itself.

* hand-derived closed forms (tests/golden/hand_attention.json);
* torch's scaled_dot_product_attention (is_causal) for a prefill with nothing
  cached -- a library routine that defines causal attention;
* the brute-force dense oracle (explicit visibility matrix, scipy softmax, no
  pages) on small random hybrid batches;
* invariants the pages fix: chunked == one-shot ("vllm-learning-book 05.
  Chunked Prefill", section 3; "Chunked Prefill 技术深度解析", section 7.2
  recommends the check), a decode equals the last row of the prefill that
  contains it, softmax rows sum to 1;
* closed forms: q = 0 gives the mean of the visible V, one visible key gives
  that V, a planted key under a large scale wins the argmax;
* page-order invariance and the GQA head map.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.dense import attention_dense, visibility
from support import make_step, to_np64

GOLD = os.path.join(os.path.dirname(__file__), "golden")
SCALES = {"ln3": math.log(3.0), "ln2": math.log(2.0), "1": 1.0}


def _single_seq_cache(k, v, page_size=16, pool_extra=3, seed=0):
    """Put one sequence's logical K/V ([L, Hkv, D]) into a paged cache with a
    shuffled page order using the oracle's own slots."""
    L, Hkv, D = k.shape
    n = -(-L // page_size)
    perm = torch.randperm(n + pool_extra, generator=torch.Generator().manual_seed(seed))
    bt = perm[:n].to(torch.int32).view(1, n)
    kc = torch.full((n + pool_extra, Hkv, page_size, D), float("nan"), dtype=k.dtype)
    vc = kc.clone()
    qsl = torch.tensor([0, L], dtype=torch.int32)
    sl = torch.tensor([L], dtype=torch.int32)
    slots = oracle.slot_mapping(bt, qsl, sl, page_size)
    oracle.kv_append(kc, vc, k, v, slots)
    return kc, vc, bt


def test_hand_closed_forms():
    with open(os.path.join(GOLD, "hand_attention.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        q = torch.tensor(c["q"], dtype=torch.float32)[:, None, :]      # [q_len, 1, D]
        k = torch.tensor(c["k"], dtype=torch.float32)[:, None, :]      # [L, 1, D]
        v = torch.tensor(c["v"], dtype=torch.float32)[:, None, :]
        kc, vc, bt = _single_seq_cache(k, v)
        qsl = torch.tensor([0, c["q_len"]], dtype=torch.int32)
        sl = torch.tensor([c["seq_len"]], dtype=torch.int32)
        scale = SCALES[c["scale"]]
        out = oracle.attention(q, kc, vc, bt, qsl, sl, scale)
        np.testing.assert_allclose(out[:, 0, :], np.array(c["out"]), rtol=0, atol=1e-12,
                                   err_msg=c["name"])
        for row, want in enumerate(c["probs"]):
            p, _ = oracle.probs(q, kc, vc, bt, qsl, sl, scale, row, 0)
            np.testing.assert_allclose(p, want, rtol=0, atol=1e-15, err_msg=c["name"])


@pytest.mark.parametrize("L,Hq,Hkv,D", [(40, 4, 2, 16), (75, 8, 8, 32), (33, 6, 2, 64)])
def test_oneshot_prefill_matches_torch_sdpa(L, Hq, Hkv, D):
    g = torch.Generator().manual_seed(L * 7 + D)
    q = torch.randn(L, Hq, D, generator=g)
    k = torch.randn(L, Hkv, D, generator=g)
    v = torch.randn(L, Hkv, D, generator=g)
    kc, vc, bt = _single_seq_cache(k, v, seed=L)
    qsl = torch.tensor([0, L], dtype=torch.int32)
    sl = torch.tensor([L], dtype=torch.int32)
    scale = 1 / math.sqrt(D)
    out = oracle.attention(q, kc, vc, bt, qsl, sl, scale)
    G = Hq // Hkv
    qq = q.double().permute(1, 0, 2)[None]
    kk = k.double().repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    vv = v.double().repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, is_causal=True,
                                                           scale=scale)
    np.testing.assert_allclose(out, ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def _random_batch(seed, max_seqs=6, Hq=4, Hkv=2, D=32, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    S = int(torch.randint(1, max_seqs + 1, (1,), generator=g))
    q_lens, seq_lens = [], []
    for _ in range(S):
        ql = 1 if torch.rand(1, generator=g) < 0.5 else int(torch.randint(2, 40, (1,), generator=g))
        pre = int(torch.randint(0, 60, (1,), generator=g))
        q_lens.append(ql)
        seq_lens.append(ql + pre)
    return make_step(q_lens, seq_lens, Hq, Hkv, D, dtype, seed)


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_paged_oracle_matches_dense_bruteforce(seed, dtype):
    st = _random_batch(seed, dtype=dtype)
    m, oc = st["meta"], st["oracle_cache"]
    slots = oracle.slot_mapping(m.block_table, m.query_start_loc, m.seq_lens, 16)
    oracle.kv_append(oc.k, oc.v, st["k_new"], st["v_new"], slots)
    scale = 1 / math.sqrt(st["q"].shape[-1])
    out = oracle.attention(st["q"], oc.k, oc.v, m.block_table, m.query_start_loc,
                           m.seq_lens, scale)
    ref = attention_dense(to_np64(st["q"]), [to_np64(k) for k in st["k_seqs"]],
                          [to_np64(v) for v in st["v_seqs"]], m.q_lens, scale)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_visibility_matrix_shape():
    m = visibility(3, 5)
    assert m.tolist() == [[True, True, True, False, False],
                          [True, True, True, True, False],
                          [True, True, True, True, True]]


def _seq_problem(L, Hq=4, Hkv=2, D=16, seed=3):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(L, Hq, D, generator=g)
    k = torch.randn(L, Hkv, D, generator=g)
    v = torch.randn(L, Hkv, D, generator=g)
    kc, vc, bt = _single_seq_cache(k, v, seed=seed)
    return q, k, v, kc, vc, bt


def test_chunked_equals_oneshot():
    L, C = 96, 32
    q, k, v, kc, vc, bt = _seq_problem(L)
    scale = 0.25
    one = oracle.attention(q, kc, vc, bt, torch.tensor([0, L], dtype=torch.int32),
                           torch.tensor([L], dtype=torch.int32), scale)
    parts = []
    for c0 in range(0, L, C):
        # the chunk's step sees the cache up to its own end only
        qsl = torch.tensor([0, C], dtype=torch.int32)
        sl = torch.tensor([c0 + C], dtype=torch.int32)
        parts.append(oracle.attention(q[c0:c0 + C], kc, vc, bt, qsl, sl, scale))
    np.testing.assert_allclose(np.concatenate(parts), one, rtol=0, atol=1e-12)


def test_ragged_chunks_equal_oneshot():
    L = 77
    q, k, v, kc, vc, bt = _seq_problem(L, seed=5)
    scale = 0.3
    one = oracle.attention(q, kc, vc, bt, torch.tensor([0, L], dtype=torch.int32),
                           torch.tensor([L], dtype=torch.int32), scale)
    bounds = [0, 5, 6, 30, 64, 77]
    parts = []
    for a, b in zip(bounds[:-1], bounds[1:]):
        parts.append(oracle.attention(q[a:b], kc, vc, bt,
                                      torch.tensor([0, b - a], dtype=torch.int32),
                                      torch.tensor([b], dtype=torch.int32), scale))
    np.testing.assert_allclose(np.concatenate(parts), one, rtol=0, atol=1e-12)


def test_decode_equals_last_prefill_row():
    L = 50
    q, k, v, kc, vc, bt = _seq_problem(L, seed=9)
    scale = 0.2
    one = oracle.attention(q, kc, vc, bt, torch.tensor([0, L], dtype=torch.int32),
                           torch.tensor([L], dtype=torch.int32), scale)
    for p in (0, 17, L - 1):
        dec = oracle.attention(q[p:p + 1], kc, vc, bt, torch.tensor([0, 1], dtype=torch.int32),
                               torch.tensor([p + 1], dtype=torch.int32), scale)
        np.testing.assert_allclose(dec[0], one[p], rtol=0, atol=1e-12)


def test_softmax_rows_sum_to_one_and_ones_in_ones_out():
    st = _random_batch(11)
    m, oc = st["meta"], st["oracle_cache"]
    slots = oracle.slot_mapping(m.block_table, m.query_start_loc, m.seq_lens, 16)
    oracle.kv_append(oc.k, oc.v, st["k_new"], st["v_new"], slots)
    T, Hq, _ = st["q"].shape
    for t in range(0, T, max(1, T // 7)):
        for h in (0, Hq - 1):
            p, _ = oracle.probs(st["q"], oc.k, oc.v, m.block_table, m.query_start_loc,
                                m.seq_lens, 0.5, t, h)
            assert abs(p.sum() - 1.0) < 1e-12 and (p >= 0).all()
    # V == 1 everywhere it is read: every output is exactly 1 up to rounding
    ones = torch.ones_like(oc.v)
    out = oracle.attention(st["q"], oc.k, ones, m.block_table, m.query_start_loc,
                           m.seq_lens, 0.5)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-12)


def test_zero_query_gives_mean_of_visible_values():
    st = _random_batch(13)
    m, oc = st["meta"], st["oracle_cache"]
    slots = oracle.slot_mapping(m.block_table, m.query_start_loc, m.seq_lens, 16)
    oracle.kv_append(oc.k, oc.v, st["k_new"], st["v_new"], slots)
    q0 = torch.zeros_like(st["q"])
    out = oracle.attention(q0, oc.k, oc.v, m.block_table, m.query_start_loc,
                           m.seq_lens, 1.0)
    Hq, Hkv = st["q"].shape[1], st["k_new"].shape[1]
    t = 0
    for s, (ql, L) in enumerate(zip(m.q_lens, m.seq_lens_list)):
        V = to_np64(st["v_seqs"][s])
        for i in range(ql):
            n_vis = L - ql + i + 1
            for h in range(Hq):
                want = V[:n_vis, h // (Hq // Hkv), :].mean(axis=0)
                np.testing.assert_allclose(out[t, h], want, rtol=0, atol=1e-12)
            t += 1


def test_single_visible_key_and_planted_argmax():
    g = torch.Generator().manual_seed(1)
    D = 16
    k = torch.randn(40, 1, D, generator=g)
    v = torch.randn(40, 1, D, generator=g)
    kc, vc, bt = _single_seq_cache(k, v, seed=2)
    # first row of a chunk with nothing cached: only key 0 is visible
    q = torch.randn(40, 1, D, generator=g)
    out = oracle.attention(q, kc, vc, bt, torch.tensor([0, 40], dtype=torch.int32),
                           torch.tensor([40], dtype=torch.int32), 1.0)
    np.testing.assert_allclose(out[0, 0], to_np64(v[0, 0]), rtol=0, atol=1e-12)
    # a decode whose query is aligned with key 23 under a huge scale picks V_23
    qd = (k[23] * 1.0).view(1, 1, D)
    k2 = k.clone()
    k2[23] = k[23] * 4.0
    kc2, vc2, bt2 = _single_seq_cache(k2, v, seed=2)
    out = oracle.attention(qd, kc2, vc2, bt2, torch.tensor([0, 1], dtype=torch.int32),
                           torch.tensor([40], dtype=torch.int32), 50.0)
    np.testing.assert_allclose(out[0, 0], to_np64(v[23, 0]), rtol=0, atol=1e-9)


def test_page_order_does_not_change_the_result():
    g = torch.Generator().manual_seed(4)
    L, D = 70, 32
    q = torch.randn(L, 2, D, generator=g)
    k = torch.randn(L, 1, D, generator=g)
    v = torch.randn(L, 1, D, generator=g)
    qsl = torch.tensor([0, L], dtype=torch.int32)
    sl = torch.tensor([L], dtype=torch.int32)
    outs = []
    for seed in (0, 1, 2):
        kc, vc, bt = _single_seq_cache(k, v, seed=seed, pool_extra=seed * 4)
        outs.append(oracle.attention(q, kc, vc, bt, qsl, sl, 0.2))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_gqa_head_map_is_contiguous_groups():
    g = torch.Generator().manual_seed(6)
    L, D, Hq, Hkv = 30, 16, 8, 2
    q = torch.randn(L, Hq, D, generator=g)
    k = torch.randn(L, Hkv, D, generator=g)
    v = torch.randn(L, Hkv, D, generator=g)
    kc, vc, bt = _single_seq_cache(k, v, seed=1)
    qsl = torch.tensor([0, L], dtype=torch.int32)
    sl = torch.tensor([L], dtype=torch.int32)
    gqa = oracle.attention(q, kc, vc, bt, qsl, sl, 0.3)
    km = k.repeat_interleave(Hq // Hkv, dim=1)
    vm = v.repeat_interleave(Hq // Hkv, dim=1)
    kcm, vcm, btm = _single_seq_cache(km, vm, seed=1)
    mha = oracle.attention(q, kcm, vcm, btm, qsl, sl, 0.3)
    np.testing.assert_allclose(gqa, mha, rtol=0, atol=1e-13)


def test_kv_append_is_a_bitexact_scatter():
    g = torch.Generator().manual_seed(8)
    T, Hkv, D, P = 20, 2, 8, 6
    k = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    slots = torch.randperm(P * 16, generator=g)[:T].to(torch.int64)
    slots[3] = -1
    kc = torch.full((P, Hkv, 16, D), float("nan"), dtype=torch.bfloat16)
    vc = kc.clone()
    before = kc.clone()
    oracle.kv_append(kc, vc, k, v, slots)
    written = set()
    for t in range(T):
        s = int(slots[t])
        if s < 0:
            continue
        written.add(s)
        assert torch.equal(kc[s // 16, :, s % 16].view(torch.int16), k[t].view(torch.int16))
        assert torch.equal(vc[s // 16, :, s % 16].view(torch.int16), v[t].view(torch.int16))
    for s in range(P * 16):
        if s not in written:
            assert torch.equal(kc[s // 16, :, s % 16].view(torch.int16),
                               before[s // 16, :, s % 16].view(torch.int16))
