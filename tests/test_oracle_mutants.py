"""The oracle's pins have teeth: each plausible mistake planted in a copy of
the oracle's C source (compiled on the CPU, never the real oracle) must make at
least one pin fail."""
import numpy as np
import pytest
import torch

import oracle
from oracle.dense import attention_dense
from support import make_step, to_np64

MUTANTS = {
    "mask sees one key fewer": ("int64_t last = ctx - q_len + i;",
                                "int64_t last = ctx - q_len + i - (i > 0);"),
    "mask sees one future key": ("int64_t last = ctx - q_len + i;",
                                 "int64_t last = ctx - q_len + i + (i + 1 < q_len);"),
    "mask aligned top-left": ("int64_t last = ctx - q_len + i;",
                              "int64_t last = i < ctx ? i : ctx - 1;"),
    "GQA interleaved heads": ("int g = h / (P->Hq / P->Hkv);", "int g = h % P->Hkv;"),
    "page offset uses page index": ("int64_t off = j % page_size;",
                                    "int64_t off = (j / page_size) % page_size;"),
    "block table row ignored": ("block_table[(int64_t)s * max_pages + j / page_size]",
                                "block_table[j / page_size]"),
    "scale dropped": ("x[j] = P->scale * dot;", "x[j] = dot;"),
    "softmax not normalised": ("double p = x[j] / z;", "double p = x[j];"),
    "softmax exponent sign flipped": ("x[j] = exp(x[j] - mx);", "x[j] = exp(mx - x[j]);"),
    "dot product skips last dim": ("for (int d = 0; d < D; ++d)\n      dot +=",
                                   "for (int d = 0; d < D - 1; ++d)\n      dot +="),
    "append swaps k and v": ("memcpy((char *)k_cache + dst, (const char *)k + src, row);",
                             "memcpy((char *)k_cache + dst, (const char *)v + src, row);"),
    "slot of new token off by one": ("int64_t pos = ctx - q_len + i;",
                                     "int64_t pos = ctx - q_len + i + 1;"),
}


def _pins_hold(impl) -> bool:
    """Run a reduced set of the oracle pins against ``impl``; False if any
    fails or errors."""
    try:
        # 1. causal prefill vs torch SDPA, through the variant's own append
        g = torch.Generator().manual_seed(2)
        L, Hq, Hkv, D = 37, 4, 2, 16
        q = torch.randn(L, Hq, D, generator=g)
        k = torch.randn(L, Hkv, D, generator=g)
        v = torch.randn(L, Hkv, D, generator=g)
        n = -(-L // 16)
        bt = torch.randperm(n + 2, generator=g)[:n].to(torch.int32).view(1, n)
        kc = torch.zeros(n + 2, Hkv, 16, D)
        vc = torch.zeros(n + 2, Hkv, 16, D)
        qsl = torch.tensor([0, L], dtype=torch.int32)
        sl = torch.tensor([L], dtype=torch.int32)
        slots = oracle.slot_mapping(bt, qsl, sl, 16, impl=impl)
        oracle.kv_append(kc, vc, k, v, slots, impl=impl)
        out = oracle.attention(q, kc, vc, bt, qsl, sl, 0.25, impl=impl)
        G = Hq // Hkv
        ref = torch.nn.functional.scaled_dot_product_attention(
            q.double().permute(1, 0, 2)[None],
            k.double().repeat_interleave(G, 1).permute(1, 0, 2)[None],
            v.double().repeat_interleave(G, 1).permute(1, 0, 2)[None],
            is_causal=True, scale=0.25)[0].permute(1, 0, 2).numpy()
        if not np.allclose(out, ref, rtol=0, atol=1e-10):
            return False
        # 2. hybrid batches vs the dense brute force (own slots, own append)
        for seed in (1, 2, 3):
            st = make_step([1, 20, 1, 7], [30, 45, 17, 7], 4, 2, 16, torch.float32,
                           seed + 40)
            m = st["meta"]
            kc = torch.zeros_like(st["oracle_cache"].k)
            vc = torch.zeros_like(kc)
            allq = torch.tensor([0] + list(np.cumsum(m.seq_lens_list)), dtype=torch.int32)
            full = oracle.slot_mapping(m.block_table, allq, m.seq_lens, 16, impl=impl)
            oracle.kv_append(kc, vc, torch.cat(st["k_seqs"]), torch.cat(st["v_seqs"]),
                             full, impl=impl)
            out = oracle.attention(st["q"], kc, vc, m.block_table, m.query_start_loc,
                                   m.seq_lens, 0.25, impl=impl)
            ref = attention_dense(to_np64(st["q"]), [to_np64(x) for x in st["k_seqs"]],
                                  [to_np64(x) for x in st["v_seqs"]], m.q_lens, 0.25)
            if not np.allclose(out, ref, rtol=0, atol=1e-10):
                return False
        # 3. the package's slots must agree with the variant's slots
        if not torch.equal(oracle.slot_mapping(m.block_table, m.query_start_loc,
                                               m.seq_lens, 16, impl=impl), m.slot_mapping):
            return False
        return True
    except (ValueError, AssertionError, IndexError, RuntimeError):
        return False


def test_reference_source_passes_the_battery(tmp_path):
    impl = oracle.compile_variant(oracle.source_text(), str(tmp_path / "orig.so"))
    assert _pins_hold(impl)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = oracle.source_text()
    assert src.count(before) >= 1, f"mutation anchor missing: {before!r}"
    impl = oracle.compile_variant(src.replace(before, after, 1),
                                  str(tmp_path / "mutant.so"))
    assert not _pins_hold(impl), f"pins did not catch: {name}"
