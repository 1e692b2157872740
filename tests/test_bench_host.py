"""bench.py's host-side parts, on CPU: the algorithmic counts behind every
roofline fraction, against an enumeration of the visible (query, key) pairs,
and the reference arm's JSON line (the oracle on the host cores) on the tiny
workload.

A chunk row i of a sequence with q_len new tokens and ctx keys sees keys
0 .. ctx - q_len + i ("vllm-learning-book 05. Chunked Prefill", section 3); a
pair costs QK^T and PV, 2 * D multiply-adds per query head.
"""
import json
import os
import random
import subprocess
import sys

import bench
from chunked_prefill_paged_cpa_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_step_counts_match_enumeration():
    rng = random.Random(5)
    for _ in range(25):
        n = rng.randint(1, 6)
        q_lens = [1 if rng.random() < 0.5 else rng.randint(2, 40) for _ in range(n)]
        seq_lens = [ql + rng.randint(0, 100) for ql in q_lens]
        Hq, Hkv, D = 8, 2, 64
        c = bench.step_counts(q_lens, seq_lens, Hq, Hkv, D, 2)
        pairs = sum(1 for ql, sl in zip(q_lens, seq_lens) for i in range(ql)
                    for k in range(sl) if k <= sl - ql + i)
        assert c["pairs"] == pairs
        assert c["flops"] == 2 * 2 * D * Hq * pairs
        # K and V of every cached key once (bf16), Q read and O written once
        assert c["kv_bytes"] == sum(seq_lens) * Hkv * D * 2 * 2
        assert c["bytes"] == c["kv_bytes"] + sum(q_lens) * Hq * D * 2 * 2
        # an 8-bit cache halves the KV bytes only
        c8 = bench.step_counts(q_lens, seq_lens, Hq, Hkv, D, 2, 1)
        assert c8["kv_bytes"] * 2 == c["kv_bytes"] and c8["flops"] == c["flops"]


def test_page1_default_counts():
    """The default hybrid step: 82,734 keys over 33 sequences and 512 query
    tokens at the Llama-3-8B attention shape: 4,096 B per key (K and V, 8 kv
    heads, 128 dims, bf16) and 16,384 B per query token (Q and O, 32 heads)."""
    sc = workloads.scenario("page1_default")
    q_lens = [s.q_len for s in sc.plans[0].seqs]
    seq_lens = [s.seq_len for s in sc.plans[0].seqs]
    assert (sum(seq_lens), sum(q_lens)) == (82734, 512)
    c = bench.step_counts(q_lens, seq_lens, 32, 8, 128, 2)
    assert c["bytes"] == 82734 * 4096 + 512 * 16384 == 347_267_072


def test_reference_arm_line_on_tiny():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "tiny",
                        "--steps", "1", "--warmup", "3", "--ref-budget", "0.5"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["dtype"] == "f64"
    assert line["unit"] == "tokens/s" and line["value"] > 0 and line["higher_is_better"] is True
    assert line["steps"] == 1 and line["warmup"] >= 3 and line["n_gpus"] == 1
    assert line["config"]["workload"] == "tiny" and line["config"]["query_tokens"] == 33
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s",
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
