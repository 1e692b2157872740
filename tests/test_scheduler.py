"""Decode-first token-budget scheduler against the pages' own numbers."""
import json
import os

import pytest

from chunked_prefill_paged_cpa_gb300.sched import (BudgetError, Request, commit,
                                                    prompt_chunks, schedule_step)
from chunked_prefill_paged_cpa_gb300 import workloads

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_budget_sweep_pass_counts():
    g = load("budget_sweep.json")
    users, prompt = g["scenario"]["running_users"], g["scenario"]["prompt_tokens"]
    for budget, passes in g["passes_by_budget"].items():
        chunks = prompt_chunks(users, prompt, int(budget))
        assert len(chunks) == passes, (budget, chunks)
        assert sum(chunks) == prompt


def test_budget_sweep_chunk_sizes():
    g = load("budget_sweep.json")
    users, prompt = g["scenario"]["running_users"], g["scenario"]["prompt_tokens"]
    for budget, chunk in g["chunk_tokens_by_budget"].items():
        assert prompt_chunks(users, prompt, int(budget))[0] == chunk


def test_budget_below_running_is_rejected():
    g = load("budget_sweep.json")["rejected_budget"]
    running = [Request(f"u{i}", 1, 1) for i in range(g["running_users"])]
    with pytest.raises(BudgetError):
        schedule_step(running, [Request("p", 8192)], g["budget"])


def test_packed_batch_example():
    g = load("packed_batch.json")
    running = [Request(r, 10, 10) for r in g["running"]]
    waiting = [Request(w["rid"], w["prompt_tokens"]) for w in g["waiting"]]
    plan = schedule_step(running, waiting, g["budget"])
    assert plan.as_dict() == g["expected"]
    assert plan.num_tokens == g["total"]


def test_threshold_caps_one_request():
    running = [Request("a", 5, 5)]
    waiting = [Request("p", 1000), Request("q", 1000)]
    plan = schedule_step(running, waiting, 512, long_prefill_token_threshold=100)
    assert plan.as_dict() == {"a": 1, "p": 100, "q": 100}


def test_fill_gives_remaining_budget_to_next_prompt():
    # the fill reading: a prompt that does not fit whole still gets a chunk
    running = [Request("a", 5, 5)]
    waiting = [Request("p", 300), Request("q", 1000)]
    plan = schedule_step(running, waiting, 512)
    assert plan.as_dict() == {"a": 1, "p": 300, "q": 211}


def test_commit_moves_finished_prompt_to_running():
    running = [Request("a", 5, 5)]
    waiting = [Request("p", 64)]
    plan = schedule_step(running, waiting, 65)
    assert plan.as_dict() == {"a": 1, "p": 64}
    commit(plan, running, waiting)
    assert [r.rid for r in running] == ["a", "p"] and not waiting
    plan2 = schedule_step(running, waiting, 65)
    assert [(s.rid, s.q_len, s.seq_len) for s in plan2.seqs] == [("a", 1, 7), ("p", 1, 65)]


def test_tiny_scenario_steps():
    sc = workloads.scenario("tiny")
    got = [[(s.rid, s.q_len, s.seq_len) for s in p.seqs] for p in sc.plans]
    assert got == [
        [("B", 1, 41), ("A", 32, 32)],
        [("B", 1, 42), ("A", 32, 64)],
        [("B", 1, 43), ("A", 32, 96)],
        [("B", 1, 44), ("A", 1, 97)],
    ]


@pytest.mark.parametrize("name,decodes,chunk,ctx,lo,hi", [
    ("page1_default", 32, 480, 4320, 512, 4096),
    ("large_budget", 4, 2048, 8192, 1024, 8192),
    ("long_context", 64, 512, 32256, 2048, 16384),
    ("decode_only", 256, None, None, 2048, 8192),
])
def test_named_scenarios(name, decodes, chunk, ctx, lo, hi):
    sc = workloads.scenario(name)
    assert len(sc.plans) == 1
    seqs = sc.plans[0].seqs
    dec = [s for s in seqs if s.kind == "decode"]
    pre = [s for s in seqs if s.kind == "prefill"]
    assert len(dec) == decodes
    assert all(s.q_len == 1 and lo <= s.seq_len <= hi for s in dec)
    if chunk is None:
        assert not pre
    else:
        assert [(s.q_len, s.seq_len) for s in pre] == [(chunk, ctx)]
        # offsets are whole numbers of chunks: 3840 = 8*480, 6144 = 3*2048,
        # 31744 = 62*512
        assert (ctx - chunk) % chunk == 0


def test_chunked_scenario_covers_prompt():
    sc = workloads.scenario("large_budget_chunked")
    chunks = [[s for s in p.seqs if s.rid == "P"] for p in sc.plans]
    assert [(c[0].q_len, c[0].seq_len) for c in chunks] == [
        (2048, 2048), (2048, 4096), (2048, 6144), (2048, 8192)]


def test_budget_sweep_scenarios_cover_the_prompt():
    from chunked_prefill_paged_cpa_gb300 import workloads
    for budget, steps in ((256, 37), (512, 18), (2048, 5), (16384, 1)):
        sc = workloads.budget_sweep(budget)
        assert len(sc.plans) == steps
        chunks = [s.q_len for p in sc.plans for s in p.seqs if s.rid == "P"]
        assert sum(chunks) == 8192
        # decode-first: every step carries the 32 decodes and a chunk of the rest
        for p in sc.plans:
            assert sum(1 for s in p.seqs if s.rid != "P") == 32
            assert sum(s.q_len for s in p.seqs) <= budget
    with pytest.raises(Exception):
        workloads.budget_sweep(32)
