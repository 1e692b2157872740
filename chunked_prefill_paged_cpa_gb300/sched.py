"""Decode-first token-budget scheduler step (host side, composes workloads).

Policy, as the pages describe it:

* "vllm-learning-book 05. Chunked Prefill", section 5.2 (decode-first, the V1
  default): every running request first gets one decode token, which uses
  |running| of the budget B; the remaining B - |running| goes to prefill, either
  new requests or the continuation of a chunked one.
* "Chunked Prefill" (deepconcepts.dev), "The budget points in two directions":
  a budget below the number of running users leaves no room for any prompt and
  is rejected up front (max_num_batched_tokens >= max_num_seqs).
* same page, "Checking it on a real system": the remaining budget is filled
  with prefill; ``long_prefill_token_threshold`` caps one request's share of a
  single pass.

Where "Chunked Prefill 技术深度解析" section 3.1 stops at the first prefill that
does not fit whole, this scheduler instead gives that request a chunk of
whatever budget remains (the fill reading of the two pages above).

The scheduler only decides per-sequence (q_len, seq_len); it is never timed.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass
class Request:
    """A request's cache state.  ``cached`` counts tokens already in the KV
    cache; ``prompt_len`` is the prompt length."""
    rid: str
    prompt_len: int
    cached: int = 0

    @property
    def prefill_done(self) -> bool:
        return self.cached >= self.prompt_len


@dataclass
class ScheduledSeq:
    rid: str
    q_len: int        # tokens fed through this pass
    seq_len: int      # tokens in the cache once this pass appended its K/V
    kind: str         # "decode" or "prefill"


@dataclass
class StepPlan:
    seqs: list[ScheduledSeq] = field(default_factory=list)
    budget: int = 0

    @property
    def num_tokens(self) -> int:
        return sum(s.q_len for s in self.seqs)

    @property
    def q_lens(self) -> list[int]:
        return [s.q_len for s in self.seqs]

    @property
    def seq_lens(self) -> list[int]:
        return [s.seq_len for s in self.seqs]

    def as_dict(self) -> dict:
        return {s.rid: s.q_len for s in self.seqs}


class BudgetError(ValueError):
    """The token budget cannot give every running request its decode token."""


def schedule_step(running: list[Request], waiting: list[Request], budget: int,
                  long_prefill_token_threshold: int | None = None) -> StepPlan:
    """One decode-first pass.  ``running`` requests decode one token each (in
    order); ``waiting`` requests (prompt not yet fully cached, in arrival
    order) share what is left of the budget, first come first served."""
    if budget < len(running):
        raise BudgetError(
            f"token budget {budget} is below the {len(running)} running requests: "
            "no prefill could ever be scheduled")
    plan = StepPlan(budget=budget)
    for r in running:
        plan.seqs.append(ScheduledSeq(r.rid, 1, r.cached + 1, "decode"))
    remaining = budget - len(running)
    for r in waiting:
        if remaining <= 0:
            break
        chunk = min(r.prompt_len - r.cached, remaining)
        if long_prefill_token_threshold is not None:
            chunk = min(chunk, long_prefill_token_threshold)
        if chunk <= 0:
            continue
        plan.seqs.append(ScheduledSeq(r.rid, chunk, r.cached + chunk, "prefill"))
        remaining -= chunk
    return plan


def commit(plan: StepPlan, running: list[Request], waiting: list[Request]) -> None:
    """Advance request state after the pass ran.  A request whose prompt is now
    fully cached moves from ``waiting`` to the end of ``running`` (its first
    output token was sampled from this pass's last row)."""
    by_id = {r.rid: r for r in running + waiting}
    for s in plan.seqs:
        by_id[s.rid].cached = s.seq_len
    done = [r for r in waiting if r.prefill_done]
    for r in done:
        waiting.remove(r)
        running.append(r)


def prompt_chunks(n_running: int, prompt_len: int, budget: int,
                  long_prefill_token_threshold: int | None = None) -> list[int]:
    """Chunk sizes one new prompt is cut into while ``n_running`` other users
    keep decoding (the scenario of deepconcepts.dev's simulation)."""
    running = [Request(f"u{i}", 1, 1) for i in range(n_running)]
    waiting = [Request("prompt", prompt_len, 0)]
    chunks = []
    while waiting:
        plan = schedule_step(running, waiting, budget, long_prefill_token_threshold)
        chunk = [s.q_len for s in plan.seqs if s.rid == "prompt"]
        if not chunk:
            raise BudgetError("no progress")
        chunks.append(chunk[0])
        commit(plan, running, waiting)
        running = [r for r in running if r.rid != "prompt"]
    return chunks
