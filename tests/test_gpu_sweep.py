"""The budget-sweep workload on the GPU against the fp64 oracle.

An 8192-token prompt is prefilled from scratch beside 32 running decodes under
a token budget: decode-first composition gives each step budget - 32 prompt
tokens ("Chunked Prefill" (deepconcepts.dev), "The budget points in two
directions": the simulated sweep over budgets 256 .. 16384).  Every step runs
through the fused call, in order, so each chunk attends to the earlier chunks
through the paged cache; the last step of each budget (the longest context)
is compared with the oracle on every row and head, and the free-ride grid's
largest chunk on its own step.
"""
import pytest
import torch

from chunked_prefill_paged_cpa_gb300 import ops, workloads
from test_gpu_parity import check_step_against_oracle

pytestmark = pytest.mark.gpu


def _fused(ws, inp):
    sh = ws.sc.shape
    m = inp["meta"]
    wsp = ops.workspace_for(ws.k_cache, sh.num_q_heads, m.block_table.shape[1], m.num_seqs, m.num_tokens)
    out = ops.append_attention_forward(inp["q"], inp["k"], inp["v"], m.slot_mapping,
                                       ws.k_cache, ws.v_cache, m.block_table,
                                       m.query_start_loc, m.seq_lens, sh.scale, wsp)
    torch.cuda.synchronize()
    assert ops.device_status(ws.k_cache, sh.num_q_heads, m.block_table.shape[1], wsp) == 0
    return out


@pytest.mark.parametrize("budget", [256, 512, 2048, 16384])
def test_budget_sweep_last_step_matches_oracle(cuda_device, budget):
    sc = workloads.budget_sweep(budget)
    ws = workloads.WorkloadState(sc, device=cuda_device)
    for k in range(len(sc.plans)):
        inp = ws.step(k)
        out = _fused(ws, inp)
    chunk = [s for s in inp["plan"].seqs if s.kind == "prefill"]
    assert len(chunk) == 1 and chunk[0].seq_len == 8192
    check_step_against_oracle(f"budget {budget}, step {len(sc.plans)}", ws, inp, out)


@pytest.mark.parametrize("chunk", [0, 2048])
def test_free_ride_steps_match_oracle(cuda_device, chunk):
    sc = workloads.free_ride(chunk)
    ws = workloads.WorkloadState(sc, device=cuda_device)
    inp = ws.step(0)
    out = _fused(ws, inp)
    check_step_against_oracle(f"free ride, chunk {chunk}", ws, inp, out)
