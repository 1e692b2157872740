#!/usr/bin/env python3
"""Benchmark of one hybrid-batch attention step (KV append + attention).

One step = the whole hot path over one packed hybrid batch in one C-ABI call,
``cpa_append_attention_forward``: the append of the step's new K/V into the
paged cache and the attention of every query token (the append fused into
the attention kernels where they take the shape).  The same step as the two
separate calls (``cpa_kv_append``, then ``cpa_attention_forward``) is timed
too, as a breakdown.
Default workload: the Llama-3-8B-shaped default step (32 decodes with context
~U[512, 4096] plus a 480-token chunk of an 8192-token prompt at offset 3840,
budget 512, bf16, 16-token pages).

Prints one JSON line.  ``value`` is query tokens per second with every input
resident in HBM (device time, CUDA events on the launching stream, L2 flushed
before each timed step).  ``e2e`` is the same metric through the same C-ABI
calls with host inputs: pinned host -> device copies of the step's inputs and
the device -> host copy of its output inside the timed region.

``--impl reference`` times the fp64 CPU oracle on the host cores instead (a
deliberately slow baseline, not a target).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "hybrid-batch attention step tokens/s"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def step_counts(q_lens, seq_lens, Hq, Hkv, D, elem_bytes, kv_elem_bytes=None):
    """Algorithmic work of one attention step: FLOPs over causally visible
    (query, key) pairs (QK^T and PV, 2 FLOPs per multiply-add each) and bytes
    (every sequence's K/V read once, Q read and O written once).  An 8-bit
    cache has kv_elem_bytes = 1."""
    kb = elem_bytes if kv_elem_bytes is None else kv_elem_bytes
    pairs = 0
    for ql, sl in zip(q_lens, seq_lens):
        pairs += ql * (sl - ql) + ql * (ql + 1) // 2
    flops = 4 * D * Hq * pairs
    kv_bytes = sum(seq_lens) * Hkv * D * kb * 2
    qo_bytes = sum(q_lens) * Hq * D * elem_bytes * 2
    append_bytes = sum(q_lens) * Hkv * D * (elem_bytes + kb) * 2   # read + write, K and V
    return {"pairs": pairs, "flops": flops, "bytes": kv_bytes + qo_bytes,
            "kv_bytes": kv_bytes, "append_bytes": append_bytes}


def kernel_source_hash(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "chunked_prefill_paged_cpa_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the kernel source that is built now."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[kernel][workload]
        if e.get("source_hash") != kernel_source_hash(e["sources"]):
            return None
        return float(e["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError, TypeError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------

def build_workload(name, seed, device):
    from chunked_prefill_paged_cpa_gb300 import workloads
    sc = workloads.scenario(name, seed)
    ws = workloads.WorkloadState(sc, device=device)
    initial = (ws.k_cache.clone(), ws.v_cache.clone())   # cache as the step finds it
    inp = ws.step(0)
    return sc, ws, inp, initial


def cpu_oracle_time(sc, ws, inp, initial, budget_s=20.0):
    """Time the fp64 oracle (as it stands) on the host cores over a bounded
    sample of the step's query rows.  The oracle builds its own cache from the
    pre-step cache and the step's new K/V with its own slots."""
    import numpy as np  # noqa: F401
    import oracle
    m = inp["meta"]
    kc, vc = initial[0].cpu(), initial[1].cpu()
    bt, qsl, sl = m.block_table.cpu(), m.query_start_loc.cpu(), m.seq_lens.cpu()
    slots = oracle.slot_mapping(bt, qsl, sl, sc.shape.page_size)
    oracle.kv_append(kc, vc, inp["k"].cpu(), inp["v"].cpu(), slots)
    q = inp["q"].cpu()
    T = q.shape[0]
    cores = os.cpu_count() or 1
    # per-row cost ~ visible keys; pick an evenly spaced sample of rows whose
    # estimated cost fits the budget, time it, scale to tokens/s
    q_lens, seq_lens = m.q_lens, m.seq_lens_list
    vis = []
    for ql, L in zip(q_lens, seq_lens):
        vis += [L - ql + i + 1 for i in range(ql)]
    probe = list(range(0, T, max(1, T // 64)))[:64]
    t0 = time.perf_counter()
    oracle.attention(q, kc, vc, bt, qsl, sl, sc.shape.scale, rows=probe, nthreads=cores)
    dt = time.perf_counter() - t0
    per_key = dt / max(1, sum(vis[r] for r in probe))
    total_est = per_key * sum(vis)
    if total_est <= budget_s:
        rows = list(range(T))
    else:
        stride = math.ceil(total_est / budget_s)
        rows = list(range(0, T, stride))
    t0 = time.perf_counter()
    oracle.attention(q, kc, vc, bt, qsl, sl, sc.shape.scale, rows=rows, nthreads=cores)
    dt = time.perf_counter() - t0
    frac_work = sum(vis[r] for r in rows) / sum(vis)
    step_s = dt / frac_work          # projected time of the whole step
    return {"value": T / step_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(rows)} of {T} query rows (all heads), {frac_work:.3f} of the "
                      f"step's visible keys, {dt:.1f} s on {cores} host threads; "
                      f"projected step {step_s * 1e3:.1f} ms",
            "seconds": dt}


def run_reference(args, world, rank):
    if rank != 0:
        return
    sc, ws, inp, initial = build_workload(args.config, args.seed, "cpu")
    times = []
    cb = None
    for i in range(args.warmup + args.steps):
        cb = cpu_oracle_time(sc, ws, inp, initial, budget_s=args.ref_budget)
        if i >= args.warmup:
            times.append(inp["meta"].num_tokens / cb["value"])
    ms = 1e3 * sum(times) / len(times)
    value = inp["meta"].num_tokens / (ms / 1e3)
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": workload_config(sc, inp),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cb["cores"],
                             "kind": "oracle", "sample": cb["sample"]},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(sc, inp):
    m = inp["meta"]
    sh = sc.shape
    dec = sum(1 for q in m.q_lens if q == 1)
    return {"workload": sc.name, "num_seqs": m.num_seqs, "decodes": dec,
            "query_tokens": m.num_tokens, "kv_tokens": int(sum(m.seq_lens_list)),
            "heads": f"{sh.num_q_heads}q/{sh.num_kv_heads}kv", "head_dim": sh.head_dim,
            "page_size": sh.page_size, "seed": sc.seed, "l2": "flushed before every timed step",
            "parallelism": "replicas (independent steps per GPU)"}


def run_gpu(args, world, rank, local):
    from chunked_prefill_paged_cpa_gb300 import ops
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    ops.load()
    sc, ws, inp, initial = build_workload(args.config, args.seed + rank, dev)
    sh = sc.shape
    m = inp["meta"]
    eb = torch.empty((), dtype=sh.dtype).element_size()
    counts = step_counts(m.q_lens, m.seq_lens_list, sh.num_q_heads, sh.num_kv_heads,
                         sh.head_dim, eb)
    wsp = ops.workspace_for(ws.k_cache, sh.num_q_heads, m.block_table.shape[1], m.num_seqs, m.num_tokens)
    out = torch.empty_like(inp["q"])
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)

    def step():
        ops.append_attention_forward(inp["q"], inp["k"], inp["v"], m.slot_mapping, ws.k_cache,
                                     ws.v_cache, m.block_table, m.query_start_loc, m.seq_lens,
                                     sh.scale, wsp, out=out, stream=stream)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    # this library's kernels per step, as cpa_append_attention_forward
    # dispatches them: on the step path (bf16, head_dim 64/128, GQA group
    # 1/2/4/8) the plan kernel (which also does the append) and the persistent
    # step kernel; fp32: the append, the tf32 chunk kernel and the row kernel
    G = sh.num_q_heads // sh.num_kv_heads
    step_path = sh.dtype == torch.bfloat16 and sh.head_dim in (64, 128) and G in (1, 2, 4, 8)
    fused = step_path
    launches_per_step = 2 if step_path else (3 if m.num_tokens >= 2 else 2)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    for i in range(args.steps):
        flush.fill_(i & 0xff)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    # breakdown: the same step as the two separate calls (append, attention)
    for i in range(args.steps):
        flush.fill_(i & 0xff)
        ev[i][0].record(stream)
        ops.kv_append(inp["k"], inp["v"], m.slot_mapping, ws.k_cache, ws.v_cache, stream=stream)
        ev[i][1].record(stream)
        ops.attention_forward(inp["q"], ws.k_cache, ws.v_cache, m.block_table,
                              m.query_start_loc, m.seq_lens, sh.scale, wsp, out=out,
                              stream=stream)
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    sep_step_ms = [e[0].elapsed_time(e[2]) for e in ev]
    attn_ms = [e[1].elapsed_time(e[2]) for e in ev]
    append_ms = [e[0].elapsed_time(e[1]) for e in ev]
    ms = total_ms / args.steps
    T = m.num_tokens
    value = T * world / (ms / 1e3)

    # end to end through the same C-ABI calls from pinned host buffers
    host = {k: inp[k].cpu().pin_memory() for k in ("q", "k", "v")}
    hmeta = {"slot": m.slot_mapping.cpu().pin_memory(),
             "bt": m.block_table.cpu().pin_memory(),
             "qsl": m.query_start_loc.cpu().pin_memory(),
             "sl": m.seq_lens.cpu().pin_memory()}
    dbuf = {k: torch.empty_like(v, device=dev) for k, v in host.items()}
    dmeta = {k: torch.empty_like(v, device=dev) for k, v in hmeta.items()}
    hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in list(host.values()) + list(hmeta.values()))
    d2h = hout.numel() * hout.element_size()

    # Pipelined like a serving loop: the next step's inputs go up on a copy
    # stream while this step's kernels run; each step's output comes back on
    # the copy stream after its kernels.  Inputs and outputs are double
    # buffered.  The L2 flush before each step is timed on its own and taken
    # out; the next step's input copy starts only after the flush and the next
    # flush only after the previous output copy, so no copy hides behind one.
    cs = torch.cuda.Stream(dev)
    dbuf2 = [dbuf, {k: torch.empty_like(v) for k, v in dbuf.items()}]
    dmeta2 = [dmeta, {k: torch.empty_like(v) for k, v in dmeta.items()}]
    outs2 = [out, torch.empty_like(out)]
    hout2 = [hout, torch.empty(out.shape, dtype=out.dtype, pin_memory=True)]

    def e2e_run(n, timed):
        E = lambda: torch.cuda.Event(enable_timing=timed)
        ev_in = [E() for _ in range(n)]
        ev_comp = [E() for _ in range(n)]
        ev_out = [E() for _ in range(n)]
        f0 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        f1 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def up(i):
            bi = i % 2
            with torch.cuda.stream(cs):
                if i >= 2:
                    cs.wait_event(ev_comp[i - 2])
                for k in host:
                    dbuf2[bi][k].copy_(host[k], non_blocking=True)
                for k in hmeta:
                    dmeta2[bi][k].copy_(hmeta[k], non_blocking=True)
                ev_in[i].record(cs)

        start.record(stream)
        cs.wait_stream(stream)
        for i in range(n):
            bi = i % 2
            if i >= 1:
                stream.wait_event(ev_out[i - 1])
            f0[i].record(stream)
            flush.fill_(i & 0xff)
            f1[i].record(stream)
            if i == 0:
                cs.wait_event(f1[0])
                up(0)
            stream.wait_event(ev_in[i])
            db, dm = dbuf2[bi], dmeta2[bi]
            ops.append_attention_forward(db["q"], db["k"], db["v"], dm["slot"], ws.k_cache,
                                         ws.v_cache, dm["bt"], dm["qsl"], dm["sl"], sh.scale,
                                         wsp, out=outs2[bi], stream=stream)
            ev_comp[i].record(stream)
            if i + 1 < n:
                cs.wait_event(f1[i])
                up(i + 1)
            with torch.cuda.stream(cs):
                cs.wait_event(ev_comp[i])
                hout2[bi].copy_(outs2[bi], non_blocking=True)
                ev_out[i].record(cs)
        stream.wait_event(ev_out[n - 1])
        end.record(stream)
        torch.cuda.synchronize()
        total = start.elapsed_time(end)
        fills = sum(a.elapsed_time(b) for a, b in zip(f0, f1))
        return (total - fills) / n

    e2e_run(args.warmup, False)
    barrier(world)
    e2e_ms = max_over_ranks(e2e_run(args.steps, True), world, dev)

    peaks, peak_src = load_peaks()
    attn_avg_ms = sum(attn_ms) / len(attn_ms)
    # the dominant launch group is the whole step's call: the attention
    # kernels with the append fused in (its cache writes add 4 KB per new
    # token at the Llama-3-8B shape; its reads of k/v are the attention's reads
    # of the step's own rows, already in the KV bytes)
    call_ms = ms
    call_bytes = counts["bytes"] + counts["append_bytes"] // 2
    t_bytes = counts["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_flops = counts["flops"] / (peaks["bf16_tflops"] * 1e12)
    if t_bytes >= t_flops:
        roof = {"bound": "hbm", "achieved": call_bytes / (call_ms * 1e-3) / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": counts["flops"] / (call_ms * 1e-3) / 1e12,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["peak_source"] = f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'})"
    roof["kernel"] = ("plan (with the append) + persistent step kernel "
                      "(cpa_append_attention_forward)" if fused
                      else "append + row attention (cpa_append_attention_forward)")
    roof["kernel_us"] = call_ms * 1e3
    roof["algorithmic_bytes"] = call_bytes
    roof["algorithmic_flops"] = counts["flops"]
    tr = committed_traffic("step", sc.name)
    roof["traffic"] = tr

    step_roof_s = max(t_bytes, t_flops)
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if sh.dtype == torch.bfloat16 else "f32", "data": "synthetic",
            "config": workload_config(sc, inp),
            "step_us": ms * 1e3,
            "step_roofline": {"roofline_us": step_roof_s * 1e6,
                              "frac": step_roof_s / (ms * 1e-3),
                              "t_hbm_us": t_bytes * 1e6, "t_tensor_us": t_flops * 1e6,
                              "note": "slower of step FLOPs at bf16 peak and KV/Q/O bytes at "
                                      "HBM peak, divided by the measured step (append + "
                                      "attention in one call)"},
            "append_fused": fused,
            "separate_calls": {"step_us": 1e3 * sum(sep_step_ms) / len(sep_step_ms),
                               "append_us": 1e3 * sum(append_ms) / len(append_ms),
                               "attention_us": attn_avg_ms * 1e3},
            "roofline": roof,
            "clocks": clk,
            "e2e": {"value": T * world / (e2e_ms / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms},
            "gpu_launches": launches_per_step * args.steps}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = cpu_oracle_time(sc, ws, inp, initial, budget_s=args.ref_budget)
        cb.pop("seconds", None)
        line["cpu_baseline"] = cb
    if world == 1 and not args.no_extras:
        # every configuration, timed the same way in the same run, and the
        # budget sweep with its free-ride grid (single-GPU runs only)
        del ws, inp, initial, wsp, out, dbuf, dmeta, dbuf2, dmeta2, outs2
        torch.cuda.empty_cache()
        line["workloads"] = measure_workloads(
            ["page1_default", "large_budget", "long_context", "decode_only", "oneshot_8192",
             "tiny", "page1_default_e4m3", "long_context_e4m3", "decode_only_e4m3"],
            dev, flush, stream, peaks, args.steps, args.warmup, args.seed)
        line["sweep"] = measure_sweep(dev, flush, stream, peaks, args.seed)
    if rank == 0:
        print(json.dumps(line), flush=True)



def _time_calls(fn, flush, stream, n):
    """Device time of n calls of fn, each after an L2 flush (CUDA events on
    the launching stream); returns a list of microseconds."""
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for i in range(n):
        flush.fill_(i & 0xff)
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) * 1e3 for a, b in ev]


def _fused_call(ws, inp, stream):
    """One step (append + attention) through cpa_append_attention_forward;
    repeating it is idempotent (the append writes the same bytes)."""
    from chunked_prefill_paged_cpa_gb300 import ops
    sh = ws.sc.shape
    m = inp["meta"]
    wsp = ops.workspace_for(ws.k_cache, sh.num_q_heads, m.block_table.shape[1], m.num_seqs,
                            m.num_tokens, sh.dtype)
    out = torch.empty_like(inp["q"])
    ks, vs = ws.kv_e4m3 or (1.0, 1.0)

    def call():
        ops.append_attention_forward(inp["q"], inp["k"], inp["v"], m.slot_mapping, ws.k_cache,
                                     ws.v_cache, m.block_table, m.query_start_loc, m.seq_lens,
                                     sh.scale, wsp, out=out, stream=stream, k_scale=ks,
                                     v_scale=vs)
    return call


def _roofline_entry(m, sh, us, peaks, kv_elem_bytes=None):
    eb = torch.empty((), dtype=sh.dtype).element_size()
    c = step_counts(m.q_lens, m.seq_lens_list, sh.num_q_heads, sh.num_kv_heads, sh.head_dim, eb,
                    kv_elem_bytes)
    t_b = c["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_f = c["flops"] / (peaks["bf16_tflops"] * 1e12)
    return c, {"roofline_us": max(t_b, t_f) * 1e6, "frac": max(t_b, t_f) * 1e6 / us,
               "bound": "hbm" if t_b >= t_f else "tensor",
               "t_hbm_us": t_b * 1e6, "t_tensor_us": t_f * 1e6}


def measure_workloads(names, dev, flush, stream, peaks, steps, warmup, seed):
    """Every named workload's first step through the fused call, timed like the
    headline (L2 flushed before each call, CUDA events on the launching
    stream): step time, query tokens/s and the fraction of the step roofline;
    decode-only steps also report achieved HBM bandwidth.  A name ending in
    _e4m3 is that workload over an 8-bit cache (OCP FP8 E4M3 codes, per-tensor
    scales; bf16 queries), its bytes counted at one byte per cached element."""
    from chunked_prefill_paged_cpa_gb300 import workloads
    res = {}
    for name in names:
        e4m3 = name.endswith("_e4m3")
        sc = workloads.scenario(name[:-5] if e4m3 else name, seed)
        ws = workloads.WorkloadState(sc, device=dev,
                                     kv_e4m3=workloads.E4M3_SCALES if e4m3 else None)
        inp = ws.step(0)
        m = inp["meta"]
        sh = sc.shape
        call = _fused_call(ws, inp, stream)
        for _ in range(warmup):
            flush.fill_(1)
            call()
        us = _time_calls(call, flush, stream, steps)
        mean = sum(us) / len(us)
        c, roof = _roofline_entry(m, sh, mean, peaks, 1 if e4m3 else None)
        e = {"step_us": mean, "step_us_min": min(us), "tokens_per_s": m.num_tokens / (mean * 1e-6),
             "query_tokens": m.num_tokens, "num_seqs": m.num_seqs,
             "kv_tokens": int(sum(m.seq_lens_list)),
             "dtype": "bf16" if sh.dtype == torch.bfloat16 else "f32"}
        if e4m3:
            e["kv_cache"] = {"format": "OCP FP8 E4M3", "k_scale": ws.kv_e4m3[0],
                             "v_scale": ws.kv_e4m3[1]}
        if sh.dtype == torch.bfloat16:
            e["step_roofline"] = roof
        else:
            e["step_roofline"] = None
            e["note"] = "fp32 parity configuration: launch latency only"
        if all(q == 1 for q in m.q_lens):
            gbs = (c["bytes"] + c["append_bytes"] // 2) / (mean * 1e-6) / 1e9
            e["hbm"] = {"achieved_gbs": gbs, "peak_gbs": peaks["hbm_gbs"],
                        "frac": gbs / peaks["hbm_gbs"],
                        "bytes": c["bytes"] + c["append_bytes"] // 2}
        res[name] = e
        del ws, inp, call
        torch.cuda.empty_cache()
    return res


def measure_sweep(dev, flush, stream, peaks, seed, budgets=(256, 512, 2048, 16384),
                  free_ride_grid=tuple(range(0, 2049, 64)), free_ride_steps=8):
    """Budget sweep: an 8192-token prompt prefilled from scratch beside 32
    decodes, once per token budget, every step timed (append + attention, L2
    flushed before each); per budget the mean step time, the prompt's total
    prefill time and the mean fraction of each step's roofline.  Then the
    free ride: the default step's 32 decodes beside a chunk of C tokens at
    offset 3840, C on a grid from 0 (decodes alone); the largest C whose step
    stays within 5 % of the decodes-alone step, beside the attention form of
    the pages' estimate (the chunk's FLOPs at bf16 peak fit in the time the
    decodes' KV bytes take at HBM peak)."""
    from chunked_prefill_paged_cpa_gb300 import ops, workloads
    rows = []
    for budget in budgets:
        sc = workloads.budget_sweep(budget, seed)
        ws = workloads.WorkloadState(sc, device=dev)
        sh = sc.shape
        steps = [ws.step(k) for k in range(len(sc.plans))]
        max_pages = max(x["meta"].block_table.shape[1] for x in steps)
        max_seqs = max(x["meta"].num_seqs for x in steps)
        wsp = ops.workspace_for(ws.k_cache, sh.num_q_heads, max_pages, max_seqs,
                                 max(x["meta"].num_tokens for x in steps))
        outs = [torch.empty_like(x["q"]) for x in steps]

        def one(k):
            x, m = steps[k], steps[k]["meta"]
            ops.append_attention_forward(x["q"], x["k"], x["v"], m.slot_mapping, ws.k_cache,
                                         ws.v_cache, m.block_table, m.query_start_loc,
                                         m.seq_lens, sh.scale, wsp, out=outs[k], stream=stream)

        for k in range(len(steps)):       # warm-up pass (appends are idempotent)
            one(k)
        torch.cuda.synchronize()
        us = []
        for k in range(len(steps)):
            us += _time_calls(lambda: one(k), flush, stream, 1)
        fr = [_roofline_entry(x["meta"], sh, us[k], peaks)[1]["frac"] for k, x in enumerate(steps)]
        rows.append({"budget": budget, "steps": len(steps), "chunk_tokens": budget - 32,
                     "step_us_mean": sum(us) / len(us), "step_us_max": max(us),
                     "prompt_prefill_ms": sum(us) / 1e3,
                     "decode_tokens_during_prefill": 32 * len(steps),
                     "step_roofline_frac_mean": sum(fr) / len(fr)})
        del ws, steps, outs, wsp
        torch.cuda.empty_cache()
    grid = []
    base_bytes = None
    for chunk in free_ride_grid:
        sc = workloads.free_ride(chunk, seed)
        ws = workloads.WorkloadState(sc, device=dev)
        inp = ws.step(0)
        call = _fused_call(ws, inp, stream)
        for _ in range(3):
            flush.fill_(1)
            call()
        us = _time_calls(call, flush, stream, free_ride_steps)
        m = inp["meta"]
        c, roof = _roofline_entry(m, sc.shape, sum(us) / len(us), peaks)
        if chunk == 0:
            base_bytes = c["bytes"]
        grid.append({"chunk": chunk, "step_us": sum(us) / len(us), "step_us_min": min(us),
                     "step_roofline_frac": roof["frac"]})
        del ws, inp, call
        torch.cuda.empty_cache()
    base = grid[0]["step_us"]
    free = max(g["chunk"] for g in grid if g["step_us"] <= 1.05 * base)
    # attention form of the estimate: C chunk tokens at offset P cost
    # 4*D*Hq*(P*C + C*(C+1)/2) FLOPs; set that equal to the decodes' HBM time
    # times the bf16 peak and solve for C
    sh = workloads.LLAMA3_8B
    per_pair = 4 * sh.head_dim * sh.num_q_heads
    flops_budget = base_bytes / (peaks["hbm_gbs"] * 1e9) * peaks["bf16_tflops"] * 1e12
    P = 3840
    est = -P + math.sqrt(P * P + 2 * flops_budget / per_pair)
    return {"budgets": rows,
            "free_ride": {"decodes": 32, "chunk_offset": P, "decodes_alone_us": base,
                          "measured_free_tokens": free, "criterion": "step within 5 % of the "
                          "decodes-alone step", "formula_free_tokens": est,
                          "formula": "C with 4*D*Hq*(P*C + C^2/2) / bf16 peak = decode bytes / "
                                     "HBM peak", "grid": grid}}


def run_sweep(args):
    """The sweep alone, as its own JSON line."""
    from chunked_prefill_paged_cpa_gb300 import ops
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    ops.load()
    peaks, peak_src = load_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sw = measure_sweep(dev, flush, stream, peaks, args.seed)
    line = {"metric": "budget sweep: per-step us and total prompt prefill time", "unit": "us",
            "higher_is_better": False, "n_gpus": 1, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "budget_sweep", "prompt": 8192, "decodes": 32,
                       "decode_context": "U[512, 4096]", "heads": "32q/8kv", "head_dim": 128,
                       "page_size": 16, "seed": args.seed,
                       "l2": "flushed before every timed step",
                       "peaks": f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'})"},
            "sweep": sw}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--config", default="page1_default")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--ref-budget", type=float, default=15.0,
                    help="seconds of host work per oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="budget sweep of an 8192-token prompt beside 32 decodes (one JSON line)")
    ap.add_argument("--no-extras", action="store_true",
                    help="time only the headline workload (no per-workload table, no sweep)")
    args = ap.parse_args()
    if args.sweep:
        run_sweep(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        # the oracle runs on rank 0's host cores only; other ranks exit at once
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        args.ref_budget = min(args.ref_budget, 150.0 / (args.steps + args.warmup))
        run_reference(args, world, rank)
        return
    world, rank, local = dist_setup(args)
    run_gpu(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
