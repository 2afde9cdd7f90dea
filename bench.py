#!/usr/bin/env python3
"""Benchmark of the MoE expert-parallel dispatch / combine path on GB300.

One step = one pass of the whole normal-mode path over one synthetic batch of
the prefill workload (R=8 virtual ranks x T=4096 tokens, E=256, top-8,
H=7168 bf16): layout -> notify (with its host sync) -> dispatch scatter ->
permute -> combine, with the identity expert (expert_out = permuted_x).
The same run also times the low-latency layer on the decode workload
(R=16 x 128 tokens, FP8 send + receive/pack + BF16 combine) and reports it
as ``ll_decode``.  Further legs of the same line: ``fused_path`` (dispatch
straight into the per-expert layout), ``expert_aligned`` (the permute into
128-row aligned blocks), ``graph`` (the steps without a host wait, each one
CUDA graph), ``fp8_rows`` (FP8 quantiser and FP8 dispatches), ``e2e``
(the step from pinned host buffers, copies inside the timed region), and the
other workloads timed the same way: ``skewed`` (the Zipf-skewed normal
step), ``skewed_ll`` (its low-latency layer in 256-token microbatches) and
``hier`` (the 4-node staged step).

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "dispatch+combine tokens/s and effective HBM GB/s (% of ~8 TB/s); LL µs/layer"
L2_FLUSH_BYTES = 512 << 20  # > 2x the 129 MB L2
L2_DESC = ("flushed before each timed region, not timed: a 512 MiB write, then a 512 MiB read of a second "
           "buffer, so that L2 holds none of the inputs and none of the flush's own dirty lines")


class L2Flush:
    """Cold-L2 reset between timed iterations.  Writing a buffer larger than L2
    evicts the inputs but leaves L2 full of the buffer's dirty lines, whose
    write-back would then be charged to the first timed kernel (~7 us of the
    decode send); reading a second such buffer afterwards writes them back
    before the timed region starts."""

    def __init__(self, torch):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")

    def __call__(self):
        self.w.zero_()
        self.r.max()
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes (read + write) per launch of the dominant kernel: ncu's
# dram__bytes_read.sum + dram__bytes_write.sum of one launch of the same kernel
# on a smaller case, scaled to a full launch by the rows it moves; only for a
# kernel unchanged since that capture (else the roofline's traffic is null).
TRAFFIC = {
    ("prefill", "permute"): {"bytes": 6.073e9,
                             "case": "one permute launch at T=1024 (R=8, E=256, K=8, H=7168), "
                                     "scaled by the rows moved (x 4.024)"},
}


NOMINAL_HBM_GBS = 8000.0  # the metric's "% of ~8 TB/s"


def add_nominal_pct(obj):
    """Beside every effective GB/s figure, its percentage of the nominal ~8 TB/s
    the metric names (the `frac` keys stay fractions of the measured peak)."""
    if isinstance(obj, dict):
        for k in list(obj):
            v = obj[k]
            if k in ("GBps", "effective_GBps") and isinstance(v, (int, float)):
                obj[k.replace("GBps", "pct_of_8TBps")] = round(100.0 * v / NOMINAL_HBM_GBS, 1)
            else:
                add_nominal_pct(v)
    elif isinstance(obj, list):
        for v in obj:
            add_nominal_pct(v)
    return obj


def measured_hbm_gbs():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# algorithmic bytes per unit of work (each row read or written once)
# ---------------------------------------------------------------------------

def algo_bytes(H, K, tokens, copies, pairs, staged=0):
    """staged = node copies of the hierarchical dispatch (0: flat): stage A reads
    each token once and writes one row per destination node, stage B reads each
    staged row once and writes one row per destination rank."""
    row = 2 * H
    dispatch = (tokens + copies) * row if not staged else (tokens + 2 * staged + copies) * row
    return {
        "dispatch": dispatch,
        "permute": (copies + pairs) * row,
        "combine": (pairs + tokens) * row + tokens * K * 8,
    }


def pct(xs, q):
    xs = sorted(xs)
    return xs[min(len(xs) - 1, max(0, int(round(q * (len(xs) - 1)))))]


def ll_algo_bytes(H, tokens, pairs):
    row = 2 * H
    msg = H + H // 32 + 4
    return {
        "ll_send": tokens * row + pairs * msg,
        "ll_recv": 2 * pairs * msg,
        "ll_combine": pairs * row + tokens * row,
    }


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# the CPU oracle (reported baseline; also the "reference" arm)
# ---------------------------------------------------------------------------

def oracle_sample(workload, budget_s: float, min_s: float):
    """Times the oracle's normal-mode chain on samples of the workload (T cut
    down, same R, E, K, H, router) until min_s of CPU work has been done."""
    import oracle
    from combine_get_dispatch_histograms_gb300 import inputs
    oracle.build()
    T = 128 if workload.H >= 4096 else 1024
    w = workload.replace(T=T)
    tokens = 0
    t_total = 0.0
    seed = 100
    while True:
        x, idx, wts = inputs.make_inputs(w, seed=seed)
        t = time.perf_counter()
        oracle.run_normal(x, idx, wts, w.R, w.E, w.num_channels)
        t_total += time.perf_counter() - t
        tokens += w.R * w.T
        seed += 1
        if t_total >= min_s or t_total > budget_s:
            break
    return {"value": tokens / t_total, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{tokens} tokens: {seed - 100} batches of R={w.R} x T={w.T} (E={w.E}, K={w.K}, H={w.H}), "
                      f"single-threaded plain C oracle, {t_total:.1f} s",
            "seconds": round(t_total, 3), "T": w.T}


def _oracle_worker(args):
    name, T, seed, budget = args
    from combine_get_dispatch_histograms_gb300 import inputs
    w = inputs.WORKLOADS[name].replace(T=T)
    import oracle
    tokens, t_total = 0, 0.0
    while True:
        x, idx, wts = inputs.make_inputs(w, seed=seed)
        t = time.perf_counter()
        oracle.run_normal(x, idx, wts, w.R, w.E, w.num_channels)
        t_total += time.perf_counter() - t
        tokens += w.R * w.T
        seed += 1000
        if t_total >= budget:
            return tokens, t_total


def oracle_parallel(workload, seconds: float):
    """The same oracle, one independent sample stream per host core (spawned
    processes), aggregate tokens/s."""
    import multiprocessing as mp
    import oracle
    oracle.build()
    cores = len(os.sched_getaffinity(0))
    T = 128 if workload.H >= 4096 else 1024
    ctx = mp.get_context("spawn")
    t0 = time.perf_counter()
    with ctx.Pool(cores) as pool:
        res = pool.map(_oracle_worker, [(workload.name, T, 500 + i, seconds) for i in range(cores)])
    wall = time.perf_counter() - t0
    tokens = sum(r[0] for r in res)
    busy = max(r[1] for r in res)
    return {"value": tokens / busy, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{tokens} tokens over {cores} spawned processes, batches of R={workload.R} x T={T}, "
                      f"{busy:.1f} s of oracle time per process ({wall:.1f} s wall incl. input generation)"}


def run_ll_only(args):
    """The decode low-latency layer alone (send, receive, combine), for a
    profiler on a small case: prints the per-kernel times, not the contract line."""
    import torch
    from combine_get_dispatch_histograms_gb300 import LLBuffer, inputs
    dw = inputs.WORKLOADS[args.ll_workload]
    if args.ll_tokens:
        dw = dw.replace(T=args.ll_tokens, ll_cap=args.ll_tokens)
    if args.ll_experts:
        dw = dw.replace(E=args.ll_experts)
    idx, wt = inputs.make_routing(dw, 7)
    x = inputs.make_x(dw, 7, device="cuda")
    idxd, wd = idx.cuda(), wt.cuda()
    buf = LLBuffer(dw.R, dw.E, dw.K, dw.T, dw.H, dw.ll_cap)
    pk = buf.alloc_packed()
    y = torch.zeros(pk["packed_x"].shape, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(dw.R, dw.T, dw.H, dtype=torch.bfloat16, device="cuda")
    st = torch.cuda.current_stream()
    flush = L2Flush(torch)
    times = []
    mbs = [(t0, min(dw.ll_cap, dw.T - t0)) for t0 in range(0, dw.T, dw.ll_cap)]  # microbatches of <= cap tokens
    for i in range(args.warmup + args.steps):
        for t0, n in mbs:
            flush()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            e[0].record(st)
            buf.send(x, idxd, t0, n, out=pk)
            e[1].record(st)
            buf.recv(pk)
            e[2].record(st)
            buf.combine(y, idxd, wd, pk, t0, n, out=out)
            e[3].record(st)
            torch.cuda.synchronize()
            if i >= args.warmup:
                times.append([e[j].elapsed_time(e[j + 1]) * 1e3 for j in range(3)])
    buf.check()
    med = [statistics.median(t[j] for t in times) for j in range(3)] if times else [None] * 3
    print(json.dumps({"ll_only": {"workload": dw.name, "R": dw.R, "T": dw.T, "H": dw.H, "cap": dw.ll_cap,
                                  "microbatches": len(mbs), "send_us": med[0], "recv_us": med[1],
                                  "combine_us": med[2], "per": "microbatch (median)"}}), flush=True)
    return 0


def run_reference(args, workload):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    steps = []
    for _ in range(args.warmup):
        oracle_sample(workload, budget_s=3.0, min_s=0.0)
    for _ in range(args.steps):
        r = oracle_sample(workload, budget_s=6.0, min_s=0.0)
        steps.append(r)
    value = statistics.median(s["value"] for s in steps)
    sample_ms = statistics.median(s["seconds"] for s in steps) * 1e3
    cpu = dict(steps[-1])
    cpu["value"] = value
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        # each timed step is one bounded sample of the workload (T cut down):
        # its own time, so that steps x ms_per_step is the time spent
        "ms_per_step": round(sample_ms, 1),
        "step": f"one sample of R={workload.R} x T={steps[-1]['T']} tokens of the {workload.name} workload",
        # the whole workload's step at the sampled rate, for comparison with the GPU arm
        "ms_per_full_step_extrapolated": round(1e3 * workload.R * workload.T / value, 1) if value else None,
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload.name, "R": workload.R, "E": workload.E, "K": workload.K,
                   "T": workload.T, "H": workload.H},
        "cpu_baseline": cpu,
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def kernel_entry(times_ms, nbytes, peak):
    """Median / p10 / p90 of a kernel's event times; with its algorithmic
    bytes, the effective GB/s and the fraction of the measured peak."""
    med = statistics.median(times_ms)
    e = {"us": round(med * 1e3, 2), "p10_us": round(pct(times_ms, 0.1) * 1e3, 2),
         "p90_us": round(pct(times_ms, 0.9) * 1e3, 2)}
    if nbytes is not None:
        gbs = nbytes / (med * 1e-3) / 1e9
        e.update({"algo_bytes": nbytes, "GBps": round(gbs, 1), "frac": round(gbs / peak, 3)})
    return e


def normal_leg(torch, w, seed, steps, warmup, flush):
    """One more normal-mode workload timed like the main step (layout, notify
    with its host wait, dispatch - staged for a hierarchical workload -,
    permute, combine; identity expert; L2 flushed before every step): per
    kernel times and fractions, the step time and tokens/s."""
    from combine_get_dispatch_histograms_gb300 import Context, inputs
    R, E, K, T, H, C = w.R, w.E, w.K, w.T, w.H, w.num_channels
    hier = w.num_nodes > 1
    topk_idx, topk_w = inputs.make_routing(w, seed)
    x = inputs.make_x(w, seed, device="cuda")
    idx_d, w_d = topk_idx.cuda(), topk_w.cuda()
    ctx = Context(R, E, K, T, H, num_channels=C, num_nodes=w.num_nodes)
    stream = torch.cuda.current_stream()
    lay = ctx.get_dispatch_layout(idx_d, nodes=hier)
    h = ctx.notify_dispatch(idx_d, lay)
    recv = ctx.alloc_recv(h.num_recv_rows)
    perm = dict(permuted_x=torch.empty(h.num_perm_rows, H, dtype=torch.bfloat16, device="cuda"),
                perm_src_row=torch.empty(h.num_perm_rows, dtype=torch.int32, device="cuda"))
    out = torch.empty(R, T, H, dtype=torch.bfloat16, device="cuda")
    staging = None
    if hier:
        S = h.num_stage_rows
        staging = dict(staging=torch.empty(S, H, dtype=torch.bfloat16, device="cuda"),
                       stage_src_rank=torch.empty(S, dtype=torch.int32, device="cuda"),
                       stage_src_idx=torch.empty(S, dtype=torch.int32, device="cuda"))

    def step(ev):
        ev[0].record(stream)
        ctx.get_dispatch_layout(idx_d, nodes=hier, out=lay)
        ev[1].record(stream)
        ctx.notify_dispatch(idx_d, lay, handle=h)
        ev[2].record(stream)
        if hier:
            ctx.dispatch_hier(x, idx_d, w_d, h, out=recv, staging=staging)
        else:
            ctx.dispatch(x, idx_d, w_d, h, out=recv)
        ev[3].record(stream)
        ctx.permute(h, recv, out=perm)
        ev[4].record(stream)
        ctx.combine(h, perm["permuted_x"], idx_d, w_d, out=out, hier=hier)
        ev[5].record(stream)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(warmup + steps)]
    for i in range(warmup + steps):
        flush()
        step(evs[i])
    torch.cuda.synchronize()
    ctx.check()
    evs = evs[warmup:]
    names = ["layout", "notify", "dispatch", "permute", "combine"]
    tokens, copies, pairs = R * T, h.num_recv_rows, h.num_perm_rows
    ab = algo_bytes(H, K, tokens, copies, pairs, h.num_stage_rows if hier else 0)
    peak, _ = measured_hbm_gbs()
    kernels = {n: kernel_entry([e[j].elapsed_time(e[j + 1]) for e in evs], ab.get(n), peak)
               for j, n in enumerate(names)}
    ms = sum(e[0].elapsed_time(e[5]) for e in evs) / len(evs)
    res = {"workload": w.name, "R": R, "E": E, "K": K, "T": T, "H": H, "num_nodes": w.num_nodes,
           "router": w.router, "copies": copies, "pairs": pairs, "ms_per_step": round(ms, 4),
           "tokens_per_s": round(tokens / (ms / 1e3), 1), "kernels": kernels,
           "effective_GBps": round(sum(ab.values()) / (sum(statistics.median(
               e[j].elapsed_time(e[j + 1]) for e in evs) for j in (2, 3, 4)) * 1e-3) / 1e9, 1)}
    if hier:
        res["staged_rows"] = h.num_stage_rows
        res["dispatch_note"] = "stage A (one row per destination node) + stage B (forward inside the node)"
    return res


def ll_microbatch_leg(torch, w, seed, steps, warmup, flush):
    """The low-latency layer of a workload whose T exceeds the per-region cap:
    T split into microbatches of <= cap tokens, each sent, received and
    combined (expert output: a distinct row per packed slot); per kernel the
    median over every microbatch of every timed step, and the whole batch's
    time."""
    from combine_get_dispatch_histograms_gb300 import LLBuffer, inputs
    R, E, K, T, H, cap = w.R, w.E, w.K, w.T, w.H, w.ll_cap
    L = E // R
    topk_idx, topk_w = inputs.make_routing(w, seed)
    x = inputs.make_x(w, seed, device="cuda")
    idx_d, w_d = topk_idx.cuda(), topk_w.cuda()
    buf = LLBuffer(R, E, K, T, H, cap)
    pk = buf.alloc_packed()
    y = inputs.random_rows(R * L * R * cap, H, seed, device="cuda").view(R, L, R * cap, H)
    out = torch.empty(R, T, H, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    mbs = [(t0, min(cap, T - t0)) for t0 in range(0, T, cap)]
    names = ["ll_send", "ll_recv", "ll_combine"]
    per = {n: [] for n in names}
    batch_ms = []
    peak, _ = measured_hbm_gbs()
    nbytes = {n: [] for n in names}
    idx_np = topk_idx.numpy()
    for i in range(warmup + steps):
        tot = 0.0
        for t0, n in mbs:
            flush()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            e[0].record(stream)
            buf.send(x, idx_d, t0, n, out=pk)
            e[1].record(stream)
            buf.recv(pk)
            e[2].record(stream)
            buf.combine(y, idx_d, w_d, pk, t0, n, out=out)
            e[3].record(stream)
            torch.cuda.synchronize()
            if i >= warmup:
                for j, nm in enumerate(names):
                    per[nm].append(e[j].elapsed_time(e[j + 1]))
                tot += e[0].elapsed_time(e[3])
                if i == warmup:
                    b = ll_algo_bytes(H, R * n, int((idx_np[:, t0:t0 + n] >= 0).sum()))
                    for nm in names:
                        nbytes[nm].append(b[nm])
        if i >= warmup:
            batch_ms.append(tot)
    buf.check()
    kernels = {}
    for nm in names:
        kernels[nm] = kernel_entry(per[nm], statistics.median(nbytes[nm]), peak)
        kernels[nm]["algo_bytes_note"] = "median over the microbatches"
    batch_bytes = sum(sum(nbytes[nm]) for nm in names)
    bm = statistics.median(batch_ms)
    return {"workload": w.name, "R": R, "E": E, "K": K, "T": T, "H": H, "cap": cap, "microbatches": len(mbs),
            "batch": {"algo_bytes": batch_bytes, "GBps": round(batch_bytes / (bm * 1e-3) / 1e9, 1),
                      "frac": round(batch_bytes / (bm * 1e-3) / 1e9 / peak, 3),
                      "what": "all microbatches' send, receive and combine bytes over the batch time "
                              "(per-kernel events, L2 flushed before each microbatch)"},
            "us_per_microbatch": round(statistics.median(per["ll_send"]) * 1e3 + statistics.median(
                per["ll_recv"]) * 1e3 + statistics.median(per["ll_combine"]) * 1e3, 2),
            "ms_per_batch": round(statistics.median(batch_ms), 4),
            "tokens_per_s": round(R * T / (statistics.median(batch_ms) / 1e3), 1),
            "kernels": kernels,
            "timing": "per-kernel events on one stream, L2 flushed before every microbatch"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="prefill", choices=["prefill", "skewed", "hier"])
    ap.add_argument("--tokens", type=int, default=0, help="override T (profiling on a smaller case)")
    ap.add_argument("--no-ll", action="store_true", help="skip the low-latency decode leg")
    ap.add_argument("--ll-only", action="store_true",
                    help="profiling mode: only the low-latency decode layer (no contract line)")
    ap.add_argument("--ll-workload", default="decode", choices=["decode", "skewed"],
                    help="with --ll-only: the low-latency workload (skewed runs 256-token microbatches)")
    ap.add_argument("--ll-tokens", type=int, default=0, help="with --ll-only: T = cap of the decode layer")
    ap.add_argument("--ll-experts", type=int, default=0,
                    help="with --ll-only: E of the decode layer (fewer experts: same messages, smaller buffers)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline leg")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="skip the skewed and hierarchical legs of the default prefill run")
    args = ap.parse_args()

    from combine_get_dispatch_histograms_gb300 import inputs
    workload = inputs.WORKLOADS[args.workload]
    if args.tokens:
        workload = workload.replace(T=args.tokens)
    if args.impl == "reference":
        return run_reference(args, workload)
    if args.ll_only:
        return run_ll_only(args)

    import torch
    from combine_get_dispatch_histograms_gb300 import Context, LLBuffer
    from combine_get_dispatch_histograms_gb300 import dist as epdist

    info = epdist.init_from_env("nccl")
    world, rank, local = info.world, info.rank, info.local_rank
    barrier, max_over_ranks, sum_over_ranks = epdist.barrier, epdist.max_over_ranks, epdist.sum_over_ranks

    w = workload
    R, E, K, T, H, C = w.R, w.E, w.K, w.T, w.H, w.num_channels
    hier = w.num_nodes > 1
    seed = epdist.rank_seed(0, rank)  # every rank processes its own batch (weak scaling)
    topk_idx, topk_w = inputs.make_routing(w, seed)
    x = inputs.make_x(w, seed, device="cuda")
    idx_d, w_d = topk_idx.cuda(), topk_w.cuda()
    ctx = Context(R, E, K, T, H, num_channels=C, num_nodes=w.num_nodes)
    stream = torch.cuda.current_stream()
    flush = L2Flush(torch)

    # sizes from one notify, then buffers allocated once
    lay = ctx.get_dispatch_layout(idx_d, nodes=hier)
    handle = ctx.notify_dispatch(idx_d, lay)
    recv = ctx.alloc_recv(handle.num_recv_rows)
    perm = dict(permuted_x=torch.empty(handle.num_perm_rows, H, dtype=torch.bfloat16, device="cuda"),
                perm_src_row=torch.empty(handle.num_perm_rows, dtype=torch.int32, device="cuda"))
    out = torch.empty(R, T, H, dtype=torch.bfloat16, device="cuda")
    staging = None
    if hier:
        S = handle.num_stage_rows
        staging = dict(staging=torch.empty(S, H, dtype=torch.bfloat16, device="cuda"),
                       stage_src_rank=torch.empty(S, dtype=torch.int32, device="cuda"),
                       stage_src_idx=torch.empty(S, dtype=torch.int32, device="cuda"))
    tokens = R * T
    copies = handle.num_recv_rows
    pairs = handle.num_perm_rows
    names = ["layout", "notify", "dispatch", "permute", "combine"]
    launches = {"layout": 1, "notify": 2, "dispatch": 2 if hier else 1, "permute": 1, "combine": 1}

    def step(ev=None):
        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        mark(0)
        ctx.get_dispatch_layout(idx_d, nodes=hier, out=lay)
        mark(1)
        ctx.notify_dispatch(idx_d, lay, handle=handle)
        mark(2)
        if hier:
            ctx.dispatch_hier(x, idx_d, w_d, handle, out=recv, staging=staging)
        else:
            ctx.dispatch(x, idx_d, w_d, handle, out=recv)
        mark(3)
        ctx.permute(handle, recv, out=perm)
        mark(4)
        ctx.combine(handle, perm["permuted_x"], idx_d, w_d, out=out, hier=hier)
        mark(5)

    for _ in range(args.warmup):
        flush()
        step()
    ctx.check()
    torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush()  # L2 flush between steps, outside the step's events
        step(evs[i])
    torch.cuda.synchronize()
    barrier()
    wall = time.perf_counter() - wall0
    ctx.check()
    per = {n: [] for n in names}
    step_ms = []
    for ev in evs:
        for j, n in enumerate(names):
            per[n].append(ev[j].elapsed_time(ev[j + 1]))
        step_ms.append(ev[0].elapsed_time(ev[5]))
    local_ms = sum(step_ms) / len(step_ms)
    ms = max_over_ranks(local_ms)
    total_tokens = sum_over_ranks(tokens)
    value = total_tokens / (ms / 1e3)

    # ---- fused path: dispatch straight into the expert-major layout --------------
    fused = None
    if not hier:
        fperm = dict(permuted_x=perm["permuted_x"], perm_src_token=torch.empty(pairs, dtype=torch.int32, device="cuda"),
                     perm_weight=torch.empty(pairs, dtype=torch.float32, device="cuda"))

        def fstep(ev=None):
            def mark(i):
                if ev is not None:
                    ev[i].record(stream)
            mark(0)
            ctx.get_dispatch_layout(idx_d, out=lay)
            mark(1)
            ctx.notify_dispatch(idx_d, lay, handle=handle)
            mark(2)
            ctx.dispatch_permuted(x, idx_d, w_d, handle, out=fperm)
            mark(3)
            ctx.combine(handle, fperm["permuted_x"], idx_d, w_d, out=out)
            mark(4)

        for _ in range(args.warmup):
            flush()
            fstep()
        fev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush()
            fstep(fev[i])
        torch.cuda.synchronize()
        ctx.check()
        fms = max_over_ranks(sum(e[0].elapsed_time(e[4]) for e in fev) / args.steps)
        fd = statistics.median(e[2].elapsed_time(e[3]) for e in fev)
        fb = (tokens + pairs) * 2 * H
        peak0, _ = measured_hbm_gbs()
        fused = {"ms_per_step": round(fms, 4), "tokens_per_s": round(sum_over_ranks(tokens) / (fms / 1e3), 1),
                 "steps": "layout -> notify -> fused dispatch into the permuted layout -> combine",
                 "dispatch_permuted": {"us": round(fd * 1e3, 2), "algo_bytes": fb,
                                       "GBps": round(fb / (fd * 1e-3) / 1e9, 1),
                                       "frac": round(fb / (fd * 1e-3) / 1e9 / peak0, 3)}}
        del fperm

    # ---- expert-aligned permute: every (rank, expert) block rounded up to 128 rows ----
    aligned = None
    if not hier:
        actx = Context(R, E, K, T, H, num_channels=C, expert_alignment=128)
        ah = actx.notify_dispatch(idx_d, actx.get_dispatch_layout(idx_d))  # the receive layout is the same
        aperm = dict(permuted_x=torch.empty(ah.num_perm_rows, H, dtype=torch.bfloat16, device="cuda"),
                     perm_src_row=torch.empty(ah.num_perm_rows, dtype=torch.int32, device="cuda"))
        for _ in range(args.warmup):
            flush()
            actx.permute(ah, recv, out=aperm)
        aev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush()
            aev[i][0].record(stream)
            actx.permute(ah, recv, out=aperm)
            aev[i][1].record(stream)
        torch.cuda.synchronize()
        actx.check()
        ad = statistics.median(e[0].elapsed_time(e[1]) for e in aev)
        ab = (copies + pairs) * 2 * H  # padding rows are not written
        peak0, _ = measured_hbm_gbs()
        aligned = {"alignment": 128, "permuted_rows": ah.num_perm_rows, "pairs": pairs,
                   "permute": {"us": round(ad * 1e3, 2), "algo_bytes": ab, "GBps": round(ab / (ad * 1e-3) / 1e9, 1),
                               "frac": round(ab / (ad * 1e-3) / 1e9 / peak0, 3)}}
        del aperm, actx

    # ---- the same steps without a host synchronisation, replayed as one CUDA graph ----
    # (notify's no-wait form; buffers sized for the worst case; the kernels read
    # the row totals from the handle on the device)
    nw_graph = None
    if not hier:
        rmax, pmax, _ = ctx.max_rows
        g_recv = ctx.alloc_recv(rmax)
        g_perm = dict(permuted_x=torch.empty(pmax, H, dtype=torch.bfloat16, device="cuda"),
                      perm_src_row=torch.empty(pmax, dtype=torch.int32, device="cuda"))
        g_fused = dict(permuted_x=g_perm["permuted_x"],
                       perm_src_token=torch.empty(pmax, dtype=torch.int32, device="cuda"),
                       perm_weight=torch.empty(pmax, dtype=torch.float32, device="cuda"))
        g_out = torch.empty(R, T, H, dtype=torch.bfloat16, device="cuda")
        g_lay = {k: torch.empty_like(v) for k, v in lay.items()}
        g_h = ctx.alloc_handle()

        def nw_step():
            ctx.get_dispatch_layout(idx_d, out=g_lay)
            ctx.notify_dispatch(idx_d, g_lay, handle=g_h, wait=False)
            ctx.dispatch(x, idx_d, w_d, g_h, out=g_recv)
            ctx.permute(g_h, g_recv, out=g_perm)
            ctx.combine(g_h, g_perm["permuted_x"], idx_d, w_d, out=g_out)

        def nw_fused():
            ctx.get_dispatch_layout(idx_d, out=g_lay)
            ctx.notify_dispatch(idx_d, g_lay, handle=g_h, wait=False)
            ctx.dispatch_permuted(x, idx_d, w_d, g_h, out=g_fused)
            ctx.combine(g_h, g_fused["permuted_x"], idx_d, w_d, out=g_out)

        def nw_fewest():  # layout fused into notify, fused dispatch: four launches
            ctx.layout_notify(idx_d, handle=g_h, out=g_lay, wait=False)
            ctx.dispatch_permuted(x, idx_d, w_d, g_h, out=g_fused)
            ctx.combine(g_h, g_fused["permuted_x"], idx_d, w_d, out=g_out)

        nw_graph = {"steps": "one CUDA graph per step: layout -> notify (no host wait) -> ... ; "
                          "worst-case buffers, row totals read on the device"}
        for name, fn in (("step", nw_step), ("fused_path", nw_fused), ("fused_path_layout_in_notify", nw_fewest)):
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                fn()  # eager once outside the capture
            stream.wait_stream(side)
            torch.cuda.synchronize()
            cg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(cg):
                fn()
            for _ in range(args.warmup):
                flush()
                cg.replay()
            gev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
            for i in range(args.steps):
                flush()
                gev[i][0].record(stream)
                cg.replay()
                gev[i][1].record(stream)
            torch.cuda.synchronize()
            ctx.check()
            # the replayed step gives the eager step's output, bit for bit
            step()
            torch.cuda.synchronize()
            if not torch.equal(g_out.view(torch.int16), out.view(torch.int16)):
                raise RuntimeError(f"graph {name}: output differs from the eager step")
            gms = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in gev) / args.steps)
            nw_graph[name] = {"ms_per_step": round(gms, 4),
                           "tokens_per_s": round(sum_over_ranks(tokens) / (gms / 1e3), 1)}
            del cg
        del g_recv, g_perm, g_fused, g_out

    # ---- FP8 rows on the normal path: quantise once, then the fused dispatch ----
    fp8 = None
    if not hier and H % 128 == 0:
        rq = ctx.fp8_row_bytes
        xq = torch.empty(R * T, rq, dtype=torch.uint8, device="cuda")
        fq = dict(permuted_xq=torch.empty(pairs, rq, dtype=torch.uint8, device="cuda"),
                  perm_src_token=torch.empty(pairs, dtype=torch.int32, device="cuda"),
                  perm_weight=torch.empty(pairs, dtype=torch.float32, device="cuda"))
        for _ in range(args.warmup):
            flush()
            ctx.quantize_fp8(x, out=xq)
            ctx.dispatch_permuted_fp8(xq, idx_d, w_d, handle, out=fq)
        qt, dt = [], []
        for i in range(args.steps):
            flush()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record(stream)
            ctx.quantize_fp8(x, out=xq)
            e[1].record(stream)
            ctx.dispatch_permuted_fp8(xq, idx_d, w_d, handle, out=fq)
            e[2].record(stream)
            torch.cuda.synchronize()
            qt.append(e[0].elapsed_time(e[1]))
            dt.append(e[1].elapsed_time(e[2]))
        ctx.check()
        peak0, _ = measured_hbm_gbs()
        qb = tokens * (2 * H + rq)
        db = (tokens + pairs) * rq
        # quantisation fused into the dispatch: one pass from the bf16 tokens
        ot = []
        for i in range(args.warmup + args.steps):
            flush()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            e[0].record(stream)
            ctx.dispatch_permuted_quant(x, idx_d, w_d, handle, out=fq)
            e[1].record(stream)
            torch.cuda.synchronize()
            if i >= args.warmup:
                ot.append(e[0].elapsed_time(e[1]))
        ctx.check()
        # and into the receive layout (quantise + dispatch scatter in one pass)
        rq_recv = dict(recv_xq=torch.empty(copies, rq, dtype=torch.uint8, device="cuda"),
                       recv_src_rank=torch.empty(copies, dtype=torch.int32, device="cuda"),
                       recv_src_idx=torch.empty(copies, dtype=torch.int32, device="cuda"),
                       recv_topk_idx=torch.empty(copies, K, dtype=torch.int32, device="cuda"),
                       recv_topk_weights=torch.empty(copies, K, dtype=torch.float32, device="cuda"))
        st_ = []
        for i in range(args.warmup + args.steps):
            flush()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            e[0].record(stream)
            ctx.dispatch_quant(x, idx_d, w_d, handle, out=rq_recv)
            e[1].record(stream)
            torch.cuda.synchronize()
            if i >= args.warmup:
                st_.append(e[0].elapsed_time(e[1]))
        ctx.check()
        del rq_recv
        sm_ = statistics.median(st_)
        sb_ = tokens * 2 * H + copies * rq
        qm, dm = statistics.median(qt), statistics.median(dt)
        om = statistics.median(ot)
        ob = tokens * 2 * H + pairs * rq
        fp8 = {"row_bytes": rq,
               "quantize": {"us": round(qm * 1e3, 2), "algo_bytes": qb, "GBps": round(qb / qm / 1e6, 1),
                            "frac": round(qb / qm / 1e6 / peak0, 3)},
               "dispatch_permuted_fp8": {"us": round(dm * 1e3, 2), "algo_bytes": db, "GBps": round(db / dm / 1e6, 1),
                                         "frac": round(db / dm / 1e6 / peak0, 3)},
               "dispatch_permuted_quant": {"us": round(om * 1e3, 2), "algo_bytes": ob,
                                           "GBps": round(ob / om / 1e6, 1), "frac": round(ob / om / 1e6 / peak0, 3),
                                           "what": "quantise + dispatch into the permuted layout in one pass"},
               "dispatch_quant": {"us": round(sm_ * 1e3, 2), "algo_bytes": sb_, "GBps": round(sb_ / sm_ / 1e6, 1),
                                  "frac": round(sb_ / sm_ / 1e6 / peak0, 3),
                                  "what": "quantise + dispatch scatter into the receive layout in one pass"}}
        del xq, fq

    # ---- low-latency decode layer -------------------------------------------------
    ll = None
    if not args.no_ll:
        dw = inputs.WORKLOADS["decode"]
        d_idx, d_w = inputs.make_routing(dw, seed + 7)
        d_x = inputs.make_x(dw, seed + 7, device="cuda")
        d_idx_d, d_w_d = d_idx.cuda(), d_w.cuda()
        buf = LLBuffer(dw.R, dw.E, dw.K, dw.T, dw.H, dw.ll_cap)
        pk = buf.alloc_packed()
        buf.dispatch(d_x, d_idx_d, out=pk)
        # identity expert: y = bf16(code * scale) (outside the timed layer)
        y_ll = torch.empty(pk["packed_x"].shape, dtype=torch.bfloat16, device="cuda")
        for d in range(dw.R):  # slab by slab to bound the fp32 temporaries
            codes = pk["packed_x"][d].view(torch.float8_e4m3fn).float()
            y_ll[d] = (codes * pk["packed_scales"][d].repeat_interleave(128, dim=-1)).to(torch.bfloat16)
        del codes
        d_out = torch.empty(dw.R, dw.T, dw.H, dtype=torch.bfloat16, device="cuda")
        for _ in range(args.warmup):
            flush()
            buf.dispatch(d_x, d_idx_d, out=pk)
            buf.combine(y_ll, d_idx_d, d_w_d, pk, out=d_out)
        buf.check()
        lev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush()
            lev[i][0].record(stream)
            buf.send(d_x, d_idx_d, out=pk)
            lev[i][1].record(stream)
            buf.recv(pk)
            lev[i][2].record(stream)
            buf.combine(y_ll, d_idx_d, d_w_d, pk, out=d_out)
            lev[i][3].record(stream)
        torch.cuda.synchronize()
        buf.check()
        lname = ["ll_send", "ll_recv", "ll_combine"]
        # each kernel alone: L2 flushed (and its dirty lines written back)
        # right before it, so that no kernel pays for the previous one's
        # write-backs nor gains from its lines still in L2
        iso = {n: [] for n in lname}
        for i in range(args.warmup + args.steps):
            for j, n in enumerate(lname):
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                if j == 0:
                    buf.send(d_x, d_idx_d, out=pk)
                elif j == 1:
                    buf.recv(pk)
                else:
                    buf.combine(y_ll, d_idx_d, d_w_d, pk, out=d_out)
                e1.record(stream)
                torch.cuda.synchronize()
                if i >= args.warmup:
                    iso[n].append(e0.elapsed_time(e1))
        buf.check()
        layer_instrumented_us = statistics.median(e[0].elapsed_time(e[3]) for e in lev) * 1e3
        # the layer alone, events only at its ends: the per-kernel events above
        # sit between the programmatic-dependent launches and serialise them
        lay_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush()
            lay_ev[i][0].record(stream)
            buf.send(d_x, d_idx_d, out=pk)
            buf.recv(pk)
            buf.combine(y_ll, d_idx_d, d_w_d, pk, out=d_out)
            lay_ev[i][1].record(stream)
        torch.cuda.synchronize()
        buf.check()
        layer_us = statistics.median(e[0].elapsed_time(e[1]) for e in lay_ev) * 1e3
        # the same layer captured once in a CUDA graph and replayed (static shapes,
        # no host sync, no allocation inside the layer)
        graph_us = None
        try:
            gs = torch.cuda.Stream()
            gs.wait_stream(stream)
            with torch.cuda.stream(gs):
                buf.dispatch(d_x, d_idx_d, out=pk)  # warm the side stream
                buf.combine(y_ll, d_idx_d, d_w_d, pk, out=d_out)
            gs.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=gs):
                buf.dispatch(d_x, d_idx_d, out=pk)
                buf.combine(y_ll, d_idx_d, d_w_d, pk, out=d_out)
            torch.cuda.synchronize()
            gt = []
            for i in range(args.steps + 2):
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                graph.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                if i >= 2:
                    gt.append(e0.elapsed_time(e1))
            buf.check()
            graph_us = round(statistics.median(gt) * 1e3, 2)
            del graph
        except Exception as exc:  # reported, not hidden
            graph_us = f"capture failed: {exc}"
        # dual-microbatch overlap: two decode microbatches, each with its own
        # buffer, packed outputs and result, on two streams at once (the same
        # tokens twice, so that the identity expert's y serves both)
        dual = None
        try:
            buf2 = LLBuffer(dw.R, dw.E, dw.K, dw.T, dw.H, dw.ll_cap)
            pk2 = buf2.alloc_packed()
            d_out2 = torch.empty_like(d_out)
            streams = (torch.cuda.Stream(), torch.cuda.Stream())
            lanes = ((buf, pk, d_out), (buf2, pk2, d_out2))

            def dual_layer():
                for st_, (b_, p_, o_) in zip(streams, lanes):
                    st_.wait_stream(stream)
                    with torch.cuda.stream(st_):
                        b_.dispatch(d_x, d_idx_d, out=p_)
                        b_.combine(y_ll, d_idx_d, d_w_d, p_, out=o_)
                for st_ in streams:
                    stream.wait_stream(st_)

            for _ in range(args.warmup):
                flush()
                dual_layer()
            dt_ = []
            for i in range(args.steps):
                flush()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                dual_layer()
                e1.record(stream)
                torch.cuda.synchronize()
                dt_.append(e0.elapsed_time(e1))
            buf.check()
            buf2.check()
            if not torch.equal(d_out.view(torch.int16), d_out2.view(torch.int16)):
                raise RuntimeError("the two microbatches disagree")
            two_us = statistics.median(dt_) * 1e3
            dual = {"us_two_layers": round(two_us, 2), "us_per_layer": round(two_us / 2, 2),
                    "how": "two decode microbatches (send, receive, combine each) on two streams at once"}
            # the same two overlapped layers captured once in a CUDA graph (the
            # streams fork from and join the capture stream) and replayed
            try:
                gs2 = torch.cuda.Stream()
                gs2.wait_stream(stream)
                torch.cuda.synchronize()
                g2 = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g2, stream=gs2):
                    cap = torch.cuda.current_stream()
                    for st_, (b_, p_, o_) in zip(streams, lanes):
                        st_.wait_stream(cap)
                        with torch.cuda.stream(st_):
                            b_.dispatch(d_x, d_idx_d, out=p_)
                            b_.combine(y_ll, d_idx_d, d_w_d, p_, out=o_)
                    for st_ in streams:
                        cap.wait_stream(st_)
                torch.cuda.synchronize()
                gt2 = []
                for i in range(args.steps + 2):
                    flush()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    g2.replay()
                    e1.record(stream)
                    torch.cuda.synchronize()
                    if i >= 2:
                        gt2.append(e0.elapsed_time(e1))
                buf.check()
                buf2.check()
                if not torch.equal(d_out.view(torch.int16), d_out2.view(torch.int16)):
                    raise RuntimeError("the two microbatches disagree (graph)")
                dual["us_per_layer_cuda_graph"] = round(statistics.median(gt2) * 1e3 / 2, 2)
                del g2
            except Exception as exc:  # reported, not hidden
                dual["us_per_layer_cuda_graph"] = f"capture failed: {exc}"
            del buf2, pk2, d_out2
        except Exception as exc:  # reported, not hidden
            dual = f"failed: {exc}"
        # the pages' low-latency monitoring figures: the signal-wait distribution
        # (count slots, one traced layer) and the buffer utilisation
        waits = None
        try:
            trace = torch.zeros(dw.E, dw.R, dtype=torch.int64, device="cuda")
            buf.trace_waits(trace)
            flush()
            buf.dispatch(d_x, d_idx_d, out=pk)
            buf.combine(y_ll, d_idx_d, d_w_d, pk, out=d_out)
            torch.cuda.synchronize()
            buf.trace_waits(None)
            buf.check()
            tw = trace.flatten().double().cpu() / 1e3
            waits = {"p50_us": round(float(tw.quantile(0.5)), 2), "p99_us": round(float(tw.quantile(0.99)), 2),
                     "max_us": round(float(tw.max()), 2),
                     "what": "per (expert, source): receive CTA start -> its counts read (publisher wait included)"}
        except Exception as exc:  # reported, not hidden
            waits = f"failed: {exc}"
        slot_util = round(float(pk["packed_recv_count"].sum()) / (dw.E * dw.R * dw.ll_cap), 4)
        d_pairs = int((d_idx >= 0).sum())
        lbytes = ll_algo_bytes(dw.H, dw.R * dw.T, d_pairs)
        peak, _ = measured_hbm_gbs()
        layer_bytes = sum(lbytes.values())
        ll = {"workload": "decode", "R": dw.R, "T": dw.T, "H": dw.H, "cap": dw.ll_cap,
              "us_per_layer": round(layer_us, 2),
              # the layer as one unit: per-kernel fractions move bytes between
              # kernels (a kernel's dirty lines are written back during the next)
              "layer": {"algo_bytes": layer_bytes, "GBps": round(layer_bytes / (layer_us * 1e-6) / 1e9, 1),
                        "frac": round(layer_bytes / (layer_us * 1e-6) / 1e9 / peak, 3)},
              "us_per_layer_with_kernel_events": round(layer_instrumented_us, 2),
              "us_per_layer_cuda_graph": graph_us,
              "dual_microbatch_overlap": dual,
              "signal_wait": waits, "slot_utilisation": slot_util,
              "kernels": {n: kernel_entry([e[j].elapsed_time(e[j + 1]) for e in lev], lbytes[n], peak)
                          for j, n in enumerate(lname)},
              "kernels_isolated": {n: kernel_entry(iso[n], lbytes[n], peak) for n in lname},
              "kernels_isolated_how": "each kernel with L2 flushed and written back right before it "
                                      "(the chained figures above are the layer's own)",
              "l2": L2_DESC}
        del y_ll, pk, buf

    # ---- the other workloads: skewed (normal + LL microbatches) and hierarchical ----
    extra = {}
    if w.name == "prefill" and not args.tokens and not args.no_extra_workloads:
        ksteps, kwarm = min(args.steps, 10), max(3, min(args.warmup, 5))
        for name, fn, wl in (("skewed", normal_leg, inputs.WORKLOADS["skewed"]),
                             ("skewed_ll", ll_microbatch_leg, inputs.WORKLOADS["skewed"]),
                             ("hier", normal_leg, inputs.WORKLOADS["hier"])):
            try:
                extra[name] = fn(torch, wl, seed + 3, ksteps, kwarm, flush)
                extra[name]["steps"], extra[name]["warmup"] = ksteps, kwarm
            except Exception as exc:  # reported, not hidden
                extra[name] = f"failed: {exc}"
            torch.cuda.empty_cache()

    clocks = sampler.stop()

    # ---- end to end through the public API with host buffers ------------------------
    # Every step copies its inputs (x, topk_idx, topk_weights) from pinned host
    # memory and its output back, inside the timed region.  Steps are pipelined
    # the way a serving loop would run them: the inputs of step k+1 go up on a
    # copy stream and the output of step k-1 comes down on another while step k
    # computes (two slots of device inputs and outputs).
    e2e = None
    if not args.no_e2e:
        x_h = x.cpu().pin_memory()
        i_h = topk_idx.pin_memory()
        w_h = topk_w.pin_memory()
        out_h = [torch.empty(R, T, H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        x_dev = [torch.empty_like(x) for _ in range(2)]
        i_dev = [torch.empty_like(idx_d) for _ in range(2)]
        w_dev = [torch.empty_like(w_d) for _ in range(2)]
        out_dev = [torch.empty_like(out) for _ in range(2)]
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()
        in_ready = [ev() for _ in range(2)]
        done = [ev() for _ in range(2)]
        copied = [ev() for _ in range(2)]
        for e_ in done + copied:
            e_.record(stream)

        def upload(k):
            sl = k % 2
            with torch.cuda.stream(up):
                up.wait_event(done[sl])
                x_dev[sl].copy_(x_h, non_blocking=True)
                i_dev[sl].copy_(i_h, non_blocking=True)
                w_dev[sl].copy_(w_h, non_blocking=True)
                in_ready[sl].record(up)

        def compute(k):
            sl = k % 2
            stream.wait_event(in_ready[sl])
            stream.wait_event(copied[sl])
            ctx.get_dispatch_layout(i_dev[sl], nodes=hier, out=lay)
            ctx.notify_dispatch(i_dev[sl], lay, handle=handle)
            if hier:
                ctx.dispatch_hier(x_dev[sl], i_dev[sl], w_dev[sl], handle, out=recv, staging=staging)
            else:
                ctx.dispatch(x_dev[sl], i_dev[sl], w_dev[sl], handle, out=recv)
            ctx.permute(handle, recv, out=perm)
            ctx.combine(handle, perm["permuted_x"], i_dev[sl], w_dev[sl], out=out_dev[sl], hier=hier)
            done[sl].record(stream)

        def download(k):
            sl = k % 2
            with torch.cuda.stream(down):
                down.wait_event(done[sl])
                out_h[sl].copy_(out_dev[sl], non_blocking=True)
                copied[sl].record(down)

        # the same step without a host wait, one CUDA graph per input slot
        # (worst-case receive buffers, row totals read on the device): the host
        # never blocks, so copies and steps are queued well ahead
        rmax, pmax, smax = ctx.max_rows
        n_recv = ctx.alloc_recv(rmax)
        n_perm = dict(permuted_x=torch.empty(pmax, H, dtype=torch.bfloat16, device="cuda"),
                      perm_src_row=torch.empty(pmax, dtype=torch.int32, device="cuda"))
        n_stage = None
        if hier:
            n_stage = dict(staging=torch.empty(smax, H, dtype=torch.bfloat16, device="cuda"),
                           stage_src_rank=torch.empty(smax, dtype=torch.int32, device="cuda"),
                           stage_src_idx=torch.empty(smax, dtype=torch.int32, device="cuda"))
        n_lay = {k: torch.empty_like(v) for k, v in lay.items()}
        n_h = ctx.alloc_handle()

        def nowait_step(sl):
            ctx.get_dispatch_layout(i_dev[sl], nodes=hier, out=n_lay)
            ctx.notify_dispatch(i_dev[sl], n_lay, handle=n_h, wait=False)
            if hier:
                ctx.dispatch_hier(x_dev[sl], i_dev[sl], w_dev[sl], n_h, out=n_recv, staging=n_stage)
            else:
                ctx.dispatch(x_dev[sl], i_dev[sl], w_dev[sl], n_h, out=n_recv)
            ctx.permute(n_h, n_recv, out=n_perm)
            ctx.combine(n_h, n_perm["permuted_x"], i_dev[sl], w_dev[sl], out=out_dev[sl], hier=hier)

        graphs = []
        for sl in range(2):
            x_dev[sl].copy_(x)
            i_dev[sl].copy_(idx_d)
            w_dev[sl].copy_(w_d)
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                nowait_step(sl)
            stream.wait_stream(side)
            torch.cuda.synchronize()
            cg = torch.cuda.CUDAGraph()
            with torch.cuda.graph(cg):
                nowait_step(sl)
            graphs.append(cg)

        def compute_graph(k):
            sl = k % 2
            stream.wait_event(in_ready[sl])
            stream.wait_event(copied[sl])
            graphs[sl].replay()
            done[sl].record(stream)

        def run(nsteps, step_fn):
            upload(0)
            for k in range(nsteps):
                if k + 1 < nsteps:
                    upload(k + 1)
                step_fn(k)
                download(k)
            stream.wait_event(copied[(nsteps - 1) % 2])

        # a serving loop's steady state: enough steps that the pipeline's fill
        # (the first upload) and drain (the last download) are a small share
        e2e_steps = max(args.steps, 100)

        def timed(step_fn):
            run(max(2, args.warmup), step_fn)
            torch.cuda.synchronize()
            flush()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run(e2e_steps, step_fn)
            e1.record(stream)
            torch.cuda.synchronize()
            ctx.check()
            return max_over_ranks(e0.elapsed_time(e1) / e2e_steps)

        e_ms_eager = timed(compute)
        e_ms = timed(compute_graph)
        # the graph path's output equals the eager step's, bit for bit
        if not torch.equal(out_h[(e2e_steps - 1) % 2].view(torch.int16), out.cpu().view(torch.int16)):
            raise RuntimeError("end-to-end output differs from the device-resident step")
        del graphs, n_recv, n_perm, n_stage
        # plain copy rates of this machine, for context
        def rate(fn, nbytes):
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            fn()
            a1.record(stream)
            torch.cuda.synchronize()
            return round(nbytes / a0.elapsed_time(a1) / 1e6, 1)
        h2d_gbps = rate(lambda: x_dev[0].copy_(x_h, non_blocking=True), x.numel() * 2)
        d2h_gbps = rate(lambda: out_h[0].copy_(out_dev[0], non_blocking=True), out.numel() * 2)
        h2d = x.numel() * 2 + topk_idx.numel() * 8 + topk_w.numel() * 4
        e2e = {"value": total_tokens / (e_ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": out.numel() * 2, "ms_per_step": round(e_ms, 4),
               "pipelined": "inputs of step k+1 up and output of step k-1 down while step k computes",
               "steps": e2e_steps,
               "step": "no-wait notify, each step one CUDA graph replay (the host never blocks)",
               "with_host_wait": {"value": total_tokens / (e_ms_eager / 1e3), "ms_per_step": round(e_ms_eager, 4),
                                  "step": "eager calls, notify waiting on the host for the counts"},
               "h2d_GBps": h2d_gbps, "d2h_GBps": d2h_gbps}
        del x_dev, i_dev, w_dev, out_dev, out_h

    if rank != 0:
        epdist.shutdown()
        return 0

    # ---- roofline of the dominant kernel ------------------------------------------
    peak, peak_kind = measured_hbm_gbs()
    ab = algo_bytes(H, K, tokens, copies, pairs, handle.num_stage_rows if hier else 0)
    med = {n: statistics.median(per[n]) for n in names}
    kernels = {}
    for n in names:
        entry = {"us": round(med[n] * 1e3, 2), "p10_us": round(pct(per[n], 0.1) * 1e3, 2),
                 "p90_us": round(pct(per[n], 0.9) * 1e3, 2)}
        if n in ab:
            gbs = ab[n] / (med[n] * 1e-3) / 1e9
            entry.update({"algo_bytes": ab[n], "GBps": round(gbs, 1), "frac": round(gbs / peak, 3)})
        kernels[n] = entry
    dom = max(ab, key=lambda n: med[n])
    dom_avg_ms = sum(per[dom]) / len(per[dom])
    achieved = ab[dom] / (dom_avg_ms * 1e-3) / 1e9
    tr = TRAFFIC.get((w.name, dom)) if not args.tokens else None
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured"
                else "fallback 6.8 TB/s", "unit": "GB/s", "frac": round(achieved / peak, 4),
                "algo_bytes_per_launch": ab[dom], "traffic": tr["bytes"] if tr else None,
                "traffic_case": tr["case"] if tr else None}

    cpu = None
    if not args.no_cpu and world == 1:  # the CPU baseline is timed at N=1 only
        cpu = oracle_sample(w, budget_s=25.0, min_s=10.0)
        try:
            cpu["all_cores"] = oracle_parallel(w, 8.0)
        except Exception as exc:
            cpu["all_cores"] = f"unavailable: {exc}"

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "R": R, "E": E, "K": K, "T": T, "H": H, "num_channels": C,
                   "num_nodes": w.num_nodes, "router": w.router, "tokens_per_step_per_gpu": tokens,
                   "copies": copies, "pairs": pairs,
                   "l2": L2_DESC + "; every step's inputs exceed L2 anyway",
                   "timing": "CUDA events on the launching stream, per step, mean over steps, max over ranks"},
        "effective_GBps": round(sum(ab.values()) / (sum(med[n] for n in ab) * 1e-3) / 1e9, 1),
        "kernels": kernels,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": sum(launches.values()) * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": round(wall, 4),
        "ll_decode": ll,
        "fused_path": fused,
        "expert_aligned": aligned,
        "graph": nw_graph,
        "fp8_rows": fp8,
        "skewed": extra.get("skewed"),
        "skewed_ll": extra.get("skewed_ll"),
        "hier": extra.get("hier"),
    }
    print(json.dumps(add_nominal_pct(line)), flush=True)
    epdist.shutdown()
    return 0


if __name__ == "__main__":
    sys.exit(main())
