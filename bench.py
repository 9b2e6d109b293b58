#!/usr/bin/env python
"""Medusa decode-step benchmark: verifies/s at the Vicuna-7B shape on one B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one pass of the whole hot path over one batch: Medusa heads + top-k,
tree expansion, tree attention over KV cache + tree, lm_head verification with
typical acceptance, KV commit of the accepted path.  One "verify" is one
request's step (a step processes B requests).  Inputs are seeded synthetic
tensors of the workload's shapes (random-init weights), resident in HBM.
The per-step working set (1.79 GB at the 7B shape) exceeds the 126 MB L2, so
no flush is added between steps.  Under torchrun every rank runs an
independent replica (weak scaling); rank 0 prints one JSON line.

--impl reference times the CPU oracle (fp64 numpy, test infrastructure) on
the host cores, on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Medusa decode-step verifies/sec at 7B shape; % of HBM/tensor roofline"
UNIT = "verifies/s"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="vicuna7b")
    ap.add_argument("--temperature", type=float, default=0.7)
    ap.add_argument("--unroll", type=int, default=20, help="steps per captured CUDA graph")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=30.0)
    ap.add_argument("--tree", default=None,
                    help="replace the workload's tree: 'cartesian:k1,k2,...' (full product tree) or "
                         "'seeded:N[:f0,f1,...]' (seeded sparse tree of N nodes, per-depth fan-out bounds)")
    return ap.parse_args()


def select_workload(args):
    """The named workload, with its candidate tree replaced when --tree is given."""
    import dataclasses
    import synth
    wl = synth.WORKLOADS[args.workload]
    if not args.tree:
        return wl
    kind, _, rest = args.tree.partition(":")
    if kind == "cartesian":
        tree = ("cartesian", tuple(int(x) for x in rest.split(",")))
    elif kind == "seeded":
        n, _, fan = rest.partition(":")
        tree = ("seeded", int(n), tuple(int(x) for x in fan.split(",")) if fan else synth.TREE64[2])
    else:
        raise SystemExit(f"--tree: unknown kind {kind!r}")
    if kind == "cartesian" and len(tree[1]) > wl.K:
        raise SystemExit("--tree: deeper than the workload's number of heads")
    return dataclasses.replace(wl, name=f"{wl.name}/tree={args.tree}", tree=tree)


def max_over_ranks(x: float, device, ws: int) -> float:
    """The largest of every rank's x (a timed region's length: the job ends with its slowest rank)."""
    if ws <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank: int, ms: float, ws: int) -> float:
    """Whole-job units per second: every rank processed units_per_rank in at most ms."""
    return units_per_rank * ws / (ms / 1e3)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- roofline bookkeeping

def step_bytes(wl, T):
    """Algorithmic bytes of each stage of one step (weights + KV + activations + outputs)."""
    es = 2 if wl.dtype == "bf16" else 4
    B, H, V, K, Hq, Hkv, D = wl.B, wl.H, wl.V, wl.K, wl.Hq, wl.Hkv, wl.D
    L = sum(wl.kv_lens())
    heads = es * (K * H * H + K * H + K * V * H + B * H) + B * K * H * es * 2
    attn = es * (2 * L * Hkv * D + B * T * Hq * D + 2 * B * T * Hkv * D) + 4 * B * T * Hq * D
    verify = es * (V * H + B * T * H) + 4 * B * T
    return {"heads": heads, "attention": attn, "verify": verify}


def traffic_from_profile(kernel_key: str):
    """DRAM bytes per launch recorded from an ncu capture, if the kernel source is unchanged since."""
    path = os.path.join(ROOT, "profiles", f"{kernel_key}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    s = re.search(r"source_sha256:\s*([0-9a-f]+)", txt)
    src = re.search(r"source_file:\s*(\S+)", txt)
    if not (m and s and src):
        return None
    cur = hashlib.sha256(open(os.path.join(ROOT, src.group(1)), "rb").read()).hexdigest()
    return float(m.group(1)) if cur.startswith(s.group(1)) else None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d.get("hbm_gbs", 6400.0), d.get("bf16_tflops", 1800.0), "measured"
    return 6400.0, 1800.0, "fallback"


def workload_config(wl, T, tau, ws):
    """The workload keys both arms report."""
    return {"workload": wl.name, "tree": "%s %s" % (wl.tree[0], wl.tree[1:]), "batch": wl.B, "hidden": wl.H, "vocab": wl.V, "heads": wl.K, "tree_nodes": T,
            "q_heads": wl.Hq, "kv_heads": wl.Hkv, "head_dim": wl.D, "kv_len": wl.L, "temperature": tau,
            "inputs": "planted accept path", "parallelism": f"replicas x{ws}"}


# ----------------------------------------------------------------------------- our arm

def pct(xs, q):
    """q-th percentile (nearest rank) of a non-empty list."""
    s = sorted(xs)
    return s[min(len(s) - 1, max(0, int(math.ceil(q / 100.0 * len(s))) - 1))]


def run_ours(args, ws, rank, local):
    import torch
    import torch.distributed as dist

    import medusa_head_speculative_04_b300 as mb
    import synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = select_workload(args)
    inp = synth.make_inputs(wl, dev, variant="plant")
    T = inp.T
    step = mb.MedusaStep(inp.choices, wl.B, wl.H, wl.V, wl.K, wl.Hq, wl.Hkv, wl.D, wl.Lmax, wl.k_needed(),
                         inp.dtype, device=dev, kv_len_hint=max(wl.kv_lens()), keep_node_stats=False)
    kc, vc = inp.k_cache.clone(), inp.v_cache.clone()
    kv_len0 = inp.kv_len.clone()
    kl = kv_len0.clone()
    root = inp.root.clone()
    tau = args.temperature
    s = torch.cuda.Stream(dev)

    ev_pairs = []

    def one_step(timed_events=False):
        kl.copy_(kv_len0)                       # every step starts from the same prefix
        step.root.copy_(root)
        if timed_events:
            e = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(5)]
            e[0].record()
        step.heads(inp.h, inp.W1, inp.b1, inp.W2)
        if timed_events:
            e[1].record()
        step.build(kl)
        step.attention(inp.q, inp.k_new, inp.v_new, kc, vc, kl)
        if timed_events:
            e[2].record()
        # verification, acceptance and the KV commit of the winner (one launch sequence)
        step.verify_commit(inp.X, inp.lm_head, inp.k_new, inp.v_new, kc, vc, kl, tau, wl.posterior_threshold,
                           wl.posterior_alpha)
        if timed_events:
            e[3].record()
            e[4].record()
            ev_pairs.append(e)

    # eager warm-up (function attributes, tensor maps), then graphs
    with torch.cuda.stream(s):
        one_step()
    torch.cuda.synchronize()
    n0 = mb.kernel_launches()
    g1 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1, stream=s):
        one_step()
    launches_per_step = mb.kernel_launches() - n0
    # steps per timed graph: at least two replays inside the timed region
    S = max(1, min(args.unroll, args.steps // 2))
    gS = torch.cuda.CUDAGraph()          # the timed graph: steps back to back, nothing in between
    with torch.cuda.graph(gS, stream=s):
        for _ in range(S):
            one_step()
    gE = torch.cuda.CUDAGraph()          # the same steps with events between the stages
    with torch.cuda.graph(gE, stream=s):
        for _ in range(S):
            one_step(timed_events=True)
    reps, rem = divmod(args.steps, S)

    # the clock sampler starts first (its first sample takes a moment), then the
    # warm-up: the timed graph itself (its first replay uploads it), then single
    # steps, right before the timed region, so the GPU does not idle between them
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    warm = max(3, args.warmup)
    warm_steps = max(1, warm // S) * S + max(1, warm % S)
    with torch.cuda.stream(s):
        for _ in range(max(1, warm // S)):
            gS.replay()
        for _ in range(max(1, warm % S)):
            g1.replay()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    with torch.cuda.stream(s):
        start.record()
        for _ in range(reps):
            gS.replay()
        for _ in range(rem):
            g1.replay()
        end.record()
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    clocks = sampler.stop()
    ms_max = max_over_ranks(start.elapsed_time(end), dev, ws)
    status = int(step.dev_status.max().item())

    # stage breakdown and per-step spread: separate replays of the graph with events
    # between the stages (an event node between two kernels stops the second one from
    # starting before the first has finished, so these are not in the timed graph)
    n_ev = max(1, -(-200 // S))
    stage_ms = {"heads": [], "attention": [], "verify": []}
    step_ms = []
    with torch.cuda.stream(s):
        gE.replay()                             # upload / warm
    torch.cuda.synchronize()
    for _ in range(n_ev):
        with torch.cuda.stream(s):
            gE.replay()
        torch.cuda.synchronize()
        for e in ev_pairs:
            stage_ms["heads"].append(e[0].elapsed_time(e[1]))
            stage_ms["attention"].append(e[1].elapsed_time(e[2]))
            stage_ms["verify"].append(e[2].elapsed_time(e[3]))
            step_ms.append(e[0].elapsed_time(e[4]))
    accept_hist = {}
    for a in step.accept_len.cpu().tolist():
        accept_hist[str(a)] = accept_hist.get(str(a), 0) + 1

    # the steady-state loop: the next step's candidates come from the heads on this
    # step's accepted tree rows (expand, attend, verify + accept, commit, heads on
    # the tree rows), timed as its own CUDA graph of the same step count
    def steady_step():
        kl.copy_(kv_len0)
        step.build(kl)
        step.attention(inp.q, inp.k_new, inp.v_new, kc, vc, kl)
        step.verify_commit(inp.X, inp.lm_head, inp.k_new, inp.v_new, kc, vc, kl, tau, wl.posterior_threshold,
                           wl.posterior_alpha)
        step.heads_from_tree(inp.X, inp.W1, inp.b1, inp.W2)
    with torch.cuda.stream(s):
        steady_step()                       # workspace of the tree heads, kernel attributes
    torch.cuda.synchronize()
    gT = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gT, stream=s):
        for _ in range(S):
            steady_step()
    with torch.cuda.stream(s):
        for _ in range(max(1, warm // S)):
            gT.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        t0.record()
        for _ in range(reps):
            gT.replay()
        t1.record()
    torch.cuda.synchronize()
    ms_s = t0.elapsed_time(t1) / max(1, reps * S)
    steady = {"value": round(wl.B / (ms_s / 1e3), 2), "unit": UNIT, "ms_per_step": round(ms_s, 5),
              "note": "steady-state loop: tree expansion from the previous step's accepted row, attention, "
                      "verification + acceptance, commit, then the heads on each request's accepted tree row "
                      "(medusa_heads_topk_tree) for the next step; same workload and step count"}

    # end-to-end through the public API: every step copies its inputs in from
    # pinned host memory and its results out.  The inputs of step i+1 upload on a
    # copy stream while step i runs (two device buffers, ordered by events).
    pin = lambda x: x.detach().cpu().pin_memory()
    host_in = {k: pin(getattr(inp, k)) for k in ("h", "X", "q", "k_new", "v_new")}
    host_root = pin(root)
    dev_bufs = [{k: getattr(inp, k).clone() for k in host_in} for _ in range(2)]
    root_bufs = [root.clone() for _ in range(2)]
    # accept_len, best_path, best_node, next_root, accepted_tokens share one buffer; each
    # step copies it to a staging buffer of its own, read back on a third stream while the
    # next step runs
    staged = [torch.empty_like(step.results) for _ in range(2)]
    host_out = [torch.empty(step.results.shape, dtype=step.results.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values()) + host_root.numel() * 4
    d2h = step.results.numel() * step.results.element_size()
    e2e_steps = max(200, min(args.steps, 500))  # enough steps that the first upload and last read-back amortise
    cs, ds = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    finished = [torch.cuda.Event() for _ in range(2)]
    read_back = [torch.cuda.Event() for _ in range(2)]

    def upload(buf):
        cs.wait_event(consumed[buf])          # the step that last read this buffer is done
        with torch.cuda.stream(cs):
            for k, v in host_in.items():
                dev_bufs[buf][k].copy_(v, non_blocking=True)
            root_bufs[buf].copy_(host_root, non_blocking=True)
            copied[buf].record(cs)

    def run_step(buf):
        d = dev_bufs[buf]
        kl.copy_(kv_len0)
        step.run(d["h"], inp.W1, inp.b1, inp.W2, inp.lm_head, d["X"], d["q"], d["k_new"], d["v_new"], kc,
                 vc, kl, tau, wl.posterior_threshold, wl.posterior_alpha, root=root_bufs[buf])
        staged[buf].copy_(step.results)

    # the serving form of the call: one CUDA graph of MedusaStep.run per input buffer
    # (the results' staging copy is captured as the step's epilogue)
    step_graphs = []
    for b in range(2):
        g = step.capture(dev_bufs[b]["h"], inp.W1, inp.b1, inp.W2, inp.lm_head, dev_bufs[b]["X"],
                         dev_bufs[b]["q"], dev_bufs[b]["k_new"], dev_bufs[b]["v_new"], kc, vc, kl, tau,
                         wl.posterior_threshold, wl.posterior_alpha, root=root_bufs[b],
                         prologue=lambda: kl.copy_(kv_len0), epilogue=lambda b=b: staged[b].copy_(step.results),
                         stream=s)
        step_graphs.append(g)

    def e2e_run(n, graphs, start_event=None):
        with torch.cuda.stream(s):
            for ev in consumed + read_back:
                ev.record(s)
        if start_event is not None:
            cs.wait_event(start_event)
        upload(0)
        for i in range(n):
            buf = i & 1
            if i + 1 < n:
                upload(buf ^ 1)
            s.wait_event(copied[buf])
            s.wait_event(read_back[buf])          # staging buffer of step i-2 has been read
            with torch.cuda.stream(s):
                if graphs:
                    step_graphs[buf].replay()
                else:
                    run_step(buf)
                consumed[buf].record(s)
                finished[buf].record(s)
            ds.wait_event(finished[buf])
            with torch.cuda.stream(ds):
                host_out[buf].copy_(staged[buf], non_blocking=True)
                read_back[buf].record(ds)
        s.wait_stream(ds)                         # the last read-back is inside the timed region

    def e2e_time(graphs):
        e2e_run(3, graphs)
        torch.cuda.synchronize()
        if ws > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
        e2e_run(e2e_steps, graphs, start_event=e0)
        with torch.cuda.stream(s):
            e1.record(s)
        torch.cuda.synchronize()
        return replica_throughput(e2e_steps * wl.B, max_over_ranks(e0.elapsed_time(e1), dev, ws), ws)

    e2e_value = e2e_time(graphs=True)
    e2e_eager = e2e_time(graphs=False)

    if rank != 0:
        return None

    value = replica_throughput(args.steps * wl.B, ms_max, ws)
    sb = step_bytes(wl, T)
    hbm, bf16, src = measured_peaks()
    heads_ms = statistics.mean(stage_ms["heads"]) if stage_ms["heads"] else None
    roof = None
    if heads_ms:
        ach = sb["heads"] / (heads_ms / 1e3) / 1e9
        roof = {"kernel": "medusa_heads_topk (the heads stage: W1 and W2 streams with the top-k)", "bound": "hbm",
                "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s", "frac": round(ach / hbm, 4),
                "peak_source": src, "algorithmic_bytes": sb["heads"],
                "traffic": traffic_from_profile("heads_vicuna7b") if wl.name == "vicuna7b" else None}
    stages = {}
    for k, v in stage_ms.items():
        if v:
            m = statistics.mean(v)
            stages[k] = {"ms": round(m, 4), "GB/s": round(sb[k] / (m / 1e3) / 1e9, 1),
                         "frac_hbm": round(sb[k] / (m / 1e3) / 1e9 / hbm, 4)}
    total_bytes = sum(sb.values())
    ms_step = ms_max / args.steps
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": max(3, args.warmup), "warmup_steps_run": warm_steps, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic (seeded, random-init weights)",
        "config": dict(workload_config(wl, T, tau, ws),
                       l2="per-step working set %.2f GB > 126 MB L2; no flush" % (total_bytes / 1e9),
                       timing=f"CUDA graphs of {S} steps, CUDA events; stage times from a separate replay with "
                              "events between stages"),
        "roofline": roof,
        "step_roofline": {"bytes": total_bytes, "frac_hbm": round(total_bytes / (ms_step / 1e3) / 1e9 / hbm, 4)},
        "stages": stages,
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "eager_value": round(e2e_eager, 2), "steps": e2e_steps,
                "note": "MedusaStep.run captured once per input buffer (MedusaStep.capture) and replayed; every "
                        "step's inputs copied in from pinned host memory (the next step's upload overlapped on a "
                        "copy stream) and its results copied out (staged on the device, read back on a third "
                        "stream while the next step runs); eager_value: the same loop with eager "
                        "MedusaStep.run calls"},
        "step_ms_percentiles": {
            "p50": round(pct(step_ms, 50), 5), "p99": round(pct(step_ms, 99), 5), "n": len(step_ms),
            "note": "per-step times from the event-instrumented replay (events between the stages cancel the "
                    "programmatic overlap of adjacent kernels, so these sit slightly above ms_per_step)"},
        "accept_len_hist": {"counts": accept_hist,
                            "note": "accepted tokens beyond the root per request; every timed step sees the same "
                                    "inputs, so each request's count repeats in every step"},
        "steady_state": steady,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "dev_status": status,
    }
    return out, inp, wl, step, kl


# ----------------------------------------------------------------------------- oracle timing

def oracle_sample(wl, inp, temperature, budget_s, max_steps):
    """Time the CPU oracle on full decode steps of the workload (fp64 numpy).

    ``inp`` holds the step's seeded inputs (on any device); they are copied to
    host fp64 arrays before the clock starts."""
    import numpy as np
    import torch
    import oracle
    try:
        from threadpoolctl import threadpool_info
        cores = max([d.get("num_threads", 1) for d in threadpool_info()] or [os.cpu_count()])
    except Exception:
        cores = os.cpu_count()
    f = lambda t: t.detach().to("cpu", torch.float64).numpy()
    args = [f(inp.h), f(inp.W1), f(inp.b1), f(inp.W2), f(inp.lm_head), f(inp.X), f(inp.q), f(inp.k_new),
            f(inp.v_new), f(inp.k_cache), f(inp.v_cache), inp.kv_len.cpu().numpy()]
    root = inp.root.cpu().numpy()
    times = []
    res = None
    t_all = time.perf_counter()
    while len(times) < max_steps:
        t0 = time.perf_counter()
        res = oracle.run_step(*args, inp.choices, wl.k_needed(), temperature, wl.posterior_threshold,
                              wl.posterior_alpha, root=root, u_bf16=(wl.dtype == "bf16"))
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all > budget_s:
            break
    per = sum(times) / len(times)
    return {"value": round(wl.B / per, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{len(times)} full decode step(s) of {wl.name} (B={wl.B}), fp64 numpy, "
                      f"{per:.2f} s/step"}, len(times), per, res


def parity_summary(wl, step, kv_len, res, temperature):
    """The timed step's discrete outputs against the oracle's step on the same inputs.

    Near-ties are the decisions whose oracle margin is below the float tolerance
    (top-k orders, acceptance tests); a mismatch there is allowed, anywhere else it
    is an error."""
    import numpy as np
    delta = 1e-3 if wl.dtype == "bf16" else 1e-5
    g = lambda t: t.detach().cpu().numpy().astype(np.int64)
    zmax = np.abs(res.head_logits).max(axis=-1)
    near_topk = int(np.sum(res.topk_margin < delta * np.maximum(1.0, zmax)))
    m = res.accept["margin"][:, 1:]
    if temperature > 0:
        near_acc = int(np.sum(m < delta / temperature))
    else:
        near_acc = int(np.sum(m < delta * max(1.0, float(np.abs(res.logits).max()))))
    mism = {"topk_ids": int(np.sum(g(step.topk_ids) != res.topk_ids)),
            "tree_tokens": int(np.sum(g(step.tokens) != res.tokens)),
            "accepted_tokens": int(np.sum(g(step.accepted_tokens) != res.accept["accepted_tokens"])),
            "kv_len": int(np.sum(g(kv_len) != res.kv_len))}
    for k in ("accept_len", "best_node", "best_path", "next_root"):
        mism[k] = int(np.sum(g(getattr(step, k)) != res.accept[k]))
    n_mism = sum(mism.values())
    return {"near_ties": near_topk + near_acc, "near_ties_topk": near_topk, "near_ties_accept": near_acc,
            "mismatches": n_mism, "mismatch_by_output": mism, "ok": n_mism == 0 or near_topk + near_acc > 0,
            "compared": "top-k ids, tree tokens, accept_len, best_node, best_path, accepted_tokens, next_root, "
                        "kv_len of the timed step against the oracle's step on the same inputs"}


def run_reference(args, ws, rank):
    if rank != 0:
        return None
    import torch
    import synth
    wl = select_workload(args)
    # inputs come from the seeded generator (on a GPU when there is one, as it is much
    # faster there); the oracle only ever sees host copies
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = synth.make_inputs(wl, gen_dev, variant="plant")
    cb, n, per, _ = oracle_sample(wl, inp, args.temperature, args.cpu_budget_s * 4, max(1, args.steps))
    return {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": ws,
            "steps": n, "warmup": 0, "ms_per_step": round(per * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": dict(workload_config(wl, len(inp.choices) + 1, args.temperature, ws),
                           timing="host wall clock (perf_counter) per oracle step"),
            "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse_args()
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend)
    if args.impl == "reference":
        out = run_reference(args, ws, rank)
        if out:
            print(json.dumps(out))
        return
    res = run_ours(args, ws, rank, local)
    if res is None:
        return
    out, inp, wl, step, kl = res
    if not args.no_cpu_baseline and rank == 0 and ws == 1:
        cb, _, _, res_o = oracle_sample(wl, inp, args.temperature, args.cpu_budget_s, 3)
        out["cpu_baseline"] = cb
        out["parity"] = parity_summary(wl, step, kl, res_o, args.temperature)
    else:
        out["cpu_baseline"] = None
    print(json.dumps(out))


if __name__ == "__main__":
    main()
