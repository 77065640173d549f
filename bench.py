#!/usr/bin/env python
"""Benchmark of the DFlash 2 drafter hot path on GB300.

Steps by workload (--workload):

* single-sequence decode (default qwen3_8b_ctx2048, also qwen3_8b_ctx32768):
  one step = a context append of `block` new target rows (taps -> FC ->
  hidden_norm -> every layer's K/V, written at the end of the context) and
  one block of `block` rows anchored after them (draft layers, head, draft
  tokens).  The context is prefilled with ctx - block rows; each step
  re-appends the last `block` rows at the same positions, so every step sees
  ctx context rows.  Unit: draft tokens/s.
* batched drafting (qwen3_8b_batch32_ctx4096): one step = one block of every
  sequence (each with ctx context rows).  Unit: draft tokens/s.
* prefill (qwen3_8b_prefill8192): one step = one append of `prefill` rows.
  Unit: context rows/s.

value: throughput with inputs and outputs resident in HBM (CUDA events on
the launching stream).  e2e: the same through the host-buffer API (pinned
host inputs in, outputs out, copies inside the timed region).  roofline: the
kernel with the largest device time in a profiled pass of the same steps.
cpu_baseline / --impl reference: the CPU oracle on a bounded sample.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME] [--others auto|on|off]

With the default workload on one GPU the line also carries "others": the
context-32768, batch-32 and prefill-8192 workloads of the same drafter, each
timed the same way (same steps and warm-up) on the same model.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

# torchrun starts every rank with one OpenMP thread; the reference arm does its
# work on rank 0 alone, so that rank takes the host's cores as a plain run does
# (the BLAS reads the count when numpy loads)
if (os.environ.get("TORCHELASTIC_RUN_ID") and os.environ.get("RANK", "0") == "0"
        and ("--impl=reference" in sys.argv
             or any(a == "--impl" and b == "reference" for a, b in zip(sys.argv, sys.argv[1:])))):
    os.environ["OMP_NUM_THREADS"] = str(os.cpu_count() or 1)

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "DFlash block latency ms & draft tokens/s; achieved HBM GB/s vs GB300 peak"
UNIT = "draft tokens/s"
FALLBACK_HBM_GBS = 6800.0


def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    """Dense f16/bf16 tensor TFLOP/s: the sustained (seconds-long, power-capped)
    cuBLAS bf16 figure, since the contractions run inside multi-millisecond
    steps; f16 and bf16 share one rate."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), "measured sustained"
    except Exception:
        return FALLBACK_BF16_TFLOPS_SUSTAINED, "fallback sustained"


def tc_flops_per_step(wl, kernel):
    """Algorithmic FLOPs (2 per multiply-add of the quantised definition) of
    the tensor-core kernels in one step of a many-row workload; the kernels
    run each 4-bit product as two f16 MMAs (hi + lo), which these figures do
    not count."""
    g = wl.geom
    H, I, L = g.hidden, g.intermediate, g.layers
    qd, kd = g.heads * g.head_dim, g.kv_heads * g.head_dim
    if step_kind(wl) == "prefill":
        n = wl.prefill
        return 2.0 * n * H * g.tap_width + 2.0 * n * (2 * L * kd) * H if kernel == "q4_tc" else 0.0
    if step_kind(wl) == "batch":
        rows, drafts = wl.n_seqs * g.block, wl.n_seqs * (g.block - 1)
        if kernel == "q4_tc":
            return 2.0 * rows * L * ((qd + 2 * kd) * H + H * qd + 2 * I * H + H * I)
        if kernel == "head_tc":
            return 2.0 * drafts * g.vocab * H
    return 0.0


def kernel_source_hash():
    h = hashlib.sha256()
    d = os.path.join(ROOT, "block_speculative_drafting_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        if f.endswith((".cu", ".cuh")):
            with open(os.path.join(d, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or
    None when there is none for this workload or the kernels changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d[workload][kernel]
        if e.get("source_hash") != kernel_source_hash():
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms (a timed
    region of a few hundred steps still holds several samples)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def wait_first(self, limit_s=5.0):
        """Until the first sample is in (nvidia-smi has initialised), at most
        limit_s: its start-up, if it overlapped the timed steps, could hold
        up this process's CUDA calls."""
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < limit_s:
            if self.proc.poll() is not None:
                break
            time.sleep(0.02)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.t:
            self.t.join(timeout=2)

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        inside = [r for r in rows if t0 - 0.03 <= r[0] <= t1 + 0.03] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside)}


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


APPEND_CHUNK = 4096  # host rows of taps generated and appended at a time when filling contexts


def step_kind(wl):
    """What one bench step of the workload is: 'decode' (append `block` rows
    + one block of one sequence), 'batch' (one block of every sequence) or
    'prefill' (one append of `prefill` rows)."""
    if wl.prefill:
        return "prefill"
    return "batch" if wl.n_seqs > 1 else "decode"


def step_units(wl):
    """(units per step, unit name) of the workload's metric."""
    g = wl.geom
    kind = step_kind(wl)
    if kind == "prefill":
        return wl.prefill, "context rows/s"
    return wl.n_seqs * (g.block - 1), UNIT


def oracle_step_timer(wl, weights, steps_wanted, budget_s):
    """Time the CPU oracle on a bounded sample of the workload's step.
    Returns (seconds per step of the FULL workload, samples timed, cores,
    what the sample was).  The oracle model build and context prefill are
    not timed; a sample covers one sequence (batch: one of n_seqs blocks,
    scaled by n_seqs) or 64 of the prefill rows (scaled by rows)."""
    from oracle import OracleModel, OracleSeq, block

    g = wl.geom
    kind = step_kind(wl)
    om = OracleModel(g, weights)
    osq = OracleSeq(om)
    if kind == "prefill":
        rows = 64
        taps = W.make_taps(g, rows, call_id=0)
        scale = wl.prefill / rows
        what = f"append of {rows} of the {wl.prefill} rows (rows are independent), scaled by {scale:g}"

        def one():
            osq.append(0, taps)
    else:
        pre = wl.ctx - g.block if kind == "decode" else 0
        for r0 in range(0, pre if kind == "decode" else wl.ctx, APPEND_CHUNK):
            n = min(APPEND_CHUNK, (pre if kind == "decode" else wl.ctx) - r0)
            osq.append(r0, W.make_taps(g, n, call_id=(0 if kind == "decode" else 1000) + r0 // APPEND_CHUNK))
        taps = W.make_taps(g, g.block, call_id=1)
        anchor = int(W.make_anchors(g, 1)[0])
        if kind == "decode":
            scale = 1.0
            what = f"full step (append {g.block} rows + one {g.block}-row block)"

            def one():
                osq.append(pre, taps)
                block(om, osq, anchor, wl.ctx, g.block)
        else:
            scale = float(wl.n_seqs)
            what = f"one of the {wl.n_seqs} sequences' {g.block}-row blocks, scaled by {wl.n_seqs}"

            def one():
                block(om, osq, anchor, wl.ctx, g.block)
    times = []
    t_start = time.perf_counter()
    while len(times) < steps_wanted:
        t0 = time.perf_counter()
        one()
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start + times[-1] > budget_s:
            break
    return statistics.median(times) * scale, len(times), cpu_threads(), what


def run_reference(args, wl):
    rank = env_int("RANK", 0)
    if rank != 0:
        return
    g = wl.geom
    weights = W.make_weights(g)
    # the reference arm's step: the oracle on a bounded sample of the
    # workload's step, scaled to the whole step; the counts are bounded so
    # the run ends in a few minutes
    sec, n, cores, what = oracle_step_timer(wl, weights, max(1, args.steps), budget_s=args.cpu_budget)
    units, unit = step_units(wl)
    value = units / sec
    sample = f"median of {n} sample(s): {what}, of {wl.name} on the CPU oracle; oracle build and context prefill untimed"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": args.gpus, "steps": n,
        "warmup": 0, "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded Gaussian weights and taps)",
        "config": {"workload": wl.name, "n_seqs": wl.n_seqs, "ctx": wl.ctx, "block": g.block,
                   "prefill": wl.prefill, "step": step_kind(wl)},
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def build_case(model, wl, dev):
    """The workload's step on the device (inputs resident) and through host
    buffers, with its description.  Returns a dict of callables and facts."""
    import torch

    g = wl.geom
    B = g.block
    kind = step_kind(wl)
    pin = lambda a: torch.from_numpy(a).pin_memory().numpy()  # noqa: E731
    if kind == "prefill":
        n = wl.prefill
        seq = model.new_sequence(n)
        taps_h = W.make_taps(g, n, call_id=80)
        taps_d = torch.from_numpy(taps_h).to(dev)
        taps_p = pin(taps_h)
        del taps_h
        return {
            "seqs": [seq],
            "step": lambda: model.ctx_append(seq, 0, taps_d),
            "step_host": lambda: model.ctx_append(seq, 0, taps_p),
            "h2d": int(taps_p.nbytes), "d2h": 0,
            "desc": f"ctx_append({n} rows at position 0)",
            "l2": f"inputs larger than L2 ({taps_d.numel() * 4 / 1e6:.0f} MB of taps + 71 MB of weights each step)",
        }
    S = wl.n_seqs
    pre = wl.ctx - B if kind == "decode" else wl.ctx
    seqs = []
    for s in range(S):
        seq = model.new_sequence(wl.ctx + 2 * B)
        for r0 in range(0, pre, APPEND_CHUNK):
            rows = min(APPEND_CHUNK, pre - r0)
            cid = r0 // APPEND_CHUNK if kind == "decode" else 1000 + 64 * s + r0 // APPEND_CHUNK
            model.ctx_append(seq, r0, W.make_taps(g, rows, call_id=cid))
        seqs.append(seq)
    anchors = W.make_anchors(g, S).astype(np.uint32)
    anchor_d = torch.from_numpy(anchors.astype(np.int32)).to(dev)
    logits_d = torch.empty((S, B - 1, g.vocab), dtype=torch.float32, device=dev)
    tok_d = torch.empty((S, B - 1), dtype=torch.int32, device=dev)
    logits_p = pin(np.empty((S, B - 1, g.vocab), dtype=np.float32))
    tok_p = pin(np.empty((S, B - 1), dtype=np.uint32))
    positions = [wl.ctx] * S
    if kind == "decode":
        taps_h = W.make_taps(g, B, call_id=1)
        taps_d = torch.from_numpy(taps_h).to(dev)
        taps_p = pin(taps_h)
        seq = seqs[0]

        def step():
            model.ctx_append(seq, pre, taps_d)
            model.block(seqs, anchor_d, positions, B, logits=logits_d, tokens=tok_d)

        def step_host():
            model.ctx_append(seq, pre, taps_p)
            model.block(seqs, anchors, positions, B, logits=logits_p, tokens=tok_p)

        return {"seqs": seqs, "step": step, "step_host": step_host,
                "h2d": int(taps_p.nbytes + anchors.nbytes), "d2h": int(logits_p.nbytes + tok_p.nbytes),
                "desc": f"ctx_append({B} rows) + block({B} rows)",
                "l2": "inputs larger than L2 (1.3 GB of weights streamed each step)"}
    return {
        "seqs": seqs,
        "step": lambda: model.block(seqs, anchor_d, positions, B, logits=logits_d, tokens=tok_d),
        "step_host": lambda: model.block(seqs, anchors, positions, B, logits=logits_p, tokens=tok_p),
        "h2d": int(anchors.nbytes), "d2h": int(logits_p.nbytes + tok_p.nbytes),
        "desc": f"block({S} sequences x {B} rows)",
        "l2": f"inputs larger than L2 ({S * wl.ctx * 8 * g.kv_heads * g.head_dim * g.layers / 1e9:.1f} GB of K/V "
              "+ 1.2 GB of weights each step)",
    }


def max_over_ranks(x, dist=None, device="cpu"):
    """The largest of every rank's `x` (a time of the timed region): the job
    takes as long as its slowest rank.  Without a process group, x itself."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, units_per_rank, seconds):
    """Units all ranks processed per second of the slowest rank (weak scaling:
    each rank runs the same workload as an independent replica)."""
    return world * units_per_rank / seconds


OTHER_WORKLOADS = ("qwen3_8b_ctx32768", "qwen3_8b_batch32_ctx4096", "qwen3_8b_prefill8192")


def measure(args, wl, model, dev, world, dist, clocks, weights, cpu_leg):
    """One workload's numbers on an existing model (the workloads share one
    geometry): the timed steps, the profiled pass, the host-buffer e2e and,
    when asked, the CPU oracle leg.  Returns the JSON fields of its line."""
    import torch

    g = wl.geom
    B = g.block
    units, unit = step_units(wl)
    t_setup = time.perf_counter()
    case = build_case(model, wl, dev)
    step, step_host = case["step"], case["step_host"]
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    setup_s = time.perf_counter() - t_setup

    def barrier():
        if dist:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    barrier()
    n0 = model.launch_count()
    # one event between steps as well: the per-step spread (p10 / p50 / p90)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    t_wall0 = time.time()
    evs[0].record(stream)
    for i in range(args.steps):
        step()
        evs[i + 1].record(stream)
    barrier()
    t_wall1 = time.time()
    launches = model.launch_count() - n0
    ms = evs[0].elapsed_time(evs[-1]) / args.steps
    per_step = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps))
    pct = {f"ms_p{q}": per_step[min(len(per_step) - 1, int(q / 100 * len(per_step)))] for q in (10, 50, 90)}
    clk = clocks.summary(t_wall0, t_wall1)
    ms = max_over_ranks(ms, dist, dev)
    value = job_throughput(world, units, ms * 1e-3)

    # profiled pass: the same steps with every launch bracketed by events
    model.profile_start()
    pe0, pe1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pe0.record(stream)
    for _ in range(args.steps):
        step()
    pe1.record(stream)
    torch.cuda.synchronize()
    prof = model.profile_stop()
    prof_ms = pe0.elapsed_time(pe1) / args.steps
    top = max(prof.items(), key=lambda kv: kv[1][1])
    name, (nl, tms, tbytes) = top
    achieved = tbytes / (tms * 1e-3) / 1e9  # GB/s, algorithmic bytes over device time
    peak, peak_kind = measured_peaks()
    step_bytes = sum(v[2] for v in prof.values()) / args.steps
    traffic = ncu_traffic(name, wl.name)
    flops = tc_flops_per_step(wl, name)
    if flops > 0:
        # a dense contraction on the tcgen05 tensor cores: tensor-bound
        tpeak, tkind = measured_tensor_peak()
        tach = flops * args.steps / (tms * 1e-3) / 1e12
        roofline = {"bound": "tensor", "kernel": name, "achieved": tach, "peak": tpeak, "unit": "TFLOP/s",
                    "frac": tach / tpeak, "peak_source": f"{tkind} (MEASURED_PEAKS.json bf16_tflops_sustained)",
                    "traffic": traffic, "algorithmic_flops_per_launch": flops * args.steps / nl,
                    "mma_work_factor": 2.0 if name == "q4_tc" else 1.0,
                    "avg_launch_us": tms / nl * 1e3, "launches_per_step": nl / args.steps}
    else:
        roofline = {"bound": "hbm", "kernel": name, "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                    if peak_kind == "measured" else "fallback 6800 GB/s",
                    "traffic": traffic, "algorithmic_bytes_per_launch": tbytes / nl,
                    "avg_launch_us": tms / nl * 1e3, "launches_per_step": nl / args.steps}
    kernels = {k: {"launches_per_step": v[0] / args.steps, "ms_per_step": v[1] / args.steps,
                   "share": v[1] / sum(x[1] for x in prof.values()), "GBps": v[2] / (v[1] * 1e-3) / 1e9}
               for k, v in sorted(prof.items(), key=lambda kv: -kv[1][1])}

    # end to end through the host-buffer API: pinned host inputs in, outputs
    # out, every copy inside the timed region
    for _ in range(max(1, args.warmup // 2)):
        step_host()
    barrier()
    k_e2e = args.steps
    t0 = time.perf_counter()
    for _ in range(k_e2e):
        step_host()
    barrier()
    e2e_s = (time.perf_counter() - t0) / k_e2e
    e2e_s = max_over_ranks(e2e_s, dist, dev)
    e2e = {"value": job_throughput(world, units, e2e_s), "unit": unit, "ms_per_step": e2e_s * 1e3,
           "h2d_bytes_per_step": case["h2d"], "d2h_bytes_per_step": case["d2h"]}

    cpu = None
    if cpu_leg:
        sec, n, cores, what = oracle_step_timer(wl, weights, 3, budget_s=args.cpu_budget)
        cpu = {"value": units / sec, "unit": unit, "cores": cores, "kind": "oracle",
               "sample": f"median of {n} sample(s): {what}, of {wl.name}; oracle build and context prefill untimed"}
    for sq in case["seqs"]:
        sq.close()
    return {
        "value": value, "unit": unit, "ms_per_step": ms,
        "config": {"workload": wl.name, "n_seqs": wl.n_seqs, "ctx": wl.ctx, "block": B,
                   "prefill": wl.prefill, "step": case["desc"], "parallelism": f"replicas x{world}",
                   "l2": case["l2"]},
        "block_latency_ms": ms, **pct, "hbm_gbs_step": step_bytes / (ms * 1e-3) / 1e9,
        "algorithmic_bytes_per_step": step_bytes, "profiled_ms_per_step": prof_ms,
        "roofline": roofline, "kernels": kernels, "e2e": e2e, "cpu_baseline": cpu,
        "gpu_launches": launches, "clocks": clk, "setup_s": setup_s,
    }


def run_ours(args, wl):
    import torch

    import block_speculative_drafting_gb300 as dfl

    rank, world, local = env_int("RANK", 0), env_int("WORLD_SIZE", 1), env_int("LOCAL_RANK", 0)
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist = dist_mod
        dist.init_process_group("nccl")
    weights = W.make_weights(wl.geom)
    model = dfl.Model(wl.geom, weights)
    dev = torch.device("cuda", local)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    clocks.wait_first()
    cpu_leg = rank == 0 and world == 1 and not args.no_cpu_baseline
    main_line = measure(args, wl, model, dev, world, dist, clocks, weights, cpu_leg)
    # the other full-size configurations of the same drafter, each timed the
    # same way on the same model, reported beside the headline (one GPU)
    others = {}
    want_others = args.others == "on" or (args.others == "auto" and world == 1 and wl.name == "qwen3_8b_ctx2048")
    if want_others:
        for other in OTHER_WORKLOADS:
            owl = W.WORKLOADS[other]
            if owl.geom != wl.geom:
                continue
            r = measure(args, owl, model, dev, world, dist, clocks, weights, False)
            others[other] = {k: r[k] for k in ("value", "unit", "ms_per_step", "ms_p10", "ms_p50", "ms_p90",
                                               "config", "roofline", "kernels", "e2e", "hbm_gbs_step",
                                               "gpu_launches", "clocks", "setup_s")}
    clocks.stop()
    if rank == 0:
        line = {
            "metric": METRIC, "value": main_line["value"], "unit": main_line["unit"], "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": main_line["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int4xint8 (f32 accumulate)",
            "data": "synthetic (seeded Gaussian weights N(0,0.02), taps N(0,1))",
            **{k: v for k, v in main_line.items() if k not in ("value", "unit", "ms_per_step")},
        }
        if others:
            line["others"] = others
        print(json.dumps(line), flush=True)
    model.close()
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="qwen3_8b_ctx2048", choices=sorted(W.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=60.0, help="seconds of CPU oracle steps at most")
    ap.add_argument("--others", default="auto", choices=["auto", "on", "off"],
                    help="also time the other full-size workloads of the same drafter (auto: with the default "
                         "workload on one GPU)")
    args = ap.parse_args()
    wl = W.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
