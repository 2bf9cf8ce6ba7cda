#!/usr/bin/env python3
"""Benchmark of the fused hyper-connection side steps.

Workload (default): long prefill -- 4 x 16384 = 65,536 tokens, hc = 4,
d = 5120, through 40 layers = 80 side steps, each side with its own seeded
parameters and its own N(0, 2) sublayer stand-in output.  One benchmark
"step" is one pass of all 80 side steps over the batch.  Metric: tokens/s
through the full depth (plus achieved HBM GB/s of the dominant kernel
against the measured HBM peak).  By default the sides run as the chain
fused across sides (hc_chain_begin + one hc_chain_side per side, outputs
equal to hc_block_step's bit for bit); the same sides as one hc_block_step
launch each are timed beside it (--path step makes them the headline).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own replica on its own GPU with
its own batch (weak scaling, no collective on the data path); the timing is
the max over ranks.  --impl reference times the CPU oracle on the host cores
on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np
import torch

import hyper_connection_residual_mixes_gb300 as hcg
from hyper_connection_residual_mixes_gb300 import inputs

HC, D = 4, 5120
TOKENS = 65536
LAYERS = 40
SIDES = 2 * LAYERS
MIX = (2 + HC) * HC
# algorithmic bytes of one side step: each input once, each output once
BYTES_PER_TOKEN = HC * D * 2 + D * 2 + HC * 4 + HC * D * 2 + D * 2 + HC * 4   # 102,432
BYTES_WEIGHTS = MIX * HC * D * 4 + 3 * 4 + MIX * 4 + D * 4                      # 1,986,668
FLOPS_PER_TOKEN = 2 * MIX * HC * D
L2_BYTES = 135_528_448
KERNEL_NAME = "hc_block_step"


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def rank_seed(base_seed, rank):
    """Each replica draws its own batch; rank 0 runs exactly the workload's seed."""
    return base_seed + 1000 * rank


def max_over_ranks(value, device="cpu"):
    """The slowest rank's time (the job ends when the last replica does)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            pk = json.load(fh)
        return float(pk["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def source_digest(unit):
    """Hash of one translation unit under csrc/ and of every local header it
    includes (recursively): the sources a kernel in that unit is built from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "hyper_connection_residual_mixes_gb300", "csrc")
    todo, seen = [os.path.join(csrc, unit)], set()
    while todo:
        path = os.path.normpath(todo.pop(0))
        if path in seen:
            continue
        seen.add(path)
        with open(path, "rb") as fh:
            text = fh.read()
        h.update(os.path.relpath(path, ROOT).encode())
        h.update(text)
        for line in text.decode().splitlines():
            line = line.strip()
            if line.startswith('#include "'):
                todo.append(os.path.join(os.path.dirname(path), line.split('"')[1]))
    return h.hexdigest()[:16]


def ncu_traffic_per_launch(n_tokens, path_kind="step"):
    """DRAM bytes per launch from the committed ncu summary, scaled by tokens;
    None when the kernel's sources have changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "hc_chain_side_traffic.json" if path_kind == "chain"
                        else "hc_block_step_traffic.json")
    unit = "hc_slices.cu" if path_kind == "chain" else "hc_block_cluster.cu"
    try:
        with open(path) as fh:
            rec = json.load(fh)
        digest = source_digest(unit)
    except Exception:
        return None
    if rec.get("source_digest") != digest:
        return None
    return int(rec["dram_bytes_per_token"] * n_tokens + rec.get("dram_bytes_fixed", 0))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.dev = device_index

    def _gpu_id(self):
        try:
            p = torch.cuda.get_device_properties(self.dev)
            return "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        except Exception:
            return str(self.dev)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self._gpu_id(), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "power_w_max": max(power) if power else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- our arm
WORKLOADS = {
    # name: (generator, base seed, description)
    "long_prefill": (None, 4, "B=4, T=16384 (65,536 tokens), 40 layers = 80 side steps"),
    "prefill": (inputs.prefill, 3, "B=1, T=8192, outliers, attention + FFN side"),
    "decode": (inputs.decode, 1, "B=128, T=1, attention + FFN side"),
}


def build_workload(device, rank, name="long_prefill"):
    gen, base_seed, _ = WORKLOADS[name]
    seed = rank_seed(base_seed, rank)
    if name == "long_prefill":
        case = inputs.long_prefill(device=device, seed=seed, materialize_f=False)
        fs = [inputs.long_prefill_f(s, case.n, case.d, device, seed) for s in range(SIDES)]
    else:
        case = gen(device=device, seed=seed)
        fs = case.fs
    return case, fs, seed


def run_chain(case, x0, pm0, fs, ys, pres, h_norm, states, events=None, stream=None,
              y_last=None, pre_last=None):
    """The 80 sides through the fused chain.  Side s reads state s and writes
    state s + 1 (two buffers in rotation); y of side s lands in ys[s % 2]
    (or y_last for the last side), its pre in pres."""
    P = case.params
    sides = len(P)
    hcg.hc_chain_begin(x0, pm0, P[0].hc_fn, P[0].hc_scale, P[0].hc_base, state_out=states[0],
                       pre_out=pres[0], stream=stream)
    x = x0
    for s in range(sides):
        if events is not None:
            events[s][0].record(stream)
        last = s + 1 == sides
        y = y_last if (last and y_last is not None) else ys[s % 2]
        if not last:
            q = P[s + 1]
            hcg.hc_chain_side(x, fs[s], states[s % 2], P[s].norm_w, q.hc_fn, q.hc_scale, q.hc_base,
                              h_norm=h_norm, y=y, state_out=states[(s + 1) % 2],
                              pre_out=(pre_last if (s + 2 == sides and pre_last is not None)
                                       else pres[(s + 1) % 2]), stream=stream)
        else:
            hcg.hc_chain_side(x, fs[s], states[s % 2], P[s].norm_w, h_norm=h_norm, y=y, stream=stream)
        if events is not None:
            events[s][1].record(stream)
        x = y


def run_ours(args, rank, local_rank, world):
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    hcg._lib.load()
    case, fs, seed = build_workload(dev, rank, args.workload)
    n, d = case.n, case.d
    sides = len(case.params)
    x0, pm0 = case.x, case.pre_mix
    ys = [torch.empty_like(x0), torch.empty_like(x0)]
    pres = [torch.empty((n, HC), device=dev), torch.empty((n, HC), device=dev)]
    h_norm = torch.empty((n, d), dtype=torch.bfloat16, device=dev)
    params = [p.astuple() for p in case.params]
    stream = torch.cuda.current_stream(dev)
    launches = {"n": 0}
    chain = args.path == "chain"
    states = [hcg.chain_state(n, d, dev) for _ in range(2)] if chain else None

    def step_chain(events=None):
        # the sides fused across sides: each launch finishes side s and starts s + 1
        run_chain(case, x0, pm0, fs, ys, pres, h_norm, states, events, stream)
        # sides + 1 chain launches, all but the last after a one-thread epoch kernel
        launches["n"] += 2 * sides + 1

    def step_blocks(events=None):
        x, pm = x0, pm0
        for s in range(sides):
            if events is not None:
                events[s][0].record(stream)
            hcg.hc_block_step(x, pm, fs[s], *params[s], h_norm=h_norm, y=ys[s % 2],
                              pre_out=pres[s % 2])
            if events is not None:
                events[s][1].record(stream)
            launches["n"] += 1
            x, pm = ys[s % 2], pres[s % 2]

    step = step_chain if chain else step_blocks

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    launches["n"] = 0
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(sides)] for _ in range(args.steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(args.steps):
        step(ev[k])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = t0.elapsed_time(t1)
    # the dominant kernel's launches: every side step, or for the chain the sides
    # that also start the next side (all but the last)
    launch_ms = [a.elapsed_time(b) for e in ev for (a, b) in (e[:-1] if chain else e)]
    gpu_launches = launches["n"]
    if world > 1:
        elapsed_ms = max_over_ranks(elapsed_ms, dev)

    # The same workload through one hc_block_step launch per side, timed the same
    # way on fewer steps, beside the chain's figures.
    blocks = None
    if chain and args.workload == "long_prefill" and not args.no_step_path:
        k_b = max(2, args.steps // 2)
        step_blocks()
        torch.cuda.synchronize(dev)
        evb = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(sides)] for _ in range(k_b)]
        b0 = torch.cuda.Event(enable_timing=True)
        b1 = torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for k in range(k_b):
            step_blocks(evb[k])
        b1.record(stream)
        torch.cuda.synchronize(dev)
        blocks = (b0.elapsed_time(b1) / k_b, [a.elapsed_time(b) for e in evb for (a, b) in e], k_b)

    e2e = None if (args.no_e2e or args.workload != "long_prefill") else \
        run_e2e(args, dev, case, seed, world)
    out = None
    if rank == 0:
        ms_per_step = elapsed_ms / args.steps
        tokens_per_s = world * n / (ms_per_step / 1e3)
        avg_launch_s = statistics.mean(launch_ms) / 1e3
        alg_bytes = n * BYTES_PER_TOKEN + BYTES_WEIGHTS
        achieved = alg_bytes / avg_launch_s / 1e9
        peak, peak_kind = measured_peaks()
        step_bytes = sides * alg_bytes
        out = {
            "metric": "tokens/s (65,536-token long prefill through 40 layers = 80 fused "
                      "hc_block_step side steps) and achieved HBM GB/s"
                      if args.workload == "long_prefill" else
                      "tokens/s through the %s workload's %d side steps" % (args.workload, sides),
            "value": tokens_per_s,
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms_per_step,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16 streams, fp32 arithmetic",
            "data": "synthetic, seeded (x N(0,1); hc_fn N(0,0.01); f N(0,2); per-side params)",
            "config": {"workload": args.workload, "description": WORKLOADS[args.workload][2],
                       "tokens": n, "hc": HC, "d": d, "side_steps": sides,
                       "sinkhorn_iters": 20, "seed": seed, "parallelism": "replicas" if world > 1 else "single",
                       "path": ("chain: hc_chain_begin + %d hc_chain_side, each side's launch also "
                                "computing the next side's coefficients; outputs equal hc_block_step's "
                                "bit for bit" % sides) if chain else "step: %d hc_block_step launches" % sides,
                       "l2": ("inputs larger than L2 (x is %.2f GB per side, L2 %.0f MB); no flush"
                              % (n * HC * d * 2 / 1e9, L2_BYTES / 1e6))
                             if n * HC * d * 2 > L2_BYTES else
                             "inputs smaller than L2 (%.1f MB per side); not flushed: latency case"
                             % (n * HC * d * 2 / 1e6)},
            "hbm_gbs_step": step_bytes / (ms_per_step / 1e3) / 1e9,
            "hbm_frac_step": step_bytes / (ms_per_step / 1e3) / 1e9 / peak,
            "roofline": {"kernel": ("hc_chain_side (k_slices<kSide>: side i's y and h_norm fused with side "
                                    "i + 1's mixes, one CTA per SM in groups of 16)") if chain else
                                   KERNEL_NAME + " (k_block_cluster)",
                         "bound": "hbm", "achieved": achieved,
                         "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)"
                         if peak_kind == "measured" else peak_kind,
                         "traffic": ncu_traffic_per_launch(n, "chain" if chain else "step"),
                         "algorithmic_bytes_per_launch": alg_bytes,
                         "avg_launch_us": avg_launch_s * 1e6, "launches_timed": len(launch_ms)},
            "clocks": clk,
            "gpu_launches": gpu_launches,
            "e2e": e2e,
        }
        if blocks is not None:
            b_ms, b_launch, k_b = blocks
            b_avg_s = statistics.mean(b_launch) / 1e3
            out["hc_block_step_path"] = {
                "value": world * n / (b_ms / 1e3), "unit": "tokens/s", "ms_per_step": b_ms, "steps": k_b,
                "roofline_frac": alg_bytes / b_avg_s / 1e9 / peak, "avg_launch_us": b_avg_s * 1e6,
                "traffic": ncu_traffic_per_launch(n, "step"),
                "note": "the same sides as one hc_block_step launch each, timed after the chain's "
                        "steps (rank 0's clock); outputs identical to the chain's bit for bit"}
        if world == 1 and not args.no_cpu_baseline and args.workload == "long_prefill":
            out["cpu_baseline"] = cpu_baseline_sample(case, fs, target_s=args.cpu_seconds)
        if chain and args.workload == "long_prefill" and not args.no_configs:
            out["chain_equals_step"] = chain_equals_steps(case, fs, dev, stream)
            out["model_order"] = run_model_order(case, fs, ys, h_norm, states, dev, stream)
    if rank == 0 and world == 1 and args.workload == "long_prefill" and not args.no_configs:
        del fs, case, ys, h_norm, states
        torch.cuda.empty_cache()
        out["configs"] = run_configs(dev, measured_peaks()[0], stream)
        out["stream_counts"] = run_stream_counts(dev, stream)
    return out


def _event_ms(fn, k, stream, flush=None):
    """CUDA-event durations (ms) of k calls of fn on `stream`.  With `flush` (a
    device buffer larger than L2) the buffer is rewritten before every call,
    outside the timed events, so that no call finds its inputs in L2."""
    out = []
    for _ in range(k):
        if flush is not None:
            flush.add_(1)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        out.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in out]


def _graph_ms(make_fn, k, stream, flush):
    """CUDA-event durations (ms) of k replays of a CUDA graph holding one call.
    make_fn(st) returns the call with its launches on stream st; it is
    captured once on a side stream (after the eager calls that precede it)
    and replayed on `stream`, with L2 flushed before every replay."""
    cs = torch.cuda.Stream(device=stream.device)
    cs.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cs):
        make_fn(cs)()
    stream.wait_stream(cs)
    for _ in range(3):
        graph.replay()
    return _event_ms(graph.replay, k, stream, flush)


def _oracle_rate(fn, units, what):
    """The oracle on a sample, timed on one host core: units per second."""
    t0 = time.perf_counter()
    fn()
    dt = time.perf_counter() - t0
    return {"value": units / dt, "cores": 1, "kind": "oracle", "sample": "%s (%.2f s)" % (what, dt)}


def run_configs(dev, peak, stream):
    """Every workload besides the long prefill, timed with CUDA events on the
    launching stream: tiny (16 tokens, one side), decode (128 tokens, two
    sides), the Sinkhorn-only stress (2^20 rows) and the prefill (8,192 tokens
    with outliers, two sides, through one hc_block_step per side and through
    the chain).  Inputs smaller than L2 are timed with L2 flushed before every
    call; each record carries its roofline fraction and the oracle timed on a
    sample of the same inputs."""
    import oracle
    oracle.build()
    flush = torch.empty(64 << 20, dtype=torch.int32, device=dev)   # 256 MB, twice the L2
    recs = {}
    side_bytes = lambda n: n * BYTES_PER_TOKEN + BYTES_WEIGHTS
    np_params = lambda p: tuple(t.detach().cpu().numpy() for t in p.astuple())

    # tiny: one side step on 16 tokens
    case = inputs.tiny(device=dev)
    p = case.params[0]
    h = torch.empty((case.n, case.d), dtype=torch.bfloat16, device=dev)
    y = torch.empty_like(case.x)
    pre = torch.empty_like(case.pre_mix)
    make = lambda st: (lambda: hcg.hc_block_step(case.x, case.pre_mix, case.fs[0], *p.astuple(), h_norm=h,
                                                 y=y, pre_out=pre, stream=st))
    fn = make(stream)
    for _ in range(5):
        fn()
    cold = _event_ms(fn, 50, stream, flush)
    warm = _event_ms(fn, 50, stream)
    graph = _graph_ms(make, 50, stream, flush)
    alg = side_bytes(case.n)
    xb, fb = inputs.bf16_bits_np(case.x), inputs.bf16_bits_np(case.fs[0])
    pmn = case.pre_mix.cpu().numpy().astype(np.float64)
    cpu = _oracle_rate(lambda: oracle.block_step(xb, pmn, fb, *np_params(p)), case.n,
                       "all 16 tokens, one side step")
    cpu["unit"] = "tokens/s"
    recs["tiny"] = {
        "workload": "tiny: B=1, T=16, one hc_block_step side (seed 0)", "tokens": case.n, "sides": 1,
        "us_per_side": 1e3 * statistics.mean(cold), "us_per_side_median": 1e3 * statistics.median(cold),
        "us_per_side_l2_warm": 1e3 * statistics.mean(warm),
        "us_per_side_graph": 1e3 * statistics.mean(graph),
        "tokens_per_s": case.n / (statistics.mean(cold) / 1e3),
        "algorithmic_bytes": alg, "hbm_gbs": alg / (statistics.mean(cold) / 1e3) / 1e9,
        "roofline_frac": alg / (statistics.mean(cold) / 1e3) / 1e9 / peak,
        "l2": "flushed before every call (256 MB written); l2_warm: back to back", "calls": len(cold),
        "graph": "the call captured once into a CUDA graph and replayed, L2 flushed before each replay",
        "cpu_baseline": cpu}

    # decode: 128 tokens, attention side then FFN side (the FFN side reads with the attention side's pre)
    case = inputs.decode(device=dev)
    pa, pf = case.params
    ya, yf = torch.empty_like(case.x), torch.empty_like(case.x)
    ha = torch.empty((case.n, case.d), dtype=torch.bfloat16, device=dev)
    prea, pref = torch.empty_like(case.pre_mix), torch.empty_like(case.pre_mix)

    def make_two(st):
        def two_sides():
            hcg.hc_block_step(case.x, case.pre_mix, case.fs[0], *pa.astuple(), h_norm=ha, y=ya, pre_out=prea,
                              stream=st)
            hcg.hc_block_step(ya, prea, case.fs[1], *pf.astuple(), h_norm=ha, y=yf, pre_out=pref, stream=st)
        return two_sides
    two_sides = make_two(stream)
    for _ in range(5):
        two_sides()
    cold = _event_ms(two_sides, 50, stream, flush)
    graph = _graph_ms(make_two, 50, stream, flush)
    alg = 2 * side_bytes(case.n)
    xb = inputs.bf16_bits_np(case.x)
    fbs = [inputs.bf16_bits_np(f) for f in case.fs]
    pmn = case.pre_mix.cpu().numpy().astype(np.float64)

    def oracle_two():
        o = oracle.block_step(xb, pmn, fbs[0], *np_params(pa))
        oracle.block_step(o["y"], o["pre"], fbs[1], *np_params(pf))
    cpu = _oracle_rate(oracle_two, case.n, "all 128 tokens through both sides")
    cpu["unit"] = "tokens/s"
    recs["decode"] = {
        "workload": "decode: B=128, T=1, attention + FFN side, two hc_block_step launches (seed 1)",
        "tokens": case.n, "sides": 2, "us_per_side": 1e3 * statistics.mean(cold) / 2,
        "us_two_sides_median": 1e3 * statistics.median(cold),
        "us_per_side_graph": 1e3 * statistics.mean(graph) / 2,
        "graph": "both sides captured once into one CUDA graph and replayed, L2 flushed before each replay",
        "tokens_per_s": case.n / (statistics.mean(cold) / 1e3),
        "algorithmic_bytes": alg, "hbm_gbs": alg / (statistics.mean(cold) / 1e3) / 1e9,
        "roofline_frac": alg / (statistics.mean(cold) / 1e3) / 1e9 / peak,
        "l2": "flushed before every two-side call (the 1.99 MB of weights per side counted)",
        "calls": len(cold), "cpu_baseline": cpu}
    del ya, yf, ha

    # Sinkhorn-only stress: 2^20 rows of N(0, 3) mixes
    m, sc, base = (t.to(dev) for t in inputs.sinkhorn_stress(device="cpu"))
    rows = m.shape[0]
    pre_s = torch.empty((rows, HC), device=dev)
    post_s = torch.empty((rows, HC), device=dev)
    comb_s = torch.empty((rows, HC, HC), device=dev)
    fn = lambda: hcg.hc_split_sinkhorn(m, sc, base, pre=pre_s, post=post_s, comb=comb_s, stream=stream)
    for _ in range(5):
        fn()
    cold = _event_ms(fn, 30, stream, flush)
    alg = rows * 192 + 12 + MIX * 4
    ms = m[:16384].cpu().numpy().astype(np.float64)
    cpu = _oracle_rate(lambda: oracle.split_sinkhorn(ms, sc.cpu().numpy(), base.cpu().numpy()), len(ms),
                       "16,384 of 1,048,576 rows")
    cpu["unit"] = "rows/s"
    recs["sinkhorn_stress"] = {
        "workload": "Sinkhorn-only stress: 1,048,576 rows, hc_split_sinkhorn, 20 rounds (seed 2)",
        "rows": rows, "us_per_call": 1e3 * statistics.mean(cold), "rows_per_s": rows / (statistics.mean(cold) / 1e3),
        "algorithmic_bytes": alg, "bytes_per_row": 192, "hbm_gbs": alg / (statistics.mean(cold) / 1e3) / 1e9,
        "roofline_frac": alg / (statistics.mean(cold) / 1e3) / 1e9 / peak,
        "l2": "flushed before every call (inputs 100.7 MB, under L2)", "calls": len(cold), "cpu_baseline": cpu}
    del m, pre_s, post_s, comb_s

    # prefill: 8,192 tokens with outliers, two sides, through hc_block_step and through the chain
    case = inputs.prefill(device=dev)
    pa, pf = case.params
    n = case.n
    ys = [torch.empty_like(case.x), torch.empty_like(case.x)]
    hn = torch.empty((n, case.d), dtype=torch.bfloat16, device=dev)
    pres = [torch.empty_like(case.pre_mix), torch.empty_like(case.pre_mix)]
    states = [hcg.chain_state(n, case.d, dev) for _ in range(2)]
    evs_step = []

    def steps(record):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        hcg.hc_block_step(case.x, case.pre_mix, case.fs[0], *pa.astuple(), h_norm=hn, y=ys[0],
                          pre_out=pres[0], stream=stream)
        e[1].record(stream)
        hcg.hc_block_step(ys[0], pres[0], case.fs[1], *pf.astuple(), h_norm=hn, y=ys[1], pre_out=pres[1],
                          stream=stream)
        e[2].record(stream)
        if record:
            evs_step.append(e)
    evs_chain = []

    def chain(record):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        e[0].record(stream)
        hcg.hc_chain_begin(case.x, case.pre_mix, pa.hc_fn, pa.hc_scale, pa.hc_base, state_out=states[0],
                           pre_out=pres[0], stream=stream)
        e[1].record(stream)
        hcg.hc_chain_side(case.x, case.fs[0], states[0], pa.norm_w, pf.hc_fn, pf.hc_scale, pf.hc_base,
                          h_norm=hn, y=ys[0], state_out=states[1], pre_out=pres[1], stream=stream)
        e[2].record(stream)
        hcg.hc_chain_side(ys[0], case.fs[1], states[1], pf.norm_w, h_norm=hn, y=ys[1], stream=stream)
        e[3].record(stream)
        if record:
            evs_chain.append(e)
    for _ in range(3):
        steps(False)
        chain(False)
    for _ in range(10):
        steps(True)
    for _ in range(10):
        chain(True)
    torch.cuda.synchronize()
    alg = side_bytes(n)
    st_launch = [e[i].elapsed_time(e[i + 1]) for e in evs_step for i in range(2)]
    st_pair = [e[0].elapsed_time(e[2]) for e in evs_step]
    ch_pair = [e[0].elapsed_time(e[3]) for e in evs_chain]
    ch_fused = [e[1].elapsed_time(e[2]) for e in evs_chain]
    rows_o = np.sort(np.random.default_rng(3).choice(n, 64, replace=False))
    ri = torch.from_numpy(rows_o).to(dev)
    xb = inputs.bf16_bits_np(case.x.index_select(0, ri))
    fbs = [inputs.bf16_bits_np(f.index_select(0, ri)) for f in case.fs]
    pmn = case.pre_mix.index_select(0, ri).cpu().numpy().astype(np.float64)

    def oracle_two():
        o = oracle.block_step(xb, pmn, fbs[0], *np_params(pa))
        oracle.block_step(o["y"], o["pre"], fbs[1], *np_params(pf))
    cpu = _oracle_rate(oracle_two, len(rows_o), "64 of 8,192 tokens through both sides")
    cpu["unit"] = "tokens/s"
    recs["prefill"] = {
        "workload": "prefill: B=1, T=8192, 1% outliers x50, attention + FFN side (seed 3)",
        "tokens": n, "sides": 2, "algorithmic_bytes_per_side": alg,
        "l2": "inputs larger than L2 (x is 335.5 MB); no flush",
        "step": {"path": "two hc_block_step launches", "us_per_side": 1e3 * statistics.mean(st_launch),
                 "tokens_per_s": n / (statistics.mean(st_pair) / 1e3),
                 "roofline_frac": alg / (statistics.mean(st_launch) / 1e3) / 1e9 / peak,
                 "meets_0_70": alg / (statistics.mean(st_launch) / 1e3) / 1e9 / peak >= 0.70},
        "chain": {"path": "hc_chain_begin + fused hc_chain_side + last hc_chain_side",
                  "us_both_sides": 1e3 * statistics.mean(ch_pair),
                  "tokens_per_s": n / (statistics.mean(ch_pair) / 1e3),
                  "roofline_frac_both_sides": 2 * alg / (statistics.mean(ch_pair) / 1e3) / 1e9 / peak,
                  "us_fused_launch": 1e3 * statistics.mean(ch_fused),
                  "roofline_frac_fused_launch": alg / (statistics.mean(ch_fused) / 1e3) / 1e9 / peak,
                  "meets_0_70": 2 * alg / (statistics.mean(ch_pair) / 1e3) / 1e9 / peak >= 0.70},
        "calls": len(evs_step), "cpu_baseline": cpu}
    return recs


def run_model_order(case, fs, ys, h_norm, states, dev, stream, steps=3):
    """The long prefill in model order (Block page, Block.forward: the sublayer
    reads h_norm_i before its output f_i exists): per side one hc_chain_side
    launch writing y_i and side i + 1's bf16 h, then hc_chain_norm making
    h_norm_{i+1} (here f_i is the stand-in sublayer output, given).  Timed with
    CUDA events per launch; the side's algorithmic bytes are counted once per
    side against the time of its two launches."""
    P = case.params
    n, d = case.n, case.d
    hp = torch.empty((n, d), dtype=torch.bfloat16, device=dev)
    evs = []

    def one(record):
        e0 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        hcg.hc_chain_begin(case.x, case.pre_mix, P[0].hc_fn, P[0].hc_scale, P[0].hc_base,
                           state_out=states[0], h_pre_out=hp, stream=stream)
        x = case.x
        marks = []
        for s in range(len(P)):
            a = torch.cuda.Event(enable_timing=True)
            m = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            hcg.hc_chain_norm(hp, states[s % 2], P[s].norm_w, h_norm=h_norm, stream=stream)
            m.record(stream)
            y = ys[s % 2]
            if s + 1 < len(P):
                q = P[s + 1]
                hcg.hc_chain_side(x, fs[s], states[s % 2], P[s].norm_w, q.hc_fn, q.hc_scale, q.hc_base,
                                  y=y, state_out=states[(s + 1) % 2], h_pre_out=hp, stream=stream)
            else:
                hcg.hc_chain_side(x, fs[s], states[s % 2], P[s].norm_w, y=y, write_h_norm=False,
                                  stream=stream)
            b.record(stream)
            marks.append((a, m, b))
            x = y
        e1 = torch.cuda.Event(enable_timing=True)
        e1.record(stream)
        if record:
            evs.append((e0, e1, marks))
    one(False)
    for _ in range(steps):
        one(True)
    torch.cuda.synchronize()
    step_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1, _ in evs)
    # the sides that also start the next side (all but the last): norm + chain launch
    pair_us = [a.elapsed_time(b) * 1e3 for _, _, mk in evs for (a, _, b) in mk[:-1]]
    norm_us = [a.elapsed_time(m) * 1e3 for _, _, mk in evs for (a, m, _) in mk]
    alg = n * BYTES_PER_TOKEN + BYTES_WEIGHTS
    peak = measured_peaks()[0]
    return {"path": "hc_chain_begin(h_pre_out) + 80 x [hc_chain_norm + hc_chain_side(h_pre_out)]",
            "ms_per_step": step_ms, "tokens_per_s": n / (step_ms / 1e3), "steps": steps,
            "us_per_side": statistics.mean(pair_us),
            "us_norm_launch": statistics.mean(norm_us),
            "roofline_frac_per_side": alg / (statistics.mean(pair_us) * 1e-6) / 1e9 / peak,
            "note": "fraction: the side's algorithmic bytes (102,432 per token + weights) over the time of "
                    "its chain launch and its hc_chain_norm launch (which moves 20,480 more bytes per token)"}


def run_stream_counts(dev, stream, n=8192, d=D):
    """Two and eight streams (the pages' kernel is generic in hc): one
    hc_block_step and one hc_block_step_backward at 8,192 tokens x d = 5120,
    timed with CUDA events (inputs larger than L2)."""
    peak = measured_peaks()[0]
    out = {}
    for hc in (2, 8):
        g = torch.Generator(device=dev).manual_seed(40 + hc)
        x = inputs.streams(g, n, hc, d, device=dev)
        pm = inputs.pre_mix(g, n, hc, device=dev)
        f = inputs.sublayer_out(g, n, d, device=dev)
        p = inputs.side_params(g, hc, d, device=dev)
        mix = (2 + hc) * hc
        fwd = lambda: hcg.hc_block_step(x, pm, f, *p.astuple(), stream=stream)
        ws = torch.empty(hcg._lib.load().hc_block_step_backward_workspace_bytes(n, hc, d), dtype=torch.uint8,
                         device=dev)
        g_hn = torch.randn((n, d), device=dev, generator=g)
        g_y = torch.randn((n, hc, d), device=dev, generator=g)
        bwd = lambda: hcg.hc_block_step_backward(x, pm, f, *p.astuple(), g_hn, g_y, workspace=ws, stream=stream)
        for _ in range(3):
            fwd()
            bwd()
        t_f = statistics.mean(_event_ms(fwd, 10, stream))
        t_b = statistics.mean(_event_ms(bwd, 5, stream))
        w_bytes = mix * hc * d * 4 + 12 + mix * 4 + d * 4
        alg_f = n * (hc * d * 2 + d * 2 + hc * 4 + hc * d * 2 + d * 2 + hc * 4) + w_bytes
        alg_b = n * (hc * d * 2 + d * 2 + hc * 4 + d * 4 + hc * d * 4 + hc * d * 4 + hc * 4 + d * 4) + 2 * w_bytes
        out["hc%d" % hc] = {
            "tokens": n, "d": d, "mix": mix,
            "forward": {"entry": "hc_block_step", "us": t_f * 1e3, "tokens_per_s": n / (t_f / 1e3),
                        "algorithmic_bytes": alg_f, "roofline_frac": alg_f / (t_f / 1e3) / 1e9 / peak},
            "backward": {"entry": "hc_block_step_backward", "us": t_b * 1e3, "tokens_per_s": n / (t_b / 1e3),
                         "algorithmic_bytes": alg_b, "roofline_frac": alg_b / (t_b / 1e3) / 1e9 / peak}}
        del x, f, g_hn, g_y, ws
    return out


def chain_equals_steps(case, fs, dev, stream):
    """The long prefill's 80 sides through the chain and through one
    hc_block_step per side, side by side on the same inputs: h_norm, y and pre
    of every side compared bit for bit."""
    n, d = case.n, case.d
    P = case.params
    ys = [torch.empty_like(case.x) for _ in range(2)]
    yc = [torch.empty_like(case.x) for _ in range(2)]
    hs = torch.empty((n, d), dtype=torch.bfloat16, device=dev)
    hcn = torch.empty_like(hs)
    ps = [torch.empty_like(case.pre_mix) for _ in range(2)]
    pc = [torch.empty_like(case.pre_mix) for _ in range(2)]
    st = [hcg.chain_state(n, d, dev) for _ in range(2)]
    hcg.hc_chain_begin(case.x, case.pre_mix, P[0].hc_fn, P[0].hc_scale, P[0].hc_base, state_out=st[0],
                       pre_out=pc[0], stream=stream)
    xs, pms, xc = case.x, case.pre_mix, case.x
    first = None
    for s in range(len(P)):
        b = s % 2
        hcg.hc_block_step(xs, pms, fs[s], *P[s].astuple(), h_norm=hs, y=ys[b], pre_out=ps[b], stream=stream)
        if s + 1 < len(P):
            q = P[s + 1]
            hcg.hc_chain_side(xc, fs[s], st[b], P[s].norm_w, q.hc_fn, q.hc_scale, q.hc_base, h_norm=hcn,
                              y=yc[b], state_out=st[1 - b], pre_out=pc[1 - b], stream=stream)
        else:
            hcg.hc_chain_side(xc, fs[s], st[b], P[s].norm_w, h_norm=hcn, y=yc[b], stream=stream)
        for name, u, v in (("h_norm", hs, hcn), ("y", ys[b], yc[b]), ("pre", ps[b], pc[b])):
            if first is None and not torch.equal(u.view(torch.int16) if u.dtype == torch.bfloat16 else u,
                                                 v.view(torch.int16) if v.dtype == torch.bfloat16 else v):
                first = "side %d %s" % (s, name)
        xs, pms, xc = ys[b], ps[b], yc[b]
    torch.cuda.synchronize()
    return {"sides": len(P), "equal": first is None, "first_difference": first,
            "compared": "h_norm, y and pre of every side, bit for bit"}


def run_e2e(args, dev, case, seed, world):
    """Same metric end to end through the public API: every step copies the
    step's inputs (x and the 80 sublayer outputs) from pinned host memory and
    reads the result (final y and pre) back.  f is double-buffered on the
    device so copies of side s+1 overlap the side-s kernel."""
    n, d = case.n, case.d
    f_bytes = n * d * 2
    need = SIDES * f_bytes + 2 * n * HC * d * 2
    try:
        host_ram = os.sysconf("SC_PHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except Exception:
        host_ram = 0
    n_host_f = SIDES if need < 0.45 * host_ram / max(1, world) else max(2, int(
        0.3 * host_ram / max(1, world) // f_bytes))
    n_host_f = min(SIDES, n_host_f)
    x_h = torch.empty((n, HC, d), dtype=torch.bfloat16, pin_memory=True)
    x_h.copy_(case.x)
    f_h = []
    for s in range(n_host_f):
        t = torch.empty((n, d), dtype=torch.bfloat16, pin_memory=True)
        t.copy_(inputs.long_prefill_f(s, n, d, dev, seed))
        f_h.append(t)
    pm_h = case.pre_mix.cpu().pin_memory()
    y_h = torch.empty((n, HC, d), dtype=torch.bfloat16, pin_memory=True)
    pre_h = torch.empty((n, HC), dtype=torch.float32, pin_memory=True)
    # Device buffers: x and pre_mix double-buffered across steps, f across sides.
    x_d = [torch.empty((n, HC, d), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    pm_d = [torch.empty((n, HC), device=dev) for _ in range(2)]
    f_d = [torch.empty((n, d), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    ys = [torch.empty((n, HC, d), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    pres = [torch.empty((n, HC), device=dev), torch.empty((n, HC), device=dev)]
    y_last = torch.empty((n, HC, d), dtype=torch.bfloat16, device=dev)
    pre_last = torch.empty((n, HC), device=dev)
    h_norm = torch.empty((n, d), dtype=torch.bfloat16, device=dev)
    params = [p.astuple() for p in case.params]
    chain = args.path == "chain"
    states = [hcg.chain_state(n, d, dev) for _ in range(2)] if chain else None
    comp = torch.cuda.current_stream(dev)
    # Each host-to-device copy is split over several streams, so that several copy
    # engines share it; every chunk is one cudaMemcpyAsync.
    n_copy = 4
    copies = [torch.cuda.Stream(dev) for _ in range(n_copy)]
    d2h = torch.cuda.Stream(dev)
    rows = [(c * n // n_copy, (c + 1) * n // n_copy) for c in range(n_copy)]
    f_free = [torch.cuda.Event() for _ in range(2)]   # kernel done with f_d[b]
    x_free = [torch.cuda.Event() for _ in range(2)]   # kernel done with x_d[b]
    y_free = torch.cuda.Event()                       # y_last read back
    ready = {}

    def issue_inputs(g):
        """Copies for global side g (step g // SIDES, side g % SIDES)."""
        i, s = divmod(g, SIDES)
        fb, xb = g % 2, i % 2
        evs = []
        for c, st in enumerate(copies):
            a, b = rows[c]
            with torch.cuda.stream(st):
                st.wait_event(f_free[fb])
                f_d[fb][a:b].copy_(f_h[s % n_host_f][a:b], non_blocking=True)
                if s == 0:
                    st.wait_event(x_free[xb])
                    x_d[xb][a:b].copy_(x_h[a:b], non_blocking=True)
                    pm_d[xb][a:b].copy_(pm_h[a:b], non_blocking=True)
                e = torch.cuda.Event()
                e.record(st)
                evs.append(e)
        ready[g] = evs

    def run(steps):
        total = steps * SIDES
        issue_inputs(0)
        x = pm = None
        for g in range(total):
            i, s = divmod(g, SIDES)
            if g + 1 < total:
                issue_inputs(g + 1)  # prefetch: the next side's f (and the next step's x)
            for e in ready.pop(g):
                comp.wait_event(e)
            if s == 0:
                x, pm = x_d[i % 2], pm_d[i % 2]
            b = s % 2
            last = s == SIDES - 1
            out, pre_o = (y_last, pre_last) if last else (ys[b], pres[b])
            if chain:
                P = case.params
                if s == 0:
                    hcg.hc_chain_begin(x, pm, P[0].hc_fn, P[0].hc_scale, P[0].hc_base,
                                       state_out=states[0], pre_out=pres[0], stream=comp)
                if s == SIDES - 2:
                    comp.wait_event(y_free)  # the previous step's result has been read back
                if not last:
                    q = P[s + 1]
                    # launch s writes side s + 1's pre (the last side's into pre_last)
                    nxt_pre = pre_last if s == SIDES - 2 else pres[(s + 1) % 2]
                    hcg.hc_chain_side(x, f_d[g % 2], states[s % 2], P[s].norm_w, q.hc_fn, q.hc_scale,
                                      q.hc_base, h_norm=h_norm, y=out, state_out=states[(s + 1) % 2],
                                      pre_out=nxt_pre, stream=comp)
                else:
                    hcg.hc_chain_side(x, f_d[g % 2], states[s % 2], P[s].norm_w, h_norm=h_norm, y=out,
                                      stream=comp)
            else:
                if last:
                    comp.wait_event(y_free)  # the previous step's result has been read back
                hcg.hc_block_step(x, pm, f_d[g % 2], *params[s], h_norm=h_norm, y=out, pre_out=pre_o,
                                  stream=comp)
            f_free[g % 2].record(comp)
            if s == 0:
                x_free[i % 2].record(comp)
            x, pm = out, pre_o
            if last:
                # the step's result back to the host
                d2h.wait_stream(comp)
                with torch.cuda.stream(d2h):
                    y_h.copy_(y_last, non_blocking=True)
                    pre_h.copy_(pre_last, non_blocking=True)
                    y_free.record(d2h)

    for e in f_free + x_free + [y_free]:
        e.record(comp)
    run(1)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    steps = max(1, min(args.steps, 5))
    t0 = time.perf_counter()
    run(steps)
    torch.cuda.synchronize(dev)
    dt = time.perf_counter() - t0
    if world > 1:
        dt = max_over_ranks(dt, dev)
    h2d = n * HC * d * 2 + n * HC * 4 + SIDES * f_bytes
    d2h = n * HC * d * 2 + n * HC * 4
    return {"value": world * n * steps / dt, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps,
            "host_f_buffers": n_host_f,
            "note": "pinned host buffers; H2D of x and all 80 f per step, D2H of final y and pre; "
                    "copies split over 4 streams and double-buffered against the kernels (the next "
                    "side's f and the next step's x load while a side computes)"
                    + ("" if n_host_f == SIDES else "; host f pool of %d reused cyclically" % n_host_f)}


# ---------------------------------------------------------------- oracle arm
def _oracle_chain(oracle, x_bits, pm, fs_bits, params_np):
    for s in range(SIDES):
        o = oracle.block_step(x_bits, pm, fs_bits[s], *params_np[s])
        x_bits, pm = o["y"], o["pre"]
    return x_bits, pm


def cpu_baseline_sample(case, fs, target_s=15.0, sample_tokens=None):
    """The oracle (single-threaded C, fp64) on a sample of tokens through all
    80 side steps; tokens/s extrapolated from the sample."""
    import oracle
    oracle.build()
    n = case.n
    params_np = [tuple(t.detach().cpu().numpy() for t in p.astuple()) for p in case.params]
    rows = torch.arange(0, n, max(1, n // 4096), device=case.x.device)
    probe = rows[:2]
    # warm: load the library and touch every code path once before timing
    _oracle_chain(oracle, inputs.bf16_bits_np(case.x.index_select(0, probe[:1])),
                  case.pre_mix.index_select(0, probe[:1]).cpu().numpy().astype(np.float64),
                  [inputs.bf16_bits_np(f.index_select(0, probe[:1])) for f in fs], params_np)
    fs_np = lambda r: [inputs.bf16_bits_np(f.index_select(0, r)) for f in fs]
    t0 = time.perf_counter()
    _oracle_chain(oracle, inputs.bf16_bits_np(case.x.index_select(0, probe)),
                  case.pre_mix.index_select(0, probe).cpu().numpy().astype(np.float64),
                  fs_np(probe), params_np)
    per_tok = (time.perf_counter() - t0) / 2
    k = sample_tokens or max(2, min(len(rows), int(target_s / max(per_tok, 1e-6))))
    sel = rows[:k]
    t0 = time.perf_counter()
    _oracle_chain(oracle, inputs.bf16_bits_np(case.x.index_select(0, sel)),
                  case.pre_mix.index_select(0, sel).cpu().numpy().astype(np.float64),
                  fs_np(sel), params_np)
    dt = time.perf_counter() - t0
    return {"value": k / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": "%d of %d tokens through all 80 side steps (%.1f s)" % (k, n, dt),
            "host_cores_available": os.cpu_count()}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    import oracle
    oracle.build()
    dev = "cpu"
    # a bounded sample of the same workload: the same generators and
    # distributions, drawn for `tok` tokens
    tok = max(1, args.reference_tokens)
    case = inputs.long_prefill(device=dev, seed=4, n=tok, materialize_f=False)
    fs = [inputs.long_prefill_f(s, tok, D, dev, 4) for s in range(SIDES)]
    params_np = [tuple(t.numpy() for t in p.astuple()) for p in case.params]
    xb = inputs.bf16_bits_np(case.x[:tok])
    pm = case.pre_mix[:tok].numpy().astype(np.float64)
    fb = [inputs.bf16_bits_np(f[:tok]) for f in fs]
    for _ in range(args.warmup):
        _oracle_chain(oracle, xb[:1], pm[:1], [f[:1] for f in fb], params_np)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_chain(oracle, xb, pm, fb, params_np)
    dt = time.perf_counter() - t0
    value = tok * args.steps / dt
    return {
        "impl": "reference",
        "metric": "tokens/s (65,536-token long prefill through 40 layers = 80 fused "
                  "hc_block_step side steps) and achieved HBM GB/s",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic, seeded",
        "config": {"workload": "long_prefill", "batch": 4, "seq_len": 16384, "tokens": TOKENS,
                   "hc": HC, "d": D, "layers": LAYERS, "side_steps": SIDES},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": "%d tokens of the long prefill through all 80 side steps per step"
                                   % tok},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_side_step_op(args, dev):
    """One hc_block_step at --hc streams (2, 4 or 8) over --tokens tokens
    (default 8,192) x d = 5120, the inputs of the stream_counts sub-record:
    for profiler captures of one stream count's side step."""
    hc, n, d = args.hc, args.tokens or 8192, D
    g = torch.Generator(device=dev).manual_seed(40 + hc)
    x = inputs.streams(g, n, hc, d, device=dev)
    pm = inputs.pre_mix(g, n, hc, device=dev)
    f = inputs.sublayer_out(g, n, d, device=dev)
    p = inputs.side_params(g, hc, d, device=dev)
    mix = (2 + hc) * hc
    alg = n * (hc * d * 2 + d * 2 + hc * 4 + hc * d * 2 + d * 2 + hc * 4) + mix * hc * d * 4 + 12 + mix * 4 + d * 4
    fn = lambda: hcg.hc_block_step(x, pm, f, *p.astuple())
    # launches per call: at four streams (d = 5120) the fused cluster kernel; else the
    # weight split, the tcgen05 projection, (with K split over CTAs, when there are
    # fewer 128-token tiles than CTA slots) the finish, and a4-a6
    slots = torch.cuda.get_device_properties(dev).multi_processor_count * (1 if hc == 8 else 2)
    launches = 1 if hc == 4 else (4 if (n + 127) // 128 < slots else 3)
    return fn, alg, n, d, "one side step at %d streams (hc_block_step)" % hc, launches


def run_backward_hc_op(args, dev):
    """hc_block_step_backward at --hc streams (2 or 8) over --tokens tokens
    (default 8,192) x d = 5120, the inputs of the stream_counts sub-record."""
    hc, n, d = args.hc, args.tokens or 8192, D
    g = torch.Generator(device=dev).manual_seed(40 + hc)
    x = inputs.streams(g, n, hc, d, device=dev)
    pm = inputs.pre_mix(g, n, hc, device=dev)
    f = inputs.sublayer_out(g, n, d, device=dev)
    p = inputs.side_params(g, hc, d, device=dev)
    ws = torch.empty(hcg._lib.load().hc_block_step_backward_workspace_bytes(n, hc, d), dtype=torch.uint8,
                     device=dev)
    g_hn = torch.randn((n, d), device=dev, generator=g)
    g_y = torch.randn((n, hc, d), device=dev, generator=g)
    mix = (2 + hc) * hc
    w_bytes = mix * hc * d * 4 + 12 + mix * 4 + d * 4
    alg = n * (hc * d * 2 + d * 2 + hc * 4 + d * 4 + hc * d * 4 + hc * d * 4 + hc * 4 + d * 4) + 2 * w_bytes
    fn = lambda: hcg.hc_block_step_backward(x, pm, f, *p.astuple(), g_hn, g_y, workspace=ws)
    # the weight split, the projection, kg_token, the g_x pass, the g_hc_fn and g_norm_w
    # partials, their two sums, the g_hc_base / g_hc_scale partials and their sum
    return fn, alg, n, d, "the side step's backward at %d streams (hc_block_step_backward)" % hc, 10


def run_op(args, local_rank):
    """One kernel of the widened rows, timed alone at the long-prefill size
    (65,536 tokens x d = 5120): the MXFP8 cast of the bf16 h_norm
    (hc_mxfp8_cast) or RMSNorm(hc_pre) with the cast in its epilogue
    (hc_pre_norm_mxfp8), or the side step's backward (hc_block_step_backward,
    its launches over the batch); or one side step at another stream count
    (side_step, --hc, 8,192 tokens); or hc_split_sinkhorn on the Sinkhorn-only
    stress rows (sinkhorn; 100 MB of inputs, below L2: for profiler captures,
    the configs sub-record times it with L2 flushed).  One step is one call
    over the whole batch.  The oracle is timed beside it on a sample (not for
    side_step and sinkhorn: the stream_counts and configs sub-records'
    workloads)."""
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    hcg._lib.load()
    if args.op == "sinkhorn":
        # the Sinkhorn-only stress rows (2^20, or --tokens rows), one hc_split_sinkhorn per step
        m, sc, base = (t.to(dev) for t in inputs.sinkhorn_stress(device="cpu"))
        if args.tokens:
            m = m[:args.tokens].contiguous()
        rows = m.shape[0]
        pre_s, post_s = torch.empty((rows, HC), device=dev), torch.empty((rows, HC), device=dev)
        comb_s = torch.empty((rows, HC, HC), device=dev)
        fn = lambda: hcg.hc_split_sinkhorn(m, sc, base, pre=pre_s, post=post_s, comb=comb_s)
        return _time_op(args, dev, local_rank, fn, rows * 192 + 12 + MIX * 4, rows, 0,
                        "the split and Sinkhorn (hc_split_sinkhorn)", None, 1)
    if args.op == "side_step" or (args.op == "backward" and args.hc != HC):
        fn, alg, n, d, what, launches = (run_side_step_op if args.op == "side_step" else run_backward_hc_op)(args, dev)
        return _time_op(args, dev, local_rank, fn, alg, n, d, what, None, launches)
    case = inputs.long_prefill(device=dev, materialize_f=False, n=args.tokens or TOKENS)
    n, d = case.n, case.d
    p = case.params[0]
    codes = torch.empty((n, d), dtype=torch.uint8, device=dev)
    scales = torch.empty((n, d // 32), dtype=torch.uint8, device=dev)
    h = hcg.hc_pre_norm(case.x, case.pre_mix, p.norm_w)
    if args.op == "mxfp8_cast":
        fn = lambda: hcg.hc_mxfp8_cast(h, codes, scales)
        alg = n * d * 2 + n * d + n * d // 32
        what = "MXFP8 cast of bf16 rows (hc_mxfp8_cast)"
    elif args.op == "backward":
        del codes, scales
        g = torch.Generator(device=dev).manual_seed(5)
        g_hn = torch.randn((n, d), device=dev, generator=g)
        g_y = torch.randn((n, HC, d), device=dev, generator=g)
        g_pre = torch.randn((n, HC), device=dev, generator=g)
        f0 = inputs.long_prefill_f(0, n, d, dev)
        ws = torch.empty(hcg._lib.load().hc_block_step_backward_workspace_bytes(n, HC, d),
                         dtype=torch.uint8, device=dev)
        fn = lambda: hcg.hc_block_step_backward(case.x, case.pre_mix, f0, *p.astuple(), g_hn, g_y,
                                                g_pre, workspace=ws)
        # inputs x, f, pre_mix, g_h_norm, g_y, g_pre; outputs g_x, g_pre_mix, g_f; the
        # parameters and their gradients once
        alg = (n * (HC * d * 2 + d * 2 + HC * 4 + d * 4 + HC * d * 4 + HC * 4)
               + n * (HC * d * 4 + HC * 4 + d * 4) + 2 * BYTES_WEIGHTS)
        what = "the side step's backward (hc_block_step_backward)"
    else:
        fn = lambda: hcg.hc_pre_norm_mxfp8(case.x, case.pre_mix, p.norm_w, codes=codes, scales=scales)
        alg = n * HC * d * 2 + n * HC * 4 + d * 4 + n * d + n * d // 32
        what = "RMSNorm(hc_pre) cast to MXFP8 in one pass (hc_pre_norm_mxfp8)"
    ctx = dict(case=case, p=p, h=h)
    if args.op == "backward":
        ctx.update(f0=f0, g_hn=g_hn, g_y=g_y, g_pre=g_pre)
    # backward: the weight split, the projection, the per-token pass, the g_x pass,
    # two block sums, the g_z block partials and their sum
    return _time_op(args, dev, local_rank, fn, alg, n, d, what, ctx, 8 if args.op == "backward" else 1)


def _time_op(args, dev, local_rank, fn, alg, n, d, what, ctx, launches):
    """Warm-up, then args.steps calls timed with CUDA events, clocks sampled
    meanwhile; the oracle on a sample where ctx carries the inputs."""
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    stream = torch.cuda.current_stream(dev)
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    peak, peak_kind = measured_peaks()
    rows_op = d == 0  # the Sinkhorn op: rows of mixes, no d
    out = {"metric": ("rows/s through %s, %s rows" % (what, format(n, ",")) if rows_op else
                      "tokens/s through %s, %s tokens x d = %d" % (what, format(n, ","), d)),
           "value": n / (ms / 1e3), "unit": "rows/s" if rows_op else "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": ("bf16 + fp32 in, fp32 arithmetic, fp32 gradients out" if args.op == "backward"
                     else "bf16 in, fp32 arithmetic, bf16 out" if args.op == "side_step"
                     else "fp32" if rows_op
                     else "bf16 in, fp32 arithmetic, e4m3 + ue8m0 out"), "data": "synthetic, seeded",
           "config": {"workload": ("sinkhorn_stress, 96 B of mixes in and 96 B out per row" if rows_op
                                   else "stream_counts, one side step at hc = %d" % args.hc if args.hc != HC
                                   else "long_prefill, one side step" if args.op == "backward"
                                   else "long_prefill, one side's h_norm"),
                      "op": args.op, "tokens": n, "d": d,
                      "l2": ("inputs of %.1f MB, below L2, back to back (for profiler captures; the configs "
                             "sub-record flushes L2)" % (n * 96 / 1e6) if rows_op
                             else "inputs larger than L2; no flush")},
           "roofline": {"bound": "hbm", "achieved": alg / (ms / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                        "frac": alg / (ms / 1e3) / 1e9 / peak, "traffic": None,
                        "peak_source": peak_kind, "algorithmic_bytes_per_launch": alg},
           "clocks": clk, "gpu_launches": args.steps * launches, "e2e": None}
    if not args.no_cpu_baseline and ctx is not None:
        import oracle
        case, p, h = ctx["case"], ctx["p"], ctx["h"]
        rows = torch.arange(0, n, n // 64, device=dev)
        hs = oracle.bf16_bits(h.index_select(0, rows).cpu())
        xs = oracle.bf16_bits(case.x.index_select(0, rows).cpu())
        pms = case.pre_mix.index_select(0, rows).cpu().numpy().astype(np.float64)
        w = p.norm_w.cpu().numpy()
        oracle.mxfp8(hs[:1])
        t0 = time.perf_counter()
        if args.op == "mxfp8_cast":
            oracle.mxfp8(hs)
        elif args.op == "backward":
            rows = rows[:4]
            sel = lambda tt: tt.index_select(0, rows).cpu().numpy().astype(np.float64)
            oracle.side_backward(oracle.bf16_to_f64(xs[:4]), pms[:4], oracle.bf16_to_f64(
                oracle.bf16_bits(ctx["f0"].index_select(0, rows).cpu())),
                *(t.cpu().numpy().astype(np.float64) for t in p.astuple()), sel(ctx["g_hn"]), sel(ctx["g_y"]),
                sel(ctx["g_pre"]))
        else:
            oracle.mxfp8(oracle.rmsnorm(oracle.pre(xs, pms), w))
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = {"value": len(rows) / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                               "sample": "%d of %d tokens (%.2f s)" % (len(rows), n, dt)}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="long_prefill",
                    help="long_prefill is the benchmark; the others serve profiling")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling runs)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--reference-tokens", type=int, default=4)
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads' sub-records and the chain/step comparison")
    ap.add_argument("--no-step-path", action="store_true",
                    help="with the chain, skip timing the one-launch-per-side path beside it")
    ap.add_argument("--path", choices=["chain", "step"], default="chain",
                    help="chain: the sides fused across sides (hc_chain_*); step: one hc_block_step per side")
    ap.add_argument("--op", choices=["mxfp8_cast", "pre_norm_mxfp8", "backward", "side_step", "sinkhorn"],
                    default=None,
                    help="time one kernel of the widened rows alone instead of the side steps "
                         "(side_step: one hc_block_step at --hc streams; sinkhorn: hc_split_sinkhorn on "
                         "the Sinkhorn-only stress rows)")
    ap.add_argument("--hc", type=int, choices=[2, 4, 8], default=4,
                    help="with --op side_step or backward: the stream count (2 and 8 on the stream_counts inputs)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="with --op: tokens (sinkhorn: rows) in the batch (default 65,536; 2^20 rows; "
                         "smaller for profiler captures)")
    args = ap.parse_args()
    rank, local_rank, world = dist_env()
    if args.op is not None and args.impl == "ours":
        out = run_op(args, local_rank) if rank == 0 else None
        if out is not None:
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group(backend=backend)
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        out = run_ours(args, rank, local_rank, world)
    if out is not None and rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        if args.impl == "ours":
            torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
