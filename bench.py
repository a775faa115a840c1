#!/usr/bin/env python
"""Throughput of the KDA forward pass (libkda) on GB300, one JSON line.

Default workload: B = 8 sequences x T = 8192 tokens, H = 32 heads, D = 128,
bf16, lower_bound = -5, zero initial state (seeded synthetic inputs; see
chunked_gated_delta_11_gb300/synth.py).  A step is one whole forward pass
over that batch (default: kda_fwd_fused, one kernel; --path split: kda_fwd,
chunk kernel then recurrence kernel), inputs resident in HBM.  Inputs (2.1 GB)
are larger than the 129 MB L2, so no flush runs between steps; for a
workload whose working set fits in L2 (h16, tiny) a buffer twice the L2 is
written before every timed step, outside that step's events.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the only reference arm: there is
no runnable reference implementation) on a bounded sample of the same workload.
Multi-GPU (torchrun): every rank runs its own replica (weak scaling, no
collective on the data path); rank 0 prints max-over-ranks timing.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA fwd tokens/s (GB300, bf16, D=128) + % of HBM/tensor roofline"
ALG_BYTES_PER_TOKEN_HEAD = 1282      # q, k, v, g_raw (4 x 256) + beta_raw 2 + out 256
ALG_FLOP_PER_TOKEN_HEAD = 121856     # chunk-form contractions, 16-token chunks
STATE_BYTES = 128 * 128 * 4          # one fp32 state (final written; initial read if given)
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
WORKLOAD_TEXT = {
    "b8": "B=8 sequences x T=8192 tokens, H=32, D=128, bf16, lower_bound=-5, zero initial state",
    "h16": "1 sequence x 4096 tokens, H=16, D=128, bf16, initial state 0.02*N(0,1)",
    "long": "1 sequence x 131072 tokens, H=32, D=128, bf16, g_raw~N(2,1), zero initial state",
    "varlen": "64 packed sequences, lengths U[1,16384] not multiples of 16, H=32, init 0.02*N(0,1)",
    "b2": "B=2 sequences x T=8192 tokens, H=32, D=128, bf16 (profiling size)",
    "slow": "1 sequence x 131072 tokens, H=32, D=128, bf16, g_raw~N(-6,1) (slow decay), zero "
            "initial state",
    "l32": "1 sequence x 32768 tokens, H=32, D=128, bf16, g_raw~N(2,1) (profiling size of the "
           "segmented path)",
    "decode": "one serving step: 256 sequences x 1 token, H=32, D=128, bf16, fp32 states "
              "0.02*N(0,1) in and out",
    "fk96": "FlashKDA benchmark row shape: 1 sequence x 8192 tokens, H=96, D=128, bf16, zero state",
    "fk64": "FlashKDA benchmark row shape: 1 sequence x 8192 tokens, H=64, D=128, bf16, zero state",
    "fk96p": "FlashKDA benchmark row shape '1024x8': 8 packed sequences x 1024 tokens (cu_seqlens), "
             "H=96, D=128, bf16, zero states",
    "fk64p": "FlashKDA benchmark row shape '1024x8': 8 packed sequences x 1024 tokens (cu_seqlens), "
             "H=64, D=128, bf16, zero states",
}
PATH_TEXT = {
    "fused": "kda_fwd_fused = fused_kernel (chunk math + tcgen05 recurrence, one launch)",
    "split": "kda_fwd = chunk_prep_kernel (K1) + recurrence_kernel (K2, tcgen05)",
    "decode": "kda_decode = decode_kernel (token-by-token recurrence, state slices in registers)",
    "segmented": "kda_fwd_segmented = seg_plan_kernel + fused_kernel (every sequence in P pieces, "
                 "X and M roles) + affine_scan_kernel + seg_fixup_kernel",
}
PATH_KERNEL = {"fused": "fused_kernel (the whole step)", "split": "whole kda_fwd step (K1 + K2)",
               "decode": "decode_kernel (the whole step)",
               "segmented": "whole kda_fwd_segmented step (4 launches)"}
PATH_LAUNCHES = {"fused": 1, "split": 2, "decode": 1, "segmented": 4}
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the
# dominant kernel (per step for the segmented path, whose roofline entry is the
# whole step), from one ncu capture of the current kernels.  The b8 figure
# is four times the b2 capture: b8 processes four times the units, and the
# traffic is the per-unit inputs, outputs and states.  The long figure comes
# from the l32 capture (a quarter of long's tokens, split into the same 5
# pieces): four times the plan, fused and fix-up launches, whose traffic
# follows the tokens, plus the scan's once, which follows the pieces and
# heads.  Absent = not captured.
MEASURED_TRAFFIC = {
    ("b2", "fused"): 538.023168e6 + 120.249344e6,
    ("b8", "fused"): 4 * (538.023168e6 + 120.249344e6),
    ("decode", "decode"): 545.300224e6 + 491.147776e6,
    # the whole kda_fwd_segmented step: its four launches
    ("long", "segmented"): 4 * (16.128e3 + (1136.457216e6 + 460.735232e6)
                                + (437.124608e6 + 169.482496e6)) + 18.886912e6,
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK), "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed loop runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    return rank, world, local


def max_over_ranks(x: float, world: int) -> float:
    """Slowest rank's value (the step time every rank reports is the max)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(tokens_per_rank: int, world: int, max_ms: float) -> float:
    """Tokens/s of the whole job: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * world / (max_ms * 1e-3)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def oracle_sample(inp, n_units, nthreads, prefix=None):
    """Run the fp64 oracle (token-by-token, as it stands) on the first n_units
    (sequence, head) units, optionally only their first `prefix` tokens;
    returns (seconds, token-heads)."""
    import numpy as np
    import torch
    import oracle
    from chunked_gated_delta_11_gb300 import synth
    H = inp["H"]
    units = [(u // H, u % H) for u in range(n_units)]
    sl = [synth.unit_slice(inp, n, h) for n, h in units]
    T = min(s["T_total"] for s in sl) if prefix is None else prefix
    f = lambda t: t[:T].to(torch.float64).numpy()
    # the sampled units side by side as the heads of one sequence
    cat = lambda key: np.concatenate([f(s[key]) for s in sl], axis=1)
    q, k, v, g, b = cat("q"), cat("k"), cat("v"), cat("g_raw"), cat("beta_raw")
    init = None
    if sl[0]["initial_state"] is not None:
        init = np.concatenate([s["initial_state"].to(torch.float64).numpy() for s in sl], axis=1)
    t0 = time.perf_counter()
    oracle.fwd_raw(q, k, v, g, b, inp["scale"], inp["lower_bound"], init, nthreads=nthreads)
    return time.perf_counter() - t0, n_units * T


def run_reference(args):
    """The reference arm: the fp64 oracle on host cores (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return 0
    import torch
    from chunked_gated_delta_11_gb300 import synth
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    inp = synth.workload_inputs(args.workload, device="cpu")
    n_units = min(cores, inp["N"] * inp["H"])
    full = min(int(x) for x in (inp["cu_seqlens"].diff() if inp["cu_seqlens"] is not None
                                else [inp["T_total"] // inp["N"]]))
    # size each step's sample so that warm-up + timed steps take about 90 s
    sec, th = oracle_sample(inp, 1, 1, prefix=min(full, 512))
    per_token = sec / th
    target = 90.0 / (args.steps + args.warmup)
    prefix = int(max(16, min(full, target / per_token)) // 16 * 16)
    for _ in range(args.warmup):
        oracle_sample(inp, n_units, cores, prefix)
    total_s, total_th = 0.0, 0
    for _ in range(args.steps):
        s, th = oracle_sample(inp, n_units, cores, prefix)
        total_s += s
        total_th += th
    tok_s = total_th / inp["H"] / total_s
    sample = (f"first {prefix} tokens of {n_units} (sequence, head) units of workload "
              f"{args.workload} per step (token-heads / H = tokens)")
    line = {
        "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": f"{args.workload}: {WORKLOAD_TEXT.get(args.workload, '')}"},
        "cpu_baseline": {"value": tok_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": tok_s, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=30)
    ap.add_argument("--repeats", type=int, default=5,
                    help="timed loops of --steps steps each; the line reports their median")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="b8")
    ap.add_argument("--path", choices=["fused", "split", "decode", "segmented"], default=None,
                    help="fused: kda_fwd_fused (one kernel); split: kda_fwd (K1 + K2); decode: "
                         "kda_decode (recurrent schedule); segmented: kda_fwd_segmented (every "
                         "sequence in pieces joined by a scan of their state maps, automatic "
                         "piece count).  Default: decode for the decode workload, fused "
                         "otherwise")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-units", type=int, default=0,
                    help="oracle sample size for cpu_baseline (0 = up to 16 units per core)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)

    import torch
    rank, world, local = dist_init()
    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()
    import chunked_gated_delta_11_gb300 as kda
    from chunked_gated_delta_11_gb300 import synth

    peaks, peak_src = load_peaks()
    inp = synth.workload_inputs(args.workload, device="cuda",
                                seed=synth.WORKLOADS[args.workload].seed + 1000 * rank)
    T, H, N = inp["T_total"], inp["H"], inp["N"]
    ws = torch.empty(kda.kda_workspace_size(T, H, N), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(inp["q"])
    fs = torch.empty((N, H, 128, 128), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    a = (inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"], inp["scale"],
         inp["lower_bound"], inp["initial_state"], inp["cu_seqlens"])

    def step_split():
        kda.kda_fwd(*a, N=N, out=out, final_state=fs, workspace=ws, stream=stream)

    def step_fused():
        kda.kda_fwd_fused(*a, N=N, out=out, final_state=fs, stream=stream)

    def step_decode():
        kda.kda_decode(*a, N=N, out=out, final_state=fs, stream=stream)

    if args.path is None:
        args.path = "decode" if args.workload == "decode" else "fused"
    segments = kda.kda_segments_auto(T, H, N) if args.path == "segmented" else 1
    ws_seg = torch.empty(max(1, kda.kda_segmented_workspace_size(T, H, N, segments=segments)),
                         dtype=torch.uint8, device="cuda") if args.path == "segmented" else None

    def step_segmented():
        kda.kda_fwd_segmented(*a, N=N, segments=segments, out=out, final_state=fs,
                              workspace=ws_seg, stream=stream)

    step = {"fused": step_fused, "split": step_split, "decode": step_decode,
            "segmented": step_segmented}[args.path]

    # a working set below the L2 would stay cached from step to step: then a
    # buffer twice the L2 is written before every timed step, outside the
    # step's own pair of events
    l2_bytes = int(getattr(torch.cuda.get_device_properties(local), "L2_cache_size", 0)
                   or 129 * 2 ** 20)
    working = sum(t.numel() * t.element_size() for t in
                  (inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"], out, fs,
                   inp["initial_state"]) if isinstance(t, torch.Tensor))
    flush = (torch.empty(2 * l2_bytes // 4, dtype=torch.float32, device="cuda")
             if working < l2_bytes else None)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert kda.kda_device_status() == 0
    sampler = ClockSampler(local)
    sampler.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    rep_ms = []
    for _ in range(max(1, args.repeats)):
        # each repeat: exactly --steps steps between a barrier + synchronize on both sides
        barrier(world)
        torch.cuda.synchronize()
        if flush is None:
            ev0.record(stream)
            for _ in range(args.steps):
                step()
            ev1.record(stream)
            torch.cuda.synchronize()
            total = ev0.elapsed_time(ev1)
        else:
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(args.steps)]
            for e0, e1 in evs:
                flush.zero_()
                e0.record(stream)
                step()
                e1.record(stream)
            torch.cuda.synchronize()
            total = sum(e0.elapsed_time(e1) for e0, e1 in evs)
        barrier(world)
        rep_ms.append(max_over_ranks(total / args.steps, world))
    clocks = sampler.stop()
    ms = statistics.median(rep_ms)
    assert kda.kda_device_status() == 0

    # the other path, and the split path's per-kernel durations, on the same stream
    reps = max(10, min(args.steps, 50))
    other = step_split if args.path in ("fused",) else step_fused
    for _ in range(3):
        other()
    ev0.record(stream)
    for _ in range(reps):
        other()
    ev1.record(stream)
    torch.cuda.synchronize()
    other_ms = ev0.elapsed_time(ev1) / reps
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    k1_ms = k2_ms = 0.0
    for _ in range(reps):
        evs[0].record(stream)
        kda.kda_chunk_prep(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"],
                           inp["scale"], inp["lower_bound"], ws, inp["cu_seqlens"], N=N,
                           stream=stream)
        evs[1].record(stream)
        kda.kda_chunk_recurrence(ws, T, H, out, inp["initial_state"], fs, inp["cu_seqlens"],
                                 N=N, stream=stream)
        evs[2].record(stream)
        evs[2].synchronize()
        k1_ms += evs[0].elapsed_time(evs[1]) / reps
        k2_ms += evs[1].elapsed_time(evs[2]) / reps

    # end to end through the public API with pinned host buffers
    host = {key: (inp[key].cpu().pin_memory() if inp[key] is not None else None)
            for key in ("q", "k", "v", "g_raw", "beta_raw", "initial_state", "cu_seqlens")}
    out_h = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    fs_h = torch.empty(fs.shape, dtype=fs.dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = out_h.numel() * out_h.element_size() + fs_h.numel() * fs_h.element_size()

    ws_host = torch.empty(kda.kda_fwd_host_workspace_size(T, H, N, host["cu_seqlens"],
                                                          schedule=args.path),
                          dtype=torch.uint8, device="cuda")

    def e2e_step():
        # kda_fwd_host through the C ABI: host buffers in, copies and passes
        # pipelined inside libkda, host buffers out
        kda.kda_forward_host(host["q"], host["k"], host["v"], host["g_raw"], host["beta_raw"],
                             inp["scale"], inp["lower_bound"], host["initial_state"],
                             host["cu_seqlens"], N=N, out=out_h, final_state=fs_h, stream=stream,
                             schedule=args.path, workspace=ws_host)

    e2e_ms = None
    if args.e2e_steps > 0:
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        ev0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        ev1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(ev0.elapsed_time(ev1) / args.e2e_steps, world)
        assert kda.kda_device_status() == 0

    # Independent batches of the same shape on two alternating streams, each
    # with its own outputs: consecutive steps overlap, so the SMs a single
    # step leaves idle at its tail (256 units on 152 SMs at b8) take the next
    # batch's units.  Reported beside the headline, which stays one step at
    # a time on one stream.
    pipelined = None
    if args.path == "fused" and flush is None and world == 1:
        side = [torch.cuda.Stream(), torch.cuda.Stream()]
        bufs = [(torch.empty_like(out), torch.empty_like(fs)) for _ in range(2)]

        def step_on(i):
            o, f = bufs[i & 1]
            kda.kda_fwd_fused(*a, N=N, out=o, final_state=f, stream=side[i & 1])

        for i in range(4):
            step_on(i)
        torch.cuda.synchronize()
        n_pipe = max(10, min(args.steps, 100))
        ev0.record(stream)
        for sd in side:
            sd.wait_event(ev0)
        for i in range(n_pipe):
            step_on(i)
        for sd in side:
            done = torch.cuda.Event()
            done.record(sd)
            stream.wait_event(done)
        ev1.record(stream)
        torch.cuda.synchronize()
        assert kda.kda_device_status() == 0
        pipe_ms = ev0.elapsed_time(ev1) / n_pipe
        pipelined = {"streams": 2, "steps": n_pipe, "ms_per_step": pipe_ms,
                     "value": T / (pipe_ms * 1e-3), "unit": "tokens/s",
                     "what": "independent batches of this shape on two alternating streams "
                             "with separate outputs; consecutive steps overlap"}

    tokens_per_step = T * world
    value = whole_job_rate(T, world, ms)
    units = N * H
    init_bytes = STATE_BYTES * units if inp["initial_state"] is not None else 0
    alg_bytes = ALG_BYTES_PER_TOKEN_HEAD * T * H + STATE_BYTES * units + init_bytes
    alg_flop = ALG_FLOP_PER_TOKEN_HEAD * T * H
    hbm = float(peaks["hbm_gbs"])
    tc = float(peaks["bf16_tflops"])
    achieved = alg_bytes / (ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "repeats": {"n": len(rep_ms), "ms_per_step": rep_ms, "median": ms, "min": min(rep_ms),
                    "max": max(rep_ms), "spread": (max(rep_ms) - min(rep_ms)) / ms},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": f"{args.workload}: {WORKLOAD_TEXT.get(args.workload, '')}",
            **({"segments": segments} if args.path == "segmented" else {}),
            "global_batch": N * world, "seq_len": T // N if inp["cu_seqlens"] is None else None,
            "heads": H, "head_dim": 128, "tokens_per_step": tokens_per_step,
            "l2": ("L2 flushed before every step (working set %.0f MB below the %.0f MB L2)"
                   % (working / 1e6, l2_bytes / 1e6) if flush is not None else
                   "states larger than L2 (no flush)" if args.workload == "decode"
                   else "inputs larger than L2 (no flush)"),
            "parallelism": f"replicas x{world}", "path": PATH_TEXT[args.path],
        },
        "roofline": {
            "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "traffic": MEASURED_TRAFFIC.get((args.workload, args.path)),
            "kernel": PATH_KERNEL[args.path],
            "alg_bytes_per_launch": alg_bytes, "alg_flop_per_launch": alg_flop,
            "tensor_frac": alg_flop / (ms * 1e-3) / 1e12 / tc,
            "roofline_ms": max(alg_bytes / hbm / 1e9, alg_flop / tc / 1e12) * 1e3,
            "peak_source": f"{peak_src} (hbm_gbs; bf16_tflops for tensor_frac)",
        },
        "kernels": {
            "fused_kernel": {"ms": ms if args.path == "fused" else other_ms},
            "split_path": {"ms": ms if args.path == "split" else
                           (other_ms if args.path == "fused" else None),
                           "chunk_prep_kernel_ms": k1_ms, "recurrence_kernel_ms": k2_ms},
            **({"decode_kernel": {"ms": ms}} if args.path == "decode" else {}),
            **({"segmented_path": {"ms": ms, "segments": segments}}
               if args.path == "segmented" else {}),
        },
        "clocks": clocks,
        "e2e": None if e2e_ms is None else {
            "value": tokens_per_step / (e2e_ms * 1e-3), "unit": "tokens/s",
            "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "api": "kda_fwd_host (C ABI, pinned host buffers)", "copies_declared": True},
        "gpu_launches": PATH_LAUNCHES[args.path] * args.steps * len(rep_ms),
        "pipelined": pipelined,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = os.cpu_count() or 1
        # about 10-100 s of CPU work: the whole step when it has at most
        # 16 units per core (b8 on 16 cores), else 16 units per core
        n_units = args.cpu_units or min(16 * cores, units)
        secs, th = oracle_sample(inp, n_units, cores)
        line["cpu_baseline"] = {
            "value": th / H / secs, "unit": "tokens/s", "cores": min(cores, n_units),
            "kind": "oracle",
            "sample": f"{n_units} (sequence, head) units x {T // N} tokens of the same inputs "
                      f"({secs:.1f} s wall)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
