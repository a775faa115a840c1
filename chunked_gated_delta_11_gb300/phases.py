"""Per-phase cycles of the recurrence's serial chain, from kda_profile_phases.

For the split path's recurrence kernel (records streamed from HBM) and for the
fused kernel, thread 0 of the first (sequence, head) CTA stamps the SM clock
at the phase boundaries of every chunk; this script runs one pass of each on a
workload of N equal sequences and prints, per phase, the median and mean SM
cycles over the chunks (the first 8 chunks left out as warm-up):

  MMA1        first MMA issued -> complete  ([Qdec ; W'] S^T, 8 bf16 steps)
  e' pass     -> corrected errors written to tensor memory (second MMA issued)
  MMA2        -> complete  ([S | O] += E'^T [Kend' ; Aqk']^T, 2 tf32 steps)
  wait record -> the next chunk's record is in shared memory
  snapshot    -> outputs read, bf16 snapshot written and decay applied, next MMA1 issued
  period      one chunk, MMA1 issue to the next MMA1 issue

  python -m chunked_gated_delta_11_gb300.phases [--workload b2] [--chunks 256]
"""
from __future__ import annotations

import argparse
import ctypes

import numpy as np
import torch

from . import _check, _ptr, kda_workspace_size, load, synth

PHASES = [("MMA1", 0, 1), ("e' pass", 1, 2), ("MMA2", 2, 3), ("wait record", 3, 4),
          ("snapshot", 4, 5), ("period", 0, 8)]


def run(kernel: int, inp: dict, max_chunks: int):
    T, H, N = inp["T_total"], inp["H"], inp["N"]
    out = torch.empty_like(inp["q"])
    fs = torch.empty((N, H, 128, 128), dtype=torch.float32, device="cuda")
    stamps = torch.zeros(8 * max_chunks, dtype=torch.int64, device="cuda")
    nb = kda_workspace_size(T, H, N)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda") if kernel == 0 else None
    st = load().kda_profile_phases(kernel, _ptr(inp["q"]), _ptr(inp["k"]), _ptr(inp["v"]),
                                   _ptr(inp["g_raw"]), _ptr(inp["beta_raw"]), inp["scale"],
                                   inp["lower_bound"], T, H, N, 128, _ptr(out), _ptr(fs),
                                   _ptr(ws), nb if ws is not None else 0, _ptr(stamps),
                                   max_chunks, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    _check(st, "kda_profile_phases")
    torch.cuda.synchronize()
    return stamps.view(max_chunks, 8).cpu().numpy()


def table(stamps: np.ndarray, skip: int = 8):
    s = stamps[skip:-1].astype(np.float64)
    nxt = stamps[skip + 1:, 0].astype(np.float64)
    rows = {}
    for name, a, b in PHASES:
        d = (nxt - s[:, 0]) if b == 8 else (s[:, b] - s[:, a])
        rows[name] = (float(np.median(d)), float(np.mean(d)))
    return rows


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="b2")
    ap.add_argument("--chunks", type=int, default=256)
    args = ap.parse_args()
    inp = synth.workload_inputs(args.workload, device="cuda")
    assert inp["cu_seqlens"] is None, "equal sequences only"
    chunks = min(args.chunks, inp["T_total"] // inp["N"] // 16)
    res = {name: table(run(kernel, inp, chunks)) for name, kernel in
           (("recurrence_kernel (K2)", 0), ("fused_kernel", 1))}
    print(f"workload {args.workload}: SM cycles per chunk, first (sequence, head) CTA, "
          f"chunks 8..{chunks - 2}")
    print("| phase | " + " | ".join(f"{k} median | mean" for k in res) + " |")
    print("|---|" + "---|---|" * len(res))
    for name, _, _ in PHASES:
        print(f"| {name} | " + " | ".join(f"{res[k][name][0]:.0f} | {res[k][name][1]:.0f}"
                                          for k in res) + " |")


if __name__ == "__main__":
    main()
