"""Seeded synthetic inputs for the KDA forward pass.

This module only draws random numbers and packs them into the tensor layout of
the C-ABI (``[T_total, H, D]`` bf16 rows, ``[T_total, H]`` bf16 beta, fp32
``[N, H, V, K]`` states, int32 ``cu_seqlens``).  It holds none of the method's
arithmetic, so both the CUDA path and the fp64 oracle can be fed from it.

Workloads (all D = d_k = d_v = 128, lower_bound = -5, scale = 128 ** -0.5):

======  =====================================================================
 name    shape and distributions
======  =====================================================================
 tiny    1 sequence of 64 tokens (4 chunks), H = 1; q, k, v, g_raw, beta_raw
         ~ N(0, 1) rounded to bf16; zero initial state
 h16     1 sequence of 4096 tokens, H = 16; initial state ~ 0.02 * N(0, 1) fp32
 b8      8 sequences of 8192 tokens, H = 32; zero initial state (throughput
         workload: B = 8, T = 8192)
 varlen  64 packed sequences, lengths uniform in [1, 16384] redrawn while a
         multiple of 16, H = 32; cu_seqlens int32; initial states ~ 0.02 N(0,1)
 long    1 sequence of 131072 tokens, H = 32; g_raw ~ N(2, 1); zero state
 slow    unscored stress variant of ``long`` with g_raw ~ N(-6, 1), i.e.
         retention close to 1 (long-range accumulation)
 b2      profiling size: 2 sequences of 8192 tokens, H = 32
 decode  one serving step: 256 sequences of 1 token, H = 32, initial states
         ~ 0.02 N(0, 1) (the decode regime: moving the states dominates)
 fk96    the shapes of FlashKDA's published benchmark rows ("FlashKDA v1: A
 fk64    Deep Dive", benchmark section; T = 8192, D = 128): 1 sequence of 8192
         tokens, H = 96 or 64; zero initial state
 fk96p   the same rows' "1024 x 8" form: 8 sequences of 1024 tokens, H = 96
 fk64p   or 64, passed packed with cu_seqlens; zero initial states
======  =====================================================================

Draw order is q, k, v, g_raw, beta_raw, initial_state; sequence lengths come
from a separate generator seeded with ``seed + 7919`` so that they do not depend
on the tensor sizes.  Values are drawn in fp32 with ``torch.randn`` and rounded
to bf16 (round to nearest even).  The same (workload, seed, device) always gives
the same bits; CPU and CUDA generators give different streams.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

D = 128
LOWER_BOUND = -5.0
SCALE = D ** -0.5


@dataclass(frozen=True)
class Workload:
    name: str
    H: int
    N: int
    T: int | None            # tokens per sequence (None: variable lengths)
    init_std: float | None   # None: zero initial state
    g_mean: float = 0.0
    max_len: int = 0         # variable lengths: upper bound
    seed: int = 0
    packed: bool = False     # equal lengths T, passed with cu_seqlens


WORKLOADS = {
    "tiny": Workload("tiny", H=1, N=1, T=64, init_std=None, seed=0),
    "h16": Workload("h16", H=16, N=1, T=4096, init_std=0.02, seed=1),
    "b8": Workload("b8", H=32, N=8, T=8192, init_std=None, seed=2),
    "varlen": Workload("varlen", H=32, N=64, T=None, init_std=0.02, max_len=16384, seed=3),
    "long": Workload("long", H=32, N=1, T=131072, init_std=None, g_mean=2.0, seed=4),
    "slow": Workload("slow", H=32, N=1, T=131072, init_std=None, g_mean=-6.0, seed=5),
    # profiling size: like b8 with 2 sequences (inputs 537 MB, still larger than L2)
    "b2": Workload("b2", H=32, N=2, T=8192, init_std=None, seed=6),
    # profiling size for the segmented path: one sequence, like long (g_raw ~ N(2, 1))
    "l32": Workload("l32", H=32, N=1, T=32768, init_std=None, g_mean=2.0, seed=8),
    # one decode step of a serving batch: 256 sequences x 1 new token, states in/out
    "decode": Workload("decode", H=32, N=256, T=1, init_std=0.02, seed=7),
    "fk96": Workload("fk96", H=96, N=1, T=8192, init_std=None, seed=9),
    "fk64": Workload("fk64", H=64, N=1, T=8192, init_std=None, seed=10),
    "fk96p": Workload("fk96p", H=96, N=8, T=1024, init_std=None, seed=11, packed=True),
    "fk64p": Workload("fk64p", H=64, N=8, T=1024, init_std=None, seed=12, packed=True),
}


def varlen_lengths(n: int, max_len: int, seed: int, min_len: int = 1) -> list[int]:
    """n lengths uniform in [min_len, max_len], redrawn while a multiple of 16."""
    g = torch.Generator(device="cpu").manual_seed(seed + 7919)
    out = []
    while len(out) < n:
        L = int(torch.randint(min_len, max_len + 1, (1,), generator=g).item())
        if L % 16 != 0:
            out.append(L)
    return out


def cu_from_lengths(lengths) -> torch.Tensor:
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + int(L))
    return torch.tensor(cu, dtype=torch.int32)


def make_inputs(T_total: int, H: int, N: int = 1, *, lengths=None, seed: int = 0,
                init_std: float | None = None, g_mean: float = 0.0, g_std: float = 1.0,
                beta_mean: float = 0.0, device="cpu", D: int = D) -> dict:
    """Draw one case.  With ``lengths`` the sequences are packed and described
    by ``cu_seqlens``; otherwise there are N equal sequences of T_total / N."""
    device = torch.device(device)
    g = torch.Generator(device=device).manual_seed(int(seed))
    if lengths is not None:
        lengths = [int(x) for x in lengths]
        N = len(lengths)
        T_total = sum(lengths)
        cu = cu_from_lengths(lengths)
    else:
        if T_total % N:
            raise ValueError("T_total must be a multiple of N without cu_seqlens")
        cu = None

    def randn(*shape, mean=0.0, std=1.0):
        x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        if mean != 0.0:
            x.add_(mean)
        return x

    q = randn(T_total, H, D).to(torch.bfloat16)
    k = randn(T_total, H, D).to(torch.bfloat16)
    v = randn(T_total, H, D).to(torch.bfloat16)
    g_raw = randn(T_total, H, D, mean=g_mean, std=g_std).to(torch.bfloat16)
    beta_raw = randn(T_total, H, mean=beta_mean).to(torch.bfloat16)
    init = None
    if init_std is not None:
        init = randn(N, H, D, D, std=init_std)
    return {
        "q": q, "k": k, "v": v, "g_raw": g_raw, "beta_raw": beta_raw,
        "initial_state": init,
        "cu_seqlens": None if cu is None else cu.to(device),
        "T_total": T_total, "H": H, "N": N, "D": D,
        "scale": SCALE, "lower_bound": LOWER_BOUND,
    }


def workload_inputs(name: str, device="cpu", seed: int | None = None) -> dict:
    """Inputs of one named workload (see the module docstring)."""
    w = WORKLOADS[name]
    seed = w.seed if seed is None else seed
    if w.T is None or w.packed:
        lengths = [w.T] * w.N if w.packed else varlen_lengths(w.N, w.max_len, seed)
        return make_inputs(0, w.H, lengths=lengths, seed=seed, init_std=w.init_std,
                           g_mean=w.g_mean, device=device)
    return make_inputs(w.T * w.N, w.H, w.N, seed=seed, init_std=w.init_std,
                       g_mean=w.g_mean, device=device)


def unit_slice(inp: dict, n: int, h: int) -> dict:
    """The inputs of one (sequence n, head h) unit, on the CPU, as a one-head,
    one-sequence case (used to compare sampled units against the oracle)."""
    if inp["cu_seqlens"] is not None:
        cu = inp["cu_seqlens"].cpu()
        bos, eos = int(cu[n]), int(cu[n + 1])
    else:
        L = inp["T_total"] // inp["N"]
        bos, eos = n * L, (n + 1) * L
    sl = slice(bos, eos)
    out = {
        "q": inp["q"][sl, h:h + 1].cpu(), "k": inp["k"][sl, h:h + 1].cpu(),
        "v": inp["v"][sl, h:h + 1].cpu(), "g_raw": inp["g_raw"][sl, h:h + 1].cpu(),
        "beta_raw": inp["beta_raw"][sl, h:h + 1].cpu(),
        "initial_state": None, "cu_seqlens": None,
        "T_total": eos - bos, "H": 1, "N": 1, "D": inp["D"],
        "scale": inp["scale"], "lower_bound": inp["lower_bound"],
        "bos": bos, "eos": eos,
    }
    if inp["initial_state"] is not None:
        out["initial_state"] = inp["initial_state"][n:n + 1, h:h + 1].cpu()
    return out
