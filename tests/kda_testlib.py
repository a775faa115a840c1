"""Helpers shared by the GPU parity tests: run the fp64 oracle on the same
seeded inputs and compare with the tolerance the method's error budget sets
(max |err| <= 1e-2 * max|ref| and ||err||_F / ||ref||_F <= 5e-3, on the output
and on the final fp32 state)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from chunked_gated_delta_11_gb300 import synth

MAX_REL = 1e-2
FRO_REL = 5e-3


def f64(t):
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


def oracle_case(inp, nthreads=None):
    """Oracle (out, final_state) for a whole case (small sizes only)."""
    cu = None if inp["cu_seqlens"] is None else inp["cu_seqlens"].cpu().numpy()
    return oracle.fwd_raw(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["g_raw"]),
                          f64(inp["beta_raw"]), inp["scale"], inp["lower_bound"],
                          f64(inp["initial_state"]), cu, N=inp["N"], nthreads=nthreads)


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    d = got - ref
    scale = np.abs(ref).max() if ref.size else 0.0
    max_rel = np.abs(d).max() / scale if ref.size and scale > 0 else float(np.abs(d).max() if d.size else 0.0)
    nref = np.linalg.norm(ref)
    fro = np.linalg.norm(d) / nref if nref > 0 else float(np.linalg.norm(d))
    return float(max_rel), float(fro)


def assert_close(got, ref, what):
    mx, fro = errors(got, ref)
    print(f"[parity] {what}: max_rel {mx:.3e} fro {fro:.3e}")
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert mx <= MAX_REL and fro <= FRO_REL, f"{what}: max_rel {mx:.3e} fro {fro:.3e}"
    return mx, fro


def compare_units(inp, out, final_state, units, nthreads=None):
    """Check sampled (sequence, head) units of a large case one by one."""
    res = []
    o_got, s_got, o_ref, s_ref = [], [], [], []
    for n, h in units:
        u = synth.unit_slice(inp, n, h)
        ro, rs = oracle_case(u, nthreads=nthreads)
        o_got.append(f64(out[u["bos"]:u["eos"], h:h + 1]))
        o_ref.append(ro)
        s_got.append(f64(final_state[n:n + 1, h:h + 1]))
        s_ref.append(rs)
    og = np.concatenate([x.reshape(-1) for x in o_got])
    orf = np.concatenate([x.reshape(-1) for x in o_ref])
    sg = np.concatenate([x.reshape(-1) for x in s_got])
    sr = np.concatenate([x.reshape(-1) for x in s_ref])
    res.append(assert_close(og, orf, f"out over units {units}"))
    res.append(assert_close(sg, sr, f"final_state over units {units}"))
    return res
