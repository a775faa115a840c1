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


class _Accum:
    """Running max |err|, max |ref|, sum err^2 and sum ref^2 over blocks."""

    def __init__(self):
        self.max_d = self.max_r = self.sd2 = self.sr2 = 0.0
        self.finite = True
        self.count = 0

    def add(self, got, ref):
        got = np.asarray(got, dtype=np.float64)
        ref = np.asarray(ref, dtype=np.float64)
        if got.size == 0:
            return
        self.finite &= bool(np.all(np.isfinite(got)))
        d = got - ref
        self.max_d = max(self.max_d, float(np.abs(d).max()))
        self.max_r = max(self.max_r, float(np.abs(ref).max()))
        self.sd2 += float((d * d).sum())
        self.sr2 += float((ref * ref).sum())
        self.count += got.size

    def errors(self):
        mx = self.max_d / self.max_r if self.max_r > 0 else self.max_d
        fro = (self.sd2 / self.sr2) ** 0.5 if self.sr2 > 0 else self.sd2 ** 0.5
        return mx, fro


def stream_parity(inp, results, slice_tokens=4096, nthreads=None):
    """Whole-tensor parity of full-size runs against the oracle.

    inp: the case (device tensors are fine); results: {name: (out, final_state)}
    from the GPU.  The oracle runs sequence by sequence in time slices of at most
    `slice_tokens` tokens over all heads, each slice starting from the fp64 state
    the previous one left (exact: the recurrence is a left-to-right scan), so host
    memory stays bounded.  Every element of `out` and of the final state enters
    the global errors; returns {name: {"out": (max_rel, fro), "state": ...}} and
    asserts the tolerance on each."""
    H, N, T = inp["H"], inp["N"], inp["T_total"]
    if inp["cu_seqlens"] is not None:
        cu = [int(x) for x in inp["cu_seqlens"].cpu().tolist()]
    else:
        L = T // N
        cu = [n * L for n in range(N + 1)]
    acc = {name: (_Accum(), _Accum()) for name in results}
    init = inp["initial_state"]
    for n in range(N):
        bos, eos = cu[n], cu[n + 1]
        state = None if init is None else f64(init[n:n + 1])
        for a in range(bos, eos, slice_tokens):
            b = min(a + slice_tokens, eos)
            ro, rs = oracle.fwd_raw(*(f64(inp[key][a:b]) for key in ("q", "k", "v", "g_raw",
                                                                     "beta_raw")),
                                    inp["scale"], inp["lower_bound"], state, N=1,
                                    nthreads=nthreads)
            for name, (out, _) in results.items():
                acc[name][0].add(f64(out[a:b]), ro)
            state = rs
        if state is None:
            state = np.zeros((1, H, inp["D"], inp["D"]))
        for name, (_, fs) in results.items():
            acc[name][1].add(f64(fs[n:n + 1]), state)
    report = {}
    for name, (ao, as_) in acc.items():
        report[name] = {"out": ao.errors(), "state": as_.errors()}
        for what, a in (("out", ao), ("final_state", as_)):
            mx, fro = a.errors()
            print(f"[parity] {name} {what} (all {a.count} elements): max_rel {mx:.3e} fro {fro:.3e}")
            assert a.finite, f"{name} {what}: non-finite values"
            assert mx <= MAX_REL and fro <= FRO_REL, f"{name} {what}: max_rel {mx:.3e} fro {fro:.3e}"
    return report
