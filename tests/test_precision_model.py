"""The rounding model of the GPU path, checked against the fp64 oracle (CPU).

A plain numpy restatement of where the kernels round, written from the
chunkwise form ("You Could Have Come Up with Kimi Delta Attention", sec. 6)
and independent of the CUDA sources:

- the normalisation applied to the 16 x 16 matrices and per-token rows (rq,
  rk) instead of the 128-channel factors, which the kernels keep unnormalised
  (q P, k P, k Q, k / P);
- intra-chunk products Mkk = kP (k/P)^T, Mqk = qP (k/P)^T and W' = A' diag(beta
  rk^2) kP with bf16 operands and fp32 accumulation (FlashKDA's chunk-kernel
  precision, "FlashKDA v1: A Deep Dive", sec. 3);
- A' = (I + R')^-1 in fp32 (forward substitution), R' = strictly-lower(diag(beta
  rk^2) Mkk);
- U' = A' diag(beta rk) V with A' diag(beta rk) as a bf16 high part plus
  remainder;
- the first recurrence product on bf16 operands (a bf16 snapshot of the fp32
  state times [Qdec; W] stored as bf16, as FlashKDA's bf16 state), fp32
  accumulation;
- the state update and output correction on tf32 operands (E, Kend and Aqk
  truncated to tf32), fp32 accumulation, the state itself kept in fp32;
- out rounded to bf16.

If this model drifts past the tolerance, a precision choice of the kernels is
wrong whatever the GPU does; the GPU parity tests then check that the kernels
match the oracle.
"""
import numpy as np
import pytest

import oracle
from chunked_gated_delta_11_gb300 import synth

f32 = np.float32
TOL_MAX, TOL_FRO = 1e-2, 5e-3   # max-abs / max|ref| and relative Frobenius


def bf16(x):
    b = np.asarray(x, dtype=f32).view(np.uint32).astype(np.uint64)
    return (((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16).astype(np.uint32).view(f32)


def tf32_trunc(x):
    return (np.asarray(x, dtype=f32).view(np.uint32) & np.uint32(0xFFFFE000)).view(f32)


def mm(a, b):
    return (a.astype(np.float64) @ b.astype(np.float64)).astype(f32)


def mm3(a, b):
    """a @ b from bf16 high/low splits of both operands, low*low dropped."""
    ah, bh = bf16(a), bf16(b)
    al, bl = bf16(a - ah), bf16(b - bh)
    return (ah.astype(np.float64) @ bh + ah.astype(np.float64) @ bl
            + al.astype(np.float64) @ bh).astype(f32)


def model_forward(inp):
    q, k, v = (inp[n].float().numpy() for n in ("q", "k", "v"))
    g = inp["g_raw"].float().numpy()
    br = inp["beta_raw"].float().numpy()
    T, H, D = q.shape
    N = inp["N"]
    L = T // N
    s, lb = f32(inp["scale"]), f32(inp["lower_bound"])
    out = np.zeros((T, H, D), f32)
    fs = np.zeros((N, H, D, D), f32)
    for n in range(N):
        S = (np.zeros((H, D, D), f32) if inp["initial_state"] is None
             else inp["initial_state"][n].numpy().astype(f32).copy())
        for c0 in range(n * L, (n + 1) * L, 16):
            sl = slice(c0, min(c0 + 16, (n + 1) * L))
            nc = sl.stop - sl.start

            def tile(x):
                t = np.zeros((H, 16, D), f32)
                t[:, :nc] = x[sl].transpose(1, 0, 2)
                return t
            qq, kk, vv, gg = tile(q), tile(k), tile(v), tile(g)
            beta = np.zeros((H, 16), f32)
            beta[:, :nc] = 1 / (1 + np.exp(-br[sl].T.astype(np.float64)))
            rq = s / np.sqrt((qq * qq).sum(-1) + f32(1e-6))
            rk = 1 / np.sqrt((kk * kk).sum(-1) + f32(1e-6))
            a = np.ones((H, 16, D), f32)
            a[:, :nc] = np.exp2(f32(lb * np.log2(np.e)) / (1 + np.exp(-gg[:, :nc])))
            P = np.cumprod(a, axis=1, dtype=f32)
            dl = P[:, -1]
            Qs = np.ones_like(a)
            Qs[:, :-1] = np.cumprod(a[:, ::-1], axis=1, dtype=f32)[:, ::-1][:, 1:]
            Qu = qq * P
            Ku = kk * P
            Ke = kk * Qs
            Ki = Ke / dl[:, None, :]
            Mkk = mm(bf16(Ku), bf16(Ki).transpose(0, 2, 1))
            Mqk = mm(bf16(Qu), bf16(Ki).transpose(0, 2, 1))
            cw = beta * rk * rk
            cu = beta * rk
            R = np.tril(cw[:, :, None] * Mkk, -1)
            I = np.eye(16)
            A = np.linalg.inv(I + R.astype(np.float64)).astype(f32)
            Aw = A * cw[:, None, :]
            Au = A * cu[:, None, :]
            Au_hi = bf16(Au)
            W = mm(bf16(Aw), bf16(Ku))
            U = mm(Au_hi, vv) + mm(bf16(Au - Au_hi), vv)
            Qd = Qu                 # the record leaves rq out of Qdec and Aqk'
            Aqk = np.tril(Mqk)
            D1 = mm(bf16(S), bf16(np.concatenate([W, Qd], 1)).transpose(0, 2, 1))
            E = tf32_trunc(U - D1[:, :, :16].transpose(0, 2, 1))
            O = rq[..., None] * (D1[:, :, 16:].transpose(0, 2, 1) + mm(tf32_trunc(Aqk), E))
            S = S * dl[:, None, :] + mm(E.transpose(0, 2, 1), tf32_trunc(Ke))
            out[sl] = bf16(O[:, :nc]).transpose(1, 0, 2)
        fs[n] = S
    return out, fs


def check(got, ref, what):
    d = got.astype(np.float64) - ref
    mx = np.abs(d).max() / np.abs(ref).max()
    fro = np.linalg.norm(d) / np.linalg.norm(ref)
    assert mx <= TOL_MAX and fro <= TOL_FRO, f"{what}: max {mx:.2e} fro {fro:.2e}"
    return mx, fro


@pytest.mark.parametrize("T,H,g_mean,init,seed", [
    (64, 1, 0.0, None, 0),        # the 4-chunk single-head case
    (1024, 2, 0.0, 0.02, 1),      # initial state, typical decay
    (1024, 2, 2.0, None, 4),      # g_raw ~ N(2, 1): fast decay
    (2048, 2, -6.0, None, 5),     # retention near 1: long accumulation
    (1000, 2, 0.0, 0.02, 7),      # ragged tail chunk (1000 = 62 * 16 + 8)
])
def test_rounding_model_within_tolerance(T, H, g_mean, init, seed):
    inp = synth.make_inputs(T, H, 1, seed=seed, g_mean=g_mean, init_std=init)
    F = lambda t: None if t is None else t.double().numpy()
    ro, rs = oracle.fwd_raw(F(inp["q"]), F(inp["k"]), F(inp["v"]), F(inp["g_raw"]),
                            F(inp["beta_raw"]), inp["scale"], inp["lower_bound"],
                            F(inp["initial_state"]))
    o, st = model_forward(inp)
    check(o, np.asarray(ro), "out")
    check(st, np.asarray(rs), "final_state")
