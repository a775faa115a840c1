"""Pins of the fp64 oracle against facts the pages and the mathematics fix.

Nothing here retypes the oracle's own loops: every expected value is a closed
form, an invariant, a special case that the page writes as a different formula,
a library routine (numpy.linalg.inv), or the oracle's other schedule (the
chunkwise form of "You Could Have Come Up with Kimi Delta Attention" sec. 6
against the token-by-token form of sec. 4).  Each test names the passage.
"""
import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(1234)


def rand_case(T, H, K, V=None, rng=RNG, lb=-5.0, init=False, N=1):
    V = K if V is None else V
    q = rng.standard_normal((T, H, K))
    k = rng.standard_normal((T, H, K))
    v = rng.standard_normal((T, H, V))
    g = rng.standard_normal((T, H, K))
    b = rng.standard_normal((T, H))
    qh, kh, la, beta = oracle.prepare(q, k, g, b, lb, eps=0.0)
    S0 = 0.3 * rng.standard_normal((N, H, V, K)) if init else None
    return dict(q=qh, k=kh, v=v, la=la, beta=beta, S0=S0, K=K, V=V, T=T, H=H, N=N,
                raw=dict(q=q, k=k, g=g, b=b))


def rel(a, b):
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


# ---------------------------------------------------------------------------
# P-a  chunkwise schedule == token-by-token schedule (sec. 6: "It must produce
#      exactly the same states and outputs as the token-by-token recurrence")
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("K", [4, 8, 128])
@pytest.mark.parametrize("C", [1, 4, 16, 64])
def test_pa_chunkwise_equals_recurrent(K, C):
    c = rand_case(70, 2, K, init=True)
    s = K ** -0.5
    o0, S0 = oracle.fwd(c["q"], c["k"], c["v"], c["la"], c["beta"], s, c["S0"])
    o1, S1 = oracle.fwd(c["q"], c["k"], c["v"], c["la"], c["beta"], s, c["S0"], chunk=C)
    assert rel(o1, o0) < 1e-12
    assert rel(S1, S0) < 1e-12


def test_pa_chunkwise_varlen_ragged():
    lengths = [1, 15, 16, 17, 33, 0, 5]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    c = rand_case(T, 3, 8, init=True, N=len(lengths))
    s = 8 ** -0.5
    o0, S0 = oracle.fwd(c["q"], c["k"], c["v"], c["la"], c["beta"], s, c["S0"], cu_seqlens=cu)
    o1, S1 = oracle.fwd(c["q"], c["k"], c["v"], c["la"], c["beta"], s, c["S0"], cu_seqlens=cu,
                        chunk=16)
    assert rel(o1, o0) < 1e-12 and rel(S1, S0) < 1e-12


# ---------------------------------------------------------------------------
# P-b  beta = 0: no write, so the state only decays (sec. 4, forget step) and
#      the read is s * S_0 Diag(prod alpha) q_t.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("chunk", [0, 16])
def test_pb_beta_zero_is_pure_decay(chunk):
    c = rand_case(40, 2, 8, init=True)
    beta = np.zeros_like(c["beta"])
    s = 0.7
    o, S = oracle.fwd(c["q"], c["k"], c["v"], c["la"], beta, s, c["S0"], chunk=chunk)
    cum = np.cumsum(c["la"], axis=0)                        # [T, H, K] log prod alpha
    for h in range(2):
        S_T = c["S0"][0, h] * np.exp(cum[-1, h])[None, :]   # column d scaled
        assert rel(S[0, h], S_T) < 1e-13
        for t in range(40):
            o_t = s * (c["S0"][0, h] * np.exp(cum[t, h])[None, :]) @ c["q"][t, h]
            assert rel(o[t, h], o_t) < 1e-12


# ---------------------------------------------------------------------------
# P-c  beta = 1 and a unit key: the write can be read back exactly,
#      S_t k_t = v_t (sec. 2.1), whatever alpha and the prior state are.  With
#      q_t = k_t the read of sec. 4 is then o_t = s * v_t.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("chunk", [0, 4, 16])
def test_pc_read_back_after_full_write(chunk):
    c = rand_case(37, 2, 16, init=True)
    beta = np.ones_like(c["beta"])
    s = 0.25
    o, _ = oracle.fwd(c["k"], c["k"], c["v"], c["la"], beta, s, c["S0"], chunk=chunk)
    np.testing.assert_allclose(o, s * c["v"], rtol=0, atol=1e-12 * np.abs(c["v"]).max())


def test_pc_alpha_one_unit_key_tail_state():
    """alpha = 1 form of the same fact, checked on the final state directly."""
    c = rand_case(9, 1, 8, init=True)
    la = np.zeros_like(c["la"])
    beta = np.ones_like(c["beta"])
    _, S = oracle.fwd(c["q"], c["k"], c["v"], la, beta, 1.0, c["S0"])
    kT, vT = c["k"][-1, 0], c["v"][-1, 0]
    assert np.linalg.norm(S[0, 0] @ kT - vT) <= 1e-12 * np.linalg.norm(vT)


# ---------------------------------------------------------------------------
# P-d  the three inverses of I + R agree with numpy.linalg.inv (sec. 6.3:
#      I + R is unit lower triangular; R nilpotent makes the Neumann series
#      finite).
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("n", [1, 2, 5, 16, 17])
def test_pd_inverses_match_library(n):
    R = np.tril(RNG.standard_normal((n, n)), -1) * 0.4
    ref = np.linalg.inv(np.eye(n) + R)
    for fn in (oracle.neumann_inverse, oracle.product_inverse, oracle.trisolve_inverse):
        A = fn(R)
        assert rel(A, ref) < 1e-11, fn.__name__
        assert rel((np.eye(n) + R) @ A, np.eye(n)) < 1e-12


def test_pd_chunk_factor_inverses_on_workload_blocks():
    """Every 16 x 16 Akk block of a real chunking: (I + R) Akk = I with R read
    back as inv(Akk) - I, which must be strictly lower triangular; and the
    Neumann and product forms of that R reproduce Akk."""
    c = rand_case(64, 2, 128)
    f = oracle.chunk_factors(c["q"], c["k"], c["v"], c["la"], c["beta"], 128 ** -0.5)
    for blk in f["Akk"].reshape(-1, 16, 16):
        R = np.linalg.inv(blk) - np.eye(16)
        assert np.abs(np.triu(R)).max() < 1e-10
        R = np.tril(R, -1)
        assert rel(oracle.neumann_inverse(R), blk) < 1e-10
        assert rel(oracle.product_inverse(R), blk) < 1e-10


# ---------------------------------------------------------------------------
# P-e  locality (sec. 2.1): for x orthogonal to k_t the write leaves S x alone:
#      S_t x = S~_t x = S_{t-1} D_t x.
# ---------------------------------------------------------------------------
def test_pe_write_is_local_in_key_space():
    c = rand_case(12, 1, 8, init=True)
    s = 1.0
    _, S_prev = oracle.fwd(c["q"][:-1], c["k"][:-1], c["v"][:-1], c["la"][:-1], c["beta"][:-1],
                           s, c["S0"])
    _, S_last = oracle.fwd(c["q"], c["k"], c["v"], c["la"], c["beta"], s, c["S0"])
    kT = c["k"][-1, 0]
    x = RNG.standard_normal(8)
    x -= kT * (kT @ x) / (kT @ kT)
    D = np.exp(c["la"][-1, 0])
    np.testing.assert_allclose(S_last[0, 0] @ x, S_prev[0, 0] @ (D * x), atol=1e-12)


# ---------------------------------------------------------------------------
# P-f  the expanded transition forms the page writes separately:
#      KDA  S_t = S_{t-1} D_t (I - beta k k^T) + beta v k^T         (sec. 4.1)
#      GDN  S_t = alpha_t S_{t-1} (I - beta k k^T) + beta v k^T     (sec. 3)
#      DN   S_t = S_{t-1} (I - beta k k^T) + beta v k^T             (sec. 2.3)
# ---------------------------------------------------------------------------
def _expanded(c, la, beta):
    T, H, K = c["k"].shape
    S = c["S0"][0].copy()
    for t in range(T):
        for h in range(H):
            k = c["k"][t, h]
            A = np.diag(np.exp(la[t, h])) @ (np.eye(K) - beta[t, h] * np.outer(k, k))
            S[h] = S[h] @ A + beta[t, h] * np.outer(c["v"][t, h], k)
    return S


@pytest.mark.parametrize("variant", ["kda", "gated", "delta"])
@pytest.mark.parametrize("chunk", [0, 16])
def test_pf_expanded_transition_forms(variant, chunk):
    c = rand_case(33, 2, 8, init=True)
    la = c["la"].copy()
    if variant == "gated":
        la = np.repeat(RNG.uniform(-3, 0, (33, 2, 1)), 8, axis=2)   # scalar alpha_t
    elif variant == "delta":
        la = np.zeros_like(la)
    _, S = oracle.fwd(c["q"], c["k"], c["v"], la, c["beta"], 1.0, c["S0"], chunk=chunk)
    assert rel(S[0], _expanded(c, la, c["beta"])) < 1e-12


# ---------------------------------------------------------------------------
# P-g  one token from a zero state: S = beta v k^T, o = s beta <k|q> v (sec. 4),
#      with q, k the L2-normalised raw inputs.  Also pins prepare().
# ---------------------------------------------------------------------------
def test_pg_single_token_closed_form():
    K = 128
    q = RNG.standard_normal((1, 1, K)) * 3.0
    k = RNG.standard_normal((1, 1, K)) * 0.5
    v = RNG.standard_normal((1, 1, K))
    g = RNG.standard_normal((1, 1, K))
    b = np.array([[0.3]])
    s = K ** -0.5
    o, S = oracle.fwd_raw(q, k, v, g, b, s, -5.0, eps=0.0)
    qh = q[0, 0] / np.linalg.norm(q[0, 0])
    kh = k[0, 0] / np.linalg.norm(k[0, 0])
    beta = 1.0 / (1.0 + np.exp(-0.3))
    np.testing.assert_allclose(S[0, 0], beta * np.outer(v[0, 0], kh), atol=1e-14)
    np.testing.assert_allclose(o[0, 0], s * beta * (kh @ qh) * v[0, 0], atol=1e-14)


def test_pg_prepare_gate_values():
    x = np.array([0.0, 40.0, -40.0, np.log(3.0)])
    g = np.tile(x, 32).reshape(1, 1, 128)
    q = np.ones((1, 1, 128))
    qh, kh, la, beta = oracle.prepare(q, q, g, np.array([[0.0]]), -5.0, eps=0.0)
    la = la[0, 0, :4]
    np.testing.assert_allclose(la, [-2.5, -5.0, 0.0, -5.0 * 0.75], atol=1e-12)
    assert beta[0, 0] == 0.5
    np.testing.assert_allclose(np.linalg.norm(qh[0, 0]), 1.0, atol=1e-15)
    # eps enters as sum(x^2) + eps: a zero vector normalises to zero
    z, _, _, _ = oracle.prepare(np.zeros((1, 1, 4)), q[:, :, :4], g[:, :, :4],
                                np.array([[0.0]]), -5.0, eps=1e-6)
    assert np.all(z == 0.0)


# ---------------------------------------------------------------------------
# P-h  streaming and packing ("flash_kda.fwd API reference": initial/final
#      state chaining; cu_seqlens packs independent sequences).
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("t1", [1, 16, 23])
def test_ph_streaming_split_equals_single_call(t1):
    c = rand_case(50, 2, 8, init=True)
    s = 0.5
    o, S = oracle.fwd(c["q"], c["k"], c["v"], c["la"], c["beta"], s, c["S0"])
    a = slice(0, t1)
    b = slice(t1, 50)
    oa, Sa = oracle.fwd(c["q"][a], c["k"][a], c["v"][a], c["la"][a], c["beta"][a], s, c["S0"])
    ob, Sb = oracle.fwd(c["q"][b], c["k"][b], c["v"][b], c["la"][b], c["beta"][b], s, Sa,
                        chunk=16)
    assert rel(np.concatenate([oa, ob]), o) < 1e-12
    assert rel(Sb, S) < 1e-12


def test_ph_varlen_equals_separate_calls():
    lengths = [7, 0, 31, 16]
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    c = rand_case(int(cu[-1]), 2, 8, init=True, N=4)
    s = 0.5
    o, S = oracle.fwd(c["q"], c["k"], c["v"], c["la"], c["beta"], s, c["S0"], cu_seqlens=cu)
    for n in range(4):
        sl = slice(cu[n], cu[n + 1])
        on, Sn = oracle.fwd(c["q"][sl], c["k"][sl], c["v"][sl], c["la"][sl], c["beta"][sl], s,
                            c["S0"][n:n + 1])
        if lengths[n]:
            assert rel(o[sl], on) < 1e-13
        assert rel(S[n], Sn[0]) < 1e-13
    # equal-length batch without cu_seqlens == the same batch with it
    c2 = rand_case(48, 2, 8, init=True, N=3)
    oA, SA = oracle.fwd(c2["q"], c2["k"], c2["v"], c2["la"], c2["beta"], s, c2["S0"], N=3)
    oB, SB = oracle.fwd(c2["q"], c2["k"], c2["v"], c2["la"], c2["beta"], s, c2["S0"],
                        cu_seqlens=[0, 16, 32, 48])
    assert rel(oA, oB) == 0.0 and rel(SA, SB) == 0.0


# ---------------------------------------------------------------------------
# Per-key-channel decay and its direction (sec. 4: "the key channels are the
# columns of S"): with keys e_0, e_1, ... (distinct basis vectors) and beta = 1
# each write lands in its own column and is then scaled only by that column's
# later retention factors:  S_T[:, j] = v_j * prod_{u > j} alpha_u[j].
# ---------------------------------------------------------------------------
def test_columnwise_decay_closed_form():
    K, T = 8, 6
    k = np.zeros((T, 1, K))
    for t in range(T):
        k[t, 0, t] = 1.0
    v = RNG.standard_normal((T, 1, K))
    la = RNG.uniform(-2, 0, (T, 1, K))
    beta = np.ones((T, 1))
    q = RNG.standard_normal((T, 1, K))
    o, S = oracle.fwd(q, k, v, la, beta, 1.0)
    expect = np.zeros((K, K))
    for j in range(T):
        expect[:, j] = v[j, 0] * np.exp(la[j + 1:, 0, j].sum())
    np.testing.assert_allclose(S[0, 0], expect, atol=1e-14)
    # read at the last token: o_T = S_T q_T
    np.testing.assert_allclose(o[-1, 0], expect @ q[-1, 0], atol=1e-13)


# ---------------------------------------------------------------------------
# Invariants: outputs are linear in v from a zero state, and invariant to a
# positive rescaling of raw q and k (L2 normalisation, "FlashKDA Delta Attention
# Algorithm", Core Architecture).
# ---------------------------------------------------------------------------
def test_linear_in_values_and_norm_invariance():
    c = rand_case(29, 2, 16)
    r = c["raw"]
    v1 = RNG.standard_normal(c["v"].shape)
    v2 = RNG.standard_normal(c["v"].shape)
    f = lambda vv, qs=1.0, ks=1.0: oracle.fwd_raw(r["q"] * qs, r["k"] * ks, vv, r["g"], r["b"],
                                                   0.3, -5.0, eps=0.0)[0]
    np.testing.assert_allclose(f(2.0 * v1 - 3.0 * v2), 2.0 * f(v1) - 3.0 * f(v2), atol=1e-12)
    np.testing.assert_allclose(f(v1, qs=7.5, ks=0.01), f(v1), atol=1e-12)


# ---------------------------------------------------------------------------
# Chunk factors reproduce the recurrence (sec. 6.3-6.5): with S_c taken from the
# token-by-token oracle run on the prefix, E^T = U - W S_c^T,
# O_c = Qdec S_c^T + Aqk E^T and S_{c+1} = S_c Diag(dlast) + E Kend match the
# token-by-token outputs and states.
# ---------------------------------------------------------------------------
def test_chunk_factors_reproduce_recurrence():
    T, H, K = 45, 2, 16
    c = rand_case(T, H, K, init=True)
    s = K ** -0.5
    f = oracle.chunk_factors(c["q"], c["k"], c["v"], c["la"], c["beta"], s)
    o_ref, _ = oracle.fwd(c["q"], c["k"], c["v"], c["la"], c["beta"], s, c["S0"])
    for ci, c0 in enumerate(range(0, T, 16)):
        n = min(16, T - c0)
        if c0:
            pre = slice(0, c0)
            _, Sc = oracle.fwd(c["q"][pre], c["k"][pre], c["v"][pre], c["la"][pre],
                               c["beta"][pre], s, c["S0"])
        else:
            Sc = c["S0"]
        end = slice(0, c0 + n)
        _, Sn = oracle.fwd(c["q"][end], c["k"][end], c["v"][end], c["la"][end],
                           c["beta"][end], s, c["S0"])
        for h in range(H):
            W, U = f["W"][ci, h][:n], f["U"][ci, h][:n]
            E = U - W @ Sc[0, h].T
            O = f["Qdec"][ci, h][:n] @ Sc[0, h].T + f["Aqk"][ci, h][:n, :n] @ E
            assert rel(O, o_ref[c0:c0 + n, h]) < 1e-11
            S_next = Sc[0, h] * f["dlast"][ci, h][None, :] + E.T @ f["Kend"][ci, h][:n]
            assert rel(S_next, Sn[0, h]) < 1e-11
            # padding rows beyond the ragged tail are zero
            assert not np.any(f["W"][ci, h][n:]) and not np.any(f["U"][ci, h][n:])


# ---------------------------------------------------------------------------
# Regression record (tests/golden/kda_t5_d4.json, written by make_golden.py
# from the oracle alone): guards the pinned oracle against silent change.
# ---------------------------------------------------------------------------
def test_golden_regression_record():
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "kda_t5_d4.json")
    rec = json.load(open(path))
    c = {k: (np.array(v) if isinstance(v, list) else v) for k, v in rec["inputs"].items()}
    o, S = oracle.fwd_raw(c["q_raw"], c["k_raw"], c["v"], c["g_raw"], c["beta_raw"], c["scale"],
                          c["lower_bound"], eps=c["eps"])
    np.testing.assert_allclose(o, np.array(rec["out"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(S, np.array(rec["final_state"]), rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------
# P-i  affine split.  Each token step is an affine map of the state (sec. 4.1:
#      S_t = S_{t-1} Diag(alpha_t)(I - beta_t k_t k_t^T) + beta_t v_t k_t^T),
#      so a segment maps its start S_0 to S_0 M + X, with M the run from the
#      identity with v = 0 and X the run from zero, and o_t = o^X_t + S_0 y_t
#      where y_t is the first run's output.  Composed over the segments this
#      must reproduce the whole run (the segmented forward pass relies on it).
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("cuts", [[0, 32, 64, 100], [0, 16, 100], [0, 0, 50, 100], [0, 37, 99, 100]])
@pytest.mark.parametrize("lb", [-0.05, -5.0])
def test_pi_affine_split_composes(cuts, lb):
    rng = np.random.default_rng(77)
    c = rand_case(100, 2, 8, V=6, rng=rng, lb=lb, init=True)
    s = 0.4
    o_ref, S_ref = oracle.fwd(c["q"], c["k"], c["v"], c["la"], c["beta"], s, c["S0"])
    S = c["S0"][0].copy()                                   # [H, V, K]
    o = np.zeros_like(o_ref)
    eye = np.broadcast_to(np.eye(8), (1, 2, 8, 8)).copy()
    for a, b in zip(cuts[:-1], cuts[1:]):
        if a == b:
            continue
        sl = slice(a, b)
        oX, X = oracle.fwd(c["q"][sl], c["k"][sl], c["v"][sl], c["la"][sl], c["beta"][sl], s)
        y, M = oracle.fwd(c["q"][sl], c["k"][sl], np.zeros((b - a, 2, 8)), c["la"][sl],
                          c["beta"][sl], s, eye)
        o[sl] = oX + np.einsum("hvk,thk->thv", S, y)
        S = np.einsum("hvk,hkj->hvj", S, M[0]) + X[0]
    assert rel(o, o_ref) < 1e-12
    assert rel(S, S_ref[0]) < 1e-12
    # and the split is not vacuous: the handed-over state changes the outputs
    if lb == -0.05:
        o_zero, _ = oracle.fwd(c["q"][cuts[-2]:], c["k"][cuts[-2]:], c["v"][cuts[-2]:],
                               c["la"][cuts[-2]:], c["beta"][cuts[-2]:], s)
        assert rel(o_zero, o_ref[cuts[-2]:]) > 1e-3
