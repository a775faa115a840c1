"""GPU parity of libkda against the fp64 oracle, through the C ABI.

Order: tensor-core convention self-test, chunk-kernel records against the
oracle's chunk factors, then the whole forward pass on every workload (full
comparison where the oracle is fast, sampled (sequence, head) units at full
size otherwise), edge cases and properties."""
import numpy as np
import pytest
import torch

import oracle
import chunked_gated_delta_11_gb300 as kda
from chunked_gated_delta_11_gb300 import synth
from kda_testlib import assert_close, compare_units, f64, oracle_case

pytestmark = pytest.mark.gpu



@pytest.fixture(scope="module", autouse=True)
def _built():
    kda.build.build()
    kda.load()
    yield
    assert kda.kda_device_status() == 0


PATHS = ["split", "fused"]  # kda_fwd (K1 + K2) and kda_fwd_fused (one kernel)


def run(inp, path="split", **kw):
    fn = kda.kda_fwd if path == "split" else kda.kda_fwd_fused
    out, fs = fn(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"], inp["scale"],
                 inp["lower_bound"], inp["initial_state"], inp["cu_seqlens"], N=inp["N"], **kw)
    assert kda.kda_device_status() == 0
    return out, fs


def to_dev(inp):
    out = dict(inp)
    for key in ("q", "k", "v", "g_raw", "beta_raw", "initial_state", "cu_seqlens"):
        if inp[key] is not None:
            out[key] = inp[key].cuda()
    return out


# ---------------------------------------------------------------------------
# tcgen05 operand conventions (values exact in tf32 / bf16 / fp32)
# ---------------------------------------------------------------------------
def _selftest_expected():
    m = np.arange(128)[:, None]
    k = np.arange(128)[None, :]
    A1 = ((m * 3 + k * 5) % 11 - 5) * 0.25
    n = np.arange(32)[:, None]
    B1 = ((n * 7 + k * 3) % 13 - 6) * 0.125
    j = np.arange(16)[None, :]
    A2 = ((m + 2 * j) % 7 - 3) * 0.5
    r = np.arange(144)[:, None]
    B2 = ((r * 5 + j * 11) % 9 - 4) * 0.25
    D0 = (m - np.arange(144)[None, :]) * 0.0625
    return A1 @ B1.T, D0 + A2 @ B2.T


def test_tcgen05_operand_conventions():
    out1, out2, status = kda.kda_selftest_tcgen05()
    assert status == 0
    e1, e2 = _selftest_expected()
    np.testing.assert_array_equal(out1.cpu().numpy(), e1.astype(np.float32))
    np.testing.assert_array_equal(out2.cpu().numpy(), e2.astype(np.float32))


# ---------------------------------------------------------------------------
# K1 records against the oracle's chunk factors
# ---------------------------------------------------------------------------
def _b1_offset(n, d):
    return (d >> 6) * 4096 + n * 128 + ((((d & 63) >> 3) ^ (n & 7)) << 4) + ((d & 7) << 1)


def _ka_offset(r, j):
    return 8192 + (j >> 3) * 4608 + r * 32 + (((((j & 7) >> 2) ^ (r >> 2)) & 1) << 4) + ((j & 3) << 2)


def decode_record(rec):
    """Record bytes -> fields (layout: [Qdec ; W'] bf16, [Kend' ; Aqk'] fp32, U', dlast)."""
    rec = np.asarray(rec, dtype=np.uint8)
    nn, dd = np.meshgrid(np.arange(32), np.arange(128), indexing="ij")
    b1 = (rec.view(np.uint16)[_b1_offset(nn, dd) // 2].astype(np.uint32) << 16).view(np.float32)
    jj, rr = np.meshgrid(np.arange(16), np.arange(144), indexing="ij")
    ka = rec.view(np.float32)[_ka_offset(rr, jj) // 4]          # [j][r]
    cc, ii_ = np.meshgrid(np.arange(128), np.arange(16), indexing="ij")
    swz = (((cc >> 1) & 1) << 1) | ((cc >> 2) & 1)
    uoff = 17408 + cc * 64 + (((ii_ >> 2) ^ swz) << 4) + ((ii_ & 3) << 2)
    U = rec.view(np.float32)[uoff // 4].T
    dl = rec[25600:26112].view(np.float32)
    rq = rec[26112:26176].view(np.float32)
    return {"Qdec": b1[:16].astype(np.float64), "W": b1[16:].astype(np.float64),
            "Kend": ka[:, :128].astype(np.float64), "Aqk": ka[:, 128:].T.astype(np.float64),
            "U": U, "dlast": dl, "rq": rq}


def record_convention(f, rk, rq):
    """The oracle's chunk factors in the record's convention: with D = diag(rk),
    rk_j = 1 / |k_j|, and rq_i = scale / |q_i|, the record holds W' = D W,
    U' = D U, Kend' = D^-1 Kend, Qdec' = diag(rq)^-1 Qdec and
    Aqk' = diag(rq)^-1 Aqk D^-1, plus rq; the recurrence's products, with each
    output row scaled by rq_i, equal the unscaled ones."""
    return {"Qdec": f["Qdec"] / rq[:, None], "W": rk[:, None] * f["W"],
            "U": rk[:, None] * f["U"], "Kend": f["Kend"] / rk[:, None],
            "Aqk": f["Aqk"] / (rq[:, None] * rk[None, :]), "dlast": f["dlast"], "rq": rq}


@pytest.mark.parametrize("lengths,H", [([64], 1), ([45], 2), ([7, 0, 33, 16], 2)])
def test_chunk_records_match_oracle_factors(lengths, H):
    inp = to_dev(synth.make_inputs(0, H, lengths=lengths, seed=11, init_std=0.02))
    T, N = inp["T_total"], inp["N"]
    ws = torch.zeros(kda.kda_workspace_size(T, H, N), dtype=torch.uint8, device="cuda")
    kda.kda_chunk_prep(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"], inp["scale"],
                       inp["lower_bound"], ws, inp["cu_seqlens"], N=N)
    torch.cuda.synchronize()
    wsh = ws.cpu().numpy()
    qh, kh, la, beta = oracle.prepare(f64(inp["q"]), f64(inp["k"]), f64(inp["g_raw"]),
                                      f64(inp["beta_raw"]), inp["lower_bound"])
    cu = inp["cu_seqlens"].cpu().numpy()
    f = oracle.chunk_factors(qh, kh, f64(inp["v"]), la, beta, inp["scale"], cu_seqlens=cu)
    kraw, qraw = f64(inp["k"]), f64(inp["q"])
    got = {k_: [] for k_ in f if k_ != "Akk"}
    got["rq"] = []
    ref = {k_: [] for k_ in got}
    chunk = 0
    for n in range(N):
        bos, eos = int(cu[n]), int(cu[n + 1])
        for c in range((eos - bos + 15) // 16):
            for h in range(H):
                slot = bos // 16 + n + c
                r = decode_record(wsh[(slot * H + h) * kda.REC_BYTES:][:kda.REC_BYTES])
                kc = np.zeros((16, 128))
                qc = np.zeros((16, 128))
                t0 = bos + 16 * c
                kc[:min(16, eos - t0)] = kraw[t0:min(t0 + 16, eos), h]
                qc[:min(16, eos - t0)] = qraw[t0:min(t0 + 16, eos), h]
                rk = 1.0 / np.sqrt((kc * kc).sum(-1) + oracle.DEFAULT_EPS)
                rq = inp["scale"] / np.sqrt((qc * qc).sum(-1) + oracle.DEFAULT_EPS)
                fr = record_convention({k_: f[k_][chunk, h] for k_ in got if k_ != "rq"}, rk, rq)
                for key in got:
                    got[key].append(r[key].reshape(-1))
                    ref[key].append(fr[key].reshape(-1))
            chunk += 1
    for key in got:
        g_ = np.concatenate(got[key])
        r_ = np.concatenate(ref[key])
        mx = np.abs(g_ - r_).max() / np.abs(r_).max()
        fro = np.linalg.norm(g_ - r_) / np.linalg.norm(r_)
        tmax, tfro = RECORD_TOL.get(key, (2e-3, 1e-3))
        assert mx < tmax and fro < tfro, f"{key}: max_rel {mx:.2e} fro {fro:.2e}"


# Qdec and W are stored as bf16 (relative rounding up to 2^-9); W and Aqk also
# come from products with bf16 operands and fp32 accumulation, the chunk-kernel
# precision of FlashKDA ("FlashKDA v1: A Deep Dive", sec. 3), each product term
# carrying up to 2^-8 relative rounding.  These are held to the output bounds
# (1e-2 of the largest entry, 5e-3 Frobenius).  U (split bf16 operands), Kend
# and dlast (fp32) stay at 2e-3 / 1e-3.
RECORD_TOL = {"W": (1e-2, 5e-3), "Aqk": (1e-2, 5e-3), "Qdec": (1e-2, 5e-3)}


# ---------------------------------------------------------------------------
# whole forward pass
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["tiny", "h16"])
@pytest.mark.parametrize("path", PATHS)
def test_fwd_small_workloads_full(name, path):
    inp = to_dev(synth.workload_inputs(name))
    out, fs = run(inp, path)
    ro, rs = oracle_case(inp)
    assert_close(f64(out), ro, f"{name} out")
    assert_close(f64(fs), rs, f"{name} final_state")


@pytest.mark.parametrize("lengths,H,init", [
    ([1], 1, False), ([15], 1, True), ([16], 3, False), ([17], 2, True), ([33], 1, False),
    ([0, 5, 0, 17, 32, 1], 2, True), ([300, 1, 47], 4, True),
])
@pytest.mark.parametrize("path", PATHS)
def test_fwd_edge_cases(lengths, H, init, path):
    inp = to_dev(synth.make_inputs(0, H, lengths=lengths, seed=sum(lengths) + H,
                                   init_std=0.02 if init else None))
    out, fs = run(inp, path)
    ro, rs = oracle_case(inp)
    if inp["T_total"]:
        assert_close(f64(out), ro, "out")
    assert_close(f64(fs), rs, "final_state")


@pytest.mark.parametrize("path", PATHS)
def test_fwd_equal_batches_without_cu_seqlens(path):
    inp = to_dev(synth.make_inputs(3 * 80, 2, 3, seed=5, init_std=0.02))
    out, fs = run(inp, path)
    ro, rs = oracle_case(inp)
    assert_close(f64(out), ro, "out")
    assert_close(f64(fs), rs, "final_state")


@pytest.mark.parametrize("path", PATHS)
def test_fwd_empty_input_returns_initial_state(path):
    inp = to_dev(synth.make_inputs(0, 2, lengths=[0, 0], seed=1, init_std=0.02))
    out, fs = run(inp, path)
    assert torch.equal(fs, inp["initial_state"])


@pytest.mark.parametrize("name,units", [
    ("b8", [(0, 0), (3, 17), (7, 31)]),
    ("long", [(0, 0), (0, 31)]),
    ("slow", [(0, 5)]),
    ("fk96", [(0, 0), (0, 95)]),      # the shapes of FlashKDA's benchmark rows
    ("fk64", [(0, 63)]),
    ("fk96p", [(0, 0), (7, 95)]),
    ("fk64p", [(3, 10)]),
])
@pytest.mark.parametrize("path", PATHS)
def test_fwd_full_size_sampled_units(name, units, path):
    inp = synth.workload_inputs(name, device="cuda")
    out, fs = run(inp, path)
    compare_units(inp, out, fs, units)


@pytest.mark.parametrize("path", PATHS)
def test_fwd_varlen_full_size_sampled_units(path):
    inp = synth.workload_inputs("varlen", device="cuda")
    out, fs = run(inp, path)
    cu = inp["cu_seqlens"].cpu().numpy()
    lens = np.diff(cu)
    longest, shortest = int(np.argmax(lens)), int(np.argmin(lens))
    compare_units(inp, out, fs, [(longest, 3), (shortest, 30), (1, 0)])


# ---------------------------------------------------------------------------
# properties
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("path", PATHS)
def test_deterministic(path):
    inp = to_dev(synth.workload_inputs("h16"))
    o1, s1 = run(inp, path)
    o2, s2 = run(inp, path)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


@pytest.mark.parametrize("path", PATHS)
def test_streaming_split_chains_state(path):
    inp = to_dev(synth.workload_inputs("h16"))
    o, s = run(inp, path)
    for t1, exact in ((2048, True), (1000, False)):
        a = {k: inp[k] for k in inp}
        b = {k: inp[k] for k in inp}
        for key in ("q", "k", "v", "g_raw", "beta_raw"):
            a[key] = inp[key][:t1].contiguous()
            b[key] = inp[key][t1:].contiguous()
        a["T_total"], b["T_total"] = t1, inp["T_total"] - t1
        oa, sa = run(a, path)
        b["initial_state"] = sa
        ob, sb = run(b, path)
        oc = torch.cat([oa, ob])
        if exact:  # chunk-aligned split: the same chunks, bit for bit
            assert torch.equal(oc, o) and torch.equal(sb, s)
        else:
            assert_close(f64(oc), f64(o), "split out")
            assert_close(f64(sb), f64(s), "split state")


@pytest.mark.parametrize("path", PATHS)
def test_varlen_packing_equals_separate_calls(path):
    lengths = [37, 16, 100]
    inp = to_dev(synth.make_inputs(0, 2, lengths=lengths, seed=3, init_std=0.02))
    o, s = run(inp, path)
    cu = inp["cu_seqlens"].cpu().tolist()
    for n in range(3):
        sl = slice(cu[n], cu[n + 1])
        one = {k: inp[k] for k in inp}
        for key in ("q", "k", "v", "g_raw", "beta_raw"):
            one[key] = inp[key][sl].contiguous()
        one["initial_state"] = inp["initial_state"][n:n + 1].contiguous()
        one["cu_seqlens"], one["N"], one["T_total"] = None, 1, lengths[n]
        on, sn = run(one, path)
        assert torch.equal(on, o[sl]) and torch.equal(sn[0], s[n])


@pytest.mark.parametrize("path", PATHS)
def test_beta_zero_is_pure_decay(path):
    # slow decay (g_raw ~ N(-4, 1)) so that the decayed state stays in fp32 range
    inp = to_dev(synth.make_inputs(64, 2, 1, seed=9, init_std=0.02, g_mean=-4.0))
    inp["beta_raw"] = torch.full_like(inp["beta_raw"], float("-inf"))
    out, fs = run(inp, path)
    ro, rs = oracle_case(inp)
    assert_close(f64(out), ro, "out")
    assert_close(f64(fs), rs, "final_state")


def test_host_buffer_entry_point():
    inp = synth.workload_inputs("tiny")
    out, fs = kda.kda_forward_host(inp["q"].pin_memory(), inp["k"].pin_memory(),
                                   inp["v"].pin_memory(), inp["g_raw"].pin_memory(),
                                   inp["beta_raw"].pin_memory(), inp["scale"],
                                   inp["lower_bound"])
    torch.cuda.synchronize()
    ro, rs = oracle_case(inp)
    assert_close(f64(out), ro, "out")
    assert_close(f64(fs), rs, "final_state")


@pytest.mark.parametrize("path", PATHS)
def test_host_buffer_entry_point_grouped(path):
    # packed sequences (one empty), initial states, three groups of sequences
    inp = synth.make_inputs(0, 2, lengths=[33, 0, 100, 17, 64, 5], seed=21, init_std=0.02)
    host = {key: (inp[key].pin_memory() if inp[key] is not None else None)
            for key in ("q", "k", "v", "g_raw", "beta_raw", "initial_state")}
    out, fs = kda.kda_forward_host(host["q"], host["k"], host["v"], host["g_raw"],
                                   host["beta_raw"], inp["scale"], inp["lower_bound"],
                                   host["initial_state"], inp["cu_seqlens"], groups=3,
                                   schedule=path)
    torch.cuda.synchronize()
    od, sd = run(to_dev(inp), path)
    assert torch.equal(out, od.cpu()) and torch.equal(fs, sd.cpu())
    ro, rs = oracle_case(inp)
    assert_close(f64(out), ro, "grouped host out")
    assert_close(f64(fs), rs, "grouped host final_state")


def test_fused_agrees_with_split_on_b8():
    inp = synth.workload_inputs("b8", device="cuda")
    o1, s1 = run(inp, "split")
    o2, s2 = run(inp, "fused")
    assert_close(f64(o2), f64(o1), "fused vs split out")
    assert_close(f64(s2), f64(s1), "fused vs split state")
    print(f"[parity] fused vs split bit-identical: out {torch.equal(o1, o2)} state {torch.equal(s1, s2)}")


# Zero query / key rows: the key norm factor rk = 1 / sqrt(0 + eps) is at its
# largest (1e3), which the record's rescaled factors (W' = D W, U' = D U,
# Kend' = D^-1 Kend) must carry without loss; a zero key row contributes
# nothing to the state and a zero query row reads nothing.
@pytest.mark.parametrize("path", PATHS + ["decode"])
def test_zero_query_and_key_rows(path):
    inp = synth.make_inputs(0, 2, lengths=[40, 19], seed=21, init_std=0.02)
    for t_, h_ in ((5, 0), (20, 1), (39, 0), (41, 1), (58, 0)):
        inp["k"][t_, h_] = 0
    for t_, h_ in ((7, 1), (20, 0), (45, 1)):
        inp["q"][t_, h_] = 0
    inp = to_dev(inp)
    if path == "decode":
        out, fs = kda.kda_decode(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"],
                                 inp["scale"], inp["lower_bound"], inp["initial_state"],
                                 inp["cu_seqlens"], N=inp["N"])
        assert kda.kda_device_status() == 0
    else:
        out, fs = run(inp, path)
    ro, rs = oracle_case(inp)
    assert_close(f64(out), ro, "out")
    assert_close(f64(fs), rs, "final_state")


@pytest.mark.parametrize("schedule", ["fused", "split", "decode", "segmented"])
def test_host_buffer_entry_point_time_slices(schedule):
    # equal sequences with initial states: the host-buffer entry point cuts
    # them in time into chunk-aligned slices chained through the state
    inp = synth.make_inputs(3 * 500, 2, 3, seed=12, init_std=0.02)
    pin = {key: (inp[key].pin_memory() if inp[key] is not None else None)
           for key in ("q", "k", "v", "g_raw", "beta_raw", "initial_state")}
    out, fs = kda.kda_forward_host(pin["q"], pin["k"], pin["v"], pin["g_raw"], pin["beta_raw"],
                                   inp["scale"], inp["lower_bound"], pin["initial_state"],
                                   N=3, schedule=schedule, groups=5)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == 0
    ro, rs = oracle_case(inp)
    assert_close(f64(out), ro, f"{schedule} host slices out")
    assert_close(f64(fs), rs, f"{schedule} host slices final_state")


@pytest.mark.parametrize("kernel", [0, 1])
def test_profile_phases_diagnostic(kernel):
    # the timed copies give kda_fwd's results and stamps in phase order
    from chunked_gated_delta_11_gb300 import phases
    inp = to_dev(synth.make_inputs(2 * 640, 2, 2, seed=31))
    st = phases.run(kernel, inp, 40)
    o_ref, s_ref = run(inp, "split")
    assert kda.kda_device_status() == 0
    for c in range(40 - 1):
        assert all(st[c, k] <= st[c, k + 1] for k in range(6)), (c, st[c])
        assert st[c, 0] < st[c + 1, 0]
    table = phases.table(st)
    assert table["period"][0] > table["MMA1"][0] > 0


@pytest.mark.parametrize("path", PATHS)
def test_concurrent_calls_on_two_streams(path):
    # Two different batches, each launched several times on its own stream
    # with its own outputs, so that the calls overlap on the GPU: the library
    # holds no state between calls that concurrent calls could share (the
    # bench's two-stream throughput runs this way).
    a = to_dev(synth.make_inputs(0, 3, lengths=[200, 77, 330], seed=71, init_std=0.02))
    b = to_dev(synth.make_inputs(0, 2, lengths=[513, 9], seed=72, init_std=0.02))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    fn = kda.kda_fwd if path == "split" else kda.kda_fwd_fused
    results = []
    torch.cuda.synchronize()
    for rep in range(3):
        for inp, st in zip((a, b), streams):
            out, fs = fn(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"], inp["scale"],
                         inp["lower_bound"], inp["initial_state"], inp["cu_seqlens"], N=inp["N"],
                         stream=st)
            if rep == 2:
                results.append((inp, out, fs))
    torch.cuda.synchronize()
    assert kda.kda_device_status() == 0
    for inp, out, fs in results:
        ro, rs = oracle_case(inp)
        assert_close(f64(out), ro, f"{path} two streams out")
        assert_close(f64(fs), rs, f"{path} two streams final_state")


GRAPH_CALLS = {
    "split": kda.kda_fwd,
    "fused": kda.kda_fwd_fused,
    "decode": kda.kda_decode,
    # four launches chained by programmatic dependent launch, workspace
    # allocated stream-ordered
    "segmented": lambda *a, **kw: kda.kda_fwd_segmented(*a, segments=3, **kw),
}


@pytest.mark.parametrize("path", list(GRAPH_CALLS))
def test_cuda_graph_capture_and_replay(path):
    # The calls launch with the programmatic-dependent-launch attribute and
    # (without a workspace) allocate stream-ordered; they must capture into a
    # CUDA graph, and each replay must give the oracle's result.
    inp = to_dev(synth.make_inputs(0, 2, lengths=[150, 64, 300], seed=81, init_std=0.02))
    fn = GRAPH_CALLS[path]
    out = torch.empty_like(inp["q"])
    fs = torch.empty((inp["N"], 2, 128, 128), dtype=torch.float32, device="cuda")
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(st):  # one eager call first (library load, attributes)
        fn(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"], inp["scale"],
           inp["lower_bound"], inp["initial_state"], inp["cu_seqlens"], N=inp["N"], out=out,
           final_state=fs, stream=st)
    st.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        fn(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"], inp["scale"],
           inp["lower_bound"], inp["initial_state"], inp["cu_seqlens"], N=inp["N"], out=out,
           final_state=fs, stream=st)
    ro, rs = oracle_case(inp)
    for _ in range(2):
        out.zero_()
        fs.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert kda.kda_device_status() == 0
        assert_close(f64(out), ro, f"{path} graph replay out")
        assert_close(f64(fs), rs, f"{path} graph replay final_state")
