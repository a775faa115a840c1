"""Device-side robustness through the C ABI: the cu_seqlens check latches its
error in the device error word, and no schedule writes outside `out` or
`final_state` (guard bands of a sentinel pattern around both, on ragged packed
inputs, checked after the call)."""
import pytest
import torch

import chunked_gated_delta_11_gb300 as kda
from chunked_gated_delta_11_gb300 import synth
from kda_testlib import assert_close, f64, oracle_case

pytestmark = pytest.mark.gpu


def to_dev(inp):
    out = dict(inp)
    for key in ("q", "k", "v", "g_raw", "beta_raw", "initial_state", "cu_seqlens"):
        if inp[key] is not None:
            out[key] = inp[key].cuda()
    return out


@pytest.mark.parametrize("cu,T,ok", [
    ([0, 5, 5, 17], 17, True),
    ([0], 0, True),                 # N = 0: rejected on the host before any launch
    ([1, 5, 17], 17, False),        # does not start at 0
    ([0, 9, 5, 17], 17, False),     # decreasing
    ([0, 5, 16], 17, False),        # does not end at T_total
])
def test_validate_cu_seqlens(cu, T, ok):
    assert kda.kda_device_status() == 0
    t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    if len(cu) == 1:
        with pytest.raises(kda.KdaError):
            kda.kda_validate_cu_seqlens(t, T)
        return
    kda.kda_validate_cu_seqlens(t, T)
    status = kda.kda_device_status()
    assert status == (0 if ok else 1)
    assert kda.kda_device_status() == 0  # the word was cleared


GUARD = 4096  # elements of sentinel on each side


def guarded(shape, dtype, fill):
    n = 1
    for s in shape:
        n *= s
    buf = torch.full((GUARD + n + GUARD,), fill, dtype=dtype, device="cuda")
    return buf, buf[GUARD:GUARD + n].view(shape)


@pytest.mark.parametrize("schedule", ["fused", "split", "decode", "segmented"])
def test_writes_stay_inside_outputs(schedule):
    inp = to_dev(synth.make_inputs(0, 2, lengths=[300, 1, 0, 47, 129], seed=71, init_std=0.02))
    T, H, N = inp["T_total"], 2, 5
    obuf, out = guarded((T, H, 128), torch.bfloat16, -7.0)
    sbuf, fs = guarded((N, H, 128, 128), torch.float32, -7.0)
    out.zero_()
    fs.zero_()
    kw = dict(N=N, out=out, final_state=fs)
    a = (inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"], inp["scale"],
         inp["lower_bound"], inp["initial_state"], inp["cu_seqlens"])
    if schedule == "fused":
        kda.kda_fwd_fused(*a, **kw)
    elif schedule == "split":
        kda.kda_fwd(*a, **kw)
    elif schedule == "decode":
        kda.kda_decode(*a, **kw)
    else:
        kda.kda_fwd_segmented(*a, segments=3, **kw)
    assert kda.kda_device_status() == 0
    for buf, n in ((obuf, out.numel()), (sbuf, fs.numel())):
        assert torch.all(buf[:GUARD] == -7.0) and torch.all(buf[GUARD + n:] == -7.0), schedule
    ro, rs = oracle_case(inp)
    assert_close(f64(out), ro, f"{schedule} out (guarded)")
    assert_close(f64(fs), rs, f"{schedule} final_state (guarded)")


def _random_cases(n, seed=2024):
    import random
    rng = random.Random(seed)
    special = [0, 1, 15, 16, 17, 31, 33, 64]
    cases = []
    for i in range(n):
        k = rng.randint(1, 6)
        lengths = [rng.choice(special) if rng.random() < 0.5 else rng.randint(1, 700)
                   for _ in range(k)]
        if sum(lengths) == 0:
            lengths[0] = 5
        cases.append((i, lengths, rng.randint(1, 3), rng.random() < 0.5, rng.randint(2, 6)))
    return cases


@pytest.mark.parametrize("case", _random_cases(8), ids=lambda c: f"case{c[0]}")
def test_random_packings_all_schedules(case):
    # seeded random packings (lengths around the chunk size, empty sequences,
    # long ones), head counts, with or without initial states, through every
    # schedule, each against the oracle
    i, lengths, H, init, pieces = case
    inp = to_dev(synth.make_inputs(0, H, lengths=lengths, seed=100 + i,
                                   init_std=0.02 if init else None))
    ro, rs = oracle_case(inp)
    a = (inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"], inp["scale"],
         inp["lower_bound"], inp["initial_state"], inp["cu_seqlens"])
    N = inp["N"]
    for name, run in (("fused", lambda: kda.kda_fwd_fused(*a, N=N)),
                      ("split", lambda: kda.kda_fwd(*a, N=N)),
                      ("decode", lambda: kda.kda_decode(*a, N=N)),
                      ("segmented", lambda: kda.kda_fwd_segmented(*a, N=N, segments=pieces))):
        out, fs = run()
        assert kda.kda_device_status() == 0, name
        assert_close(f64(out), ro, f"{name} out {lengths} H={H}")
        assert_close(f64(fs), rs, f"{name} final_state {lengths} H={H}")


@pytest.mark.parametrize("schedule", ["fused", "split", "decode", "segmented"])
def test_cuda_graph_capture_and_replay(schedule):
    # every schedule is capturable (asynchronous, no host synchronisation, no
    # allocation outside the stream-ordered kind) and replays to the same bits
    inp = to_dev(synth.make_inputs(0, 2, lengths=[300, 47, 129], seed=72, init_std=0.02))
    N = inp["N"]
    a = (inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"], inp["scale"],
         inp["lower_bound"], inp["initial_state"], inp["cu_seqlens"])
    out = torch.empty_like(inp["q"])
    fs = torch.empty((N, 2, 128, 128), dtype=torch.float32, device="cuda")
    call = {"fused": lambda s: kda.kda_fwd_fused(*a, N=N, out=out, final_state=fs, stream=s),
            "split": lambda s: kda.kda_fwd(*a, N=N, out=out, final_state=fs, stream=s),
            "decode": lambda s: kda.kda_decode(*a, N=N, out=out, final_state=fs, stream=s),
            "segmented": lambda s: kda.kda_fwd_segmented(*a, N=N, segments=3, out=out,
                                                         final_state=fs, stream=s)}[schedule]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call(side)                      # eager run (also warms the launchers up)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == 0
    o_ref, s_ref = out.clone(), fs.clone()
    out.zero_()
    fs.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        call(side)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert kda.kda_device_status() == 0
        assert torch.equal(out, o_ref) and torch.equal(fs, s_ref), schedule


def test_concurrent_streams_match_serial_calls():
    # the library keeps no per-call state: two passes on two streams at once
    # give the bits of the same passes run one after the other
    cases = [to_dev(synth.make_inputs(0, 2, lengths=L, seed=73 + i, init_std=0.02))
             for i, L in enumerate(([500, 33], [17, 260, 90]))]

    def run(inp, stream):
        return kda.kda_fwd_fused(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"],
                                 inp["scale"], inp["lower_bound"], inp["initial_state"],
                                 inp["cu_seqlens"], N=inp["N"], stream=stream)
    ref = [run(c, torch.cuda.current_stream()) for c in cases]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in cases]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    got = []
    for c, st in zip(cases, streams):
        with torch.cuda.stream(st):
            got.append(run(c, st))
    torch.cuda.synchronize()
    assert kda.kda_device_status() == 0
    for (o1, s1), (o2, s2) in zip(ref, got):
        assert torch.equal(o1, o2) and torch.equal(s1, s2)


@pytest.mark.parametrize("schedule", ["fused", "split", "decode"])
def test_no_final_state_requested(schedule):
    # final_state = NULL: the pass writes only `out`, which matches the oracle
    inp = to_dev(synth.make_inputs(0, 2, lengths=[200, 31], seed=74, init_std=0.02))
    a = (inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"], inp["scale"],
         inp["lower_bound"], inp["initial_state"], inp["cu_seqlens"])
    fn = {"fused": kda.kda_fwd_fused, "split": kda.kda_fwd, "decode": kda.kda_decode}[schedule]
    out, fs = fn(*a, N=inp["N"], output_final_state=False)
    assert fs is None
    assert kda.kda_device_status() == 0
    ro, _ = oracle_case(inp)
    assert_close(f64(out), ro, f"{schedule} out without a final state")


@pytest.mark.parametrize("schedule", ["fused", "split", "segmented"])
def test_state_updated_in_place(schedule):
    # final_state may be the initial_state buffer: each (sequence, head) reads
    # its initial state before it writes its final state
    inp = to_dev(synth.make_inputs(0, 2, lengths=[300, 70], seed=75, init_std=0.02))
    ro, rs = oracle_case(inp)
    state = inp["initial_state"].clone()
    a = (inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"], inp["scale"],
         inp["lower_bound"], state, inp["cu_seqlens"])
    kw = dict(N=inp["N"], final_state=state)
    if schedule == "fused":
        out, fs = kda.kda_fwd_fused(*a, **kw)
    elif schedule == "split":
        out, fs = kda.kda_fwd(*a, **kw)
    else:
        out, fs = kda.kda_fwd_segmented(*a, segments=3, **kw)
    assert kda.kda_device_status() == 0
    assert fs.data_ptr() == state.data_ptr()
    assert_close(f64(out), ro, f"{schedule} out (state in place)")
    assert_close(f64(state), rs, f"{schedule} final_state (in place)")


def test_bounded_wait_timeout_is_reported_and_recovers():
    # the failure-detection path of every device wait, made to run out on purpose:
    # a CTA waits on an mbarrier nothing arrives at, with a 1e5-cycle limit
    assert kda.kda_device_status() == 0
    kda.kda_selftest_timeout(100_000)
    assert kda.kda_device_status() == 5          # KDA_ERR_TIMEOUT, latched once
    assert kda.kda_device_status() == 0          # and cleared by the read
    # the context is intact: the next forward pass is correct
    inp = to_dev(synth.make_inputs(0, 2, lengths=[70, 33], seed=91, init_std=0.02))
    out, fs = kda.kda_fwd_fused(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"],
                                inp["scale"], inp["lower_bound"], inp["initial_state"],
                                inp["cu_seqlens"], N=inp["N"])
    assert kda.kda_device_status() == 0
    ro, rs = oracle_case(inp)
    assert_close(f64(out), ro, "out after a timeout")
    assert_close(f64(fs), rs, "final_state after a timeout")


def test_timeout_limit_is_checked_on_the_host():
    for bad in (0, -1, (1 << 31) + 1):
        with pytest.raises(kda.KdaError) as e:
            kda.kda_selftest_timeout(bad)
        assert e.value.status == 1
