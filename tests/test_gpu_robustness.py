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
