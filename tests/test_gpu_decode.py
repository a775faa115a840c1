"""GPU parity of the recurrent (decode) schedule, kda_decode, through the C ABI:
against the fp64 oracle's token-by-token recurrence, against the chunkwise
kernels on the same inputs, and with the state updated in place."""
import pytest
import torch

import chunked_gated_delta_11_gb300 as kda
from chunked_gated_delta_11_gb300 import synth
from kda_testlib import assert_close, compare_units, f64, oracle_case

pytestmark = pytest.mark.gpu


def to_dev(inp):
    out = dict(inp)
    for key in ("q", "k", "v", "g_raw", "beta_raw", "initial_state", "cu_seqlens"):
        if inp[key] is not None:
            out[key] = inp[key].cuda()
    return out


def decode(inp, **kw):
    out, fs = kda.kda_decode(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"],
                             inp["scale"], inp["lower_bound"], inp["initial_state"],
                             inp["cu_seqlens"], N=inp["N"], **kw)
    assert kda.kda_device_status() == 0
    return out, fs


@pytest.mark.parametrize("lengths,H,init", [
    ([64], 1, False),                     # the 4-chunk single-head case
    ([1, 3, 0, 7, 16, 33], 2, True),      # packed, one empty sequence, ragged
    ([1] * 40, 3, True),                  # one token per sequence (serving step)
])
def test_decode_matches_oracle(lengths, H, init):
    inp = to_dev(synth.make_inputs(0, H, lengths=lengths, seed=31,
                                   init_std=0.02 if init else None))
    out, fs = decode(inp)
    ro, rs = oracle_case(inp)
    assert_close(f64(out), ro, "decode out")
    assert_close(f64(fs), rs, "decode final_state")


def test_decode_state_in_place_and_chained():
    # two decode calls of 5 and 3 tokens with the state updated in place equal
    # one call over the 8 tokens (the oracle's streaming split, pin P-h)
    inp = synth.make_inputs(8 * 16, 4, 16, seed=32, init_std=0.02)
    d = to_dev(inp)
    T = inp["T_total"] // 16
    idx_a = torch.cat([torch.arange(n * T, n * T + 5) for n in range(16)])
    idx_b = torch.cat([torch.arange(n * T + 5, n * T + T) for n in range(16)])
    state = d["initial_state"].clone()
    outs = []
    for idx in (idx_a, idx_b):
        part = {key: d[key][idx.cuda()].contiguous() for key in ("q", "k", "v", "g_raw", "beta_raw")}
        part.update(scale=inp["scale"], lower_bound=inp["lower_bound"], initial_state=state,
                    cu_seqlens=None, N=16)
        o, s = decode(part, final_state=state)   # in place
        assert s.data_ptr() == state.data_ptr()
        outs.append(o)
    full, full_s = decode(d)
    got = torch.empty_like(full)
    got[idx_a.cuda()] = outs[0]
    got[idx_b.cuda()] = outs[1]
    assert_close(f64(got), f64(full), "chained decode out")
    assert_close(f64(state), f64(full_s), "chained decode state")
    ro, rs = oracle_case(d)
    assert_close(f64(full), ro, "decode out")
    assert_close(f64(full_s), rs, "decode state")


def test_decode_agrees_with_fused_on_h16():
    inp = synth.workload_inputs("h16", device="cuda")
    od, sd = decode(inp)
    of, sf = kda.kda_fwd_fused(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"],
                               inp["scale"], inp["lower_bound"], inp["initial_state"], None, N=1)
    assert_close(f64(od), f64(of), "decode vs fused out")
    assert_close(f64(sd), f64(sf), "decode vs fused state")


def test_decode_serving_step_full_size():
    # the bench's decode workload (256 sequences x 1 token, H = 32), sampled units
    inp = synth.workload_inputs("decode", device="cuda")
    out, fs = decode(inp)
    compare_units(inp, out, fs, [(0, 0), (17, 5), (128, 31), (255, 12)])
