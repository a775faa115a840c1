"""GPU parity of kda_fwd_host, the host-buffer entry point of the C ABI
(libkda pipelines the copies and the passes itself), against the fp64 oracle
and against the device-buffer entry points on the same inputs."""
import pytest
import torch

import chunked_gated_delta_11_gb300 as kda
from chunked_gated_delta_11_gb300 import synth
from kda_testlib import assert_close, f64, oracle_case

pytestmark = pytest.mark.gpu


def host(inp, pin=True):
    out = dict(inp)
    for key in ("q", "k", "v", "g_raw", "beta_raw", "initial_state"):
        if inp[key] is not None:
            out[key] = inp[key].pin_memory() if pin else inp[key].clone()
    return out


def call_host(h, **kw):
    out, fs = kda.kda_forward_host(h["q"], h["k"], h["v"], h["g_raw"], h["beta_raw"], h["scale"],
                                   h["lower_bound"], h["initial_state"], h["cu_seqlens"],
                                   N=h["N"], **kw)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == 0
    return out, fs


@pytest.mark.parametrize("schedule", ["fused", "auto", "split", "decode", "segmented"])
def test_host_bf16_states_per_head_gate(schedule):
    inp = synth.make_inputs(0, 2, lengths=[90, 0, 33, 200, 17], seed=101, init_std=0.02)
    inp["initial_state"] = inp["initial_state"].to(torch.bfloat16)
    gh = inp["g_raw"][:, :, 0].contiguous()
    inp["g_raw"] = gh
    out, fs = call_host(host(inp), schedule=schedule, groups=3)
    assert fs.dtype == torch.bfloat16
    ref = dict(inp, initial_state=inp["initial_state"].float(),
               g_raw=gh[:, :, None].expand(-1, -1, 128).contiguous())
    ro, rs = oracle_case(ref)
    assert_close(f64(out), ro, f"{schedule} host out (bf16 states, per-head gate)")
    assert_close(f64(fs), rs, f"{schedule} host final_state (bf16 states, per-head gate)")


def test_host_pageable_equals_pinned_and_device():
    inp = synth.make_inputs(4 * 300, 2, 4, seed=102, init_std=0.02)
    o1, s1 = call_host(host(inp, pin=True), groups=2)
    o2, s2 = call_host(host(inp, pin=False), groups=2)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    od, sd = kda.kda_fwd_fused(d["q"], d["k"], d["v"], d["g_raw"], d["beta_raw"], d["scale"],
                               d["lower_bound"], d["initial_state"], None, N=4)
    assert torch.equal(o1, od.cpu()) and torch.equal(s1, sd.cpu())


def test_host_caller_workspace_and_back_to_back_calls():
    # the library's cached streams and events serve consecutive calls
    a = host(synth.make_inputs(0, 3, lengths=[50, 300, 7], seed=103, init_std=0.02))
    b = host(synth.make_inputs(2 * 500, 3, 2, seed=104))
    nbytes = max(kda.kda_fwd_host_workspace_size(x["T_total"], 3, x["N"], x["cu_seqlens"], groups=4)
                 for x in (a, b))
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    ra = call_host(a, groups=4, workspace=ws)
    rb = call_host(b, groups=4, workspace=ws)
    for x, (out, fs) in ((a, ra), (b, rb)):
        ro, rs = oracle_case(x)
        assert_close(f64(out), ro, "back-to-back host out")
        assert_close(f64(fs), rs, "back-to-back host final_state")


def test_host_no_tokens_returns_initial_state():
    inp = synth.make_inputs(0, 2, lengths=[0, 0, 0], seed=105, init_std=0.02)
    out, fs = call_host(host(inp), groups=2)
    assert torch.equal(fs, inp["initial_state"])
