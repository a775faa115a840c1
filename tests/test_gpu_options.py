"""GPU parity of kda_forward's options through the C ABI, on every schedule:
bf16 initial / final states and one gate per token and head (the Gated
DeltaNet case, alpha a scalar per token)."""
import pytest
import torch

import chunked_gated_delta_11_gb300 as kda
from chunked_gated_delta_11_gb300 import synth
from kda_testlib import assert_close, f64, oracle_case

pytestmark = pytest.mark.gpu

SCHEDULES = ["fused", "split", "decode", "segmented", "auto"]


def to_dev(inp):
    out = dict(inp)
    for key in ("q", "k", "v", "g_raw", "beta_raw", "initial_state", "cu_seqlens"):
        if inp[key] is not None:
            out[key] = inp[key].cuda()
    return out


def forward(inp, schedule, **kw):
    out, fs = kda.kda_forward(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"],
                              inp["scale"], inp["lower_bound"], inp["initial_state"],
                              inp["cu_seqlens"], N=inp["N"], schedule=schedule, **kw)
    assert kda.kda_device_status() == 0
    return out, fs


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_bf16_states(schedule):
    inp = to_dev(synth.make_inputs(0, 2, lengths=[40, 1, 0, 77], seed=41, init_std=0.02))
    inp["initial_state"] = inp["initial_state"].to(torch.bfloat16)
    out, fs = forward(inp, schedule)
    assert fs.dtype == torch.bfloat16
    ref = dict(inp, initial_state=inp["initial_state"].float())   # the same bf16 values
    ro, rs = oracle_case(ref)
    assert_close(f64(out), ro, f"{schedule} out (bf16 states)")
    assert_close(f64(fs), rs, f"{schedule} final_state (bf16 states)")


@pytest.mark.parametrize("schedule", SCHEDULES)
def test_per_head_gate(schedule):
    inp = to_dev(synth.make_inputs(0, 3, lengths=[64, 19, 0, 50], seed=42, init_std=0.02))
    gh = inp["g_raw"][:, :, 0].contiguous()                    # one gate per token and head
    inp_h = dict(inp, g_raw=gh)
    out, fs = forward(inp_h, schedule)
    ref = dict(inp, g_raw=gh[:, :, None].expand(-1, -1, 128).contiguous())
    ro, rs = oracle_case(ref)
    assert_close(f64(out), ro, f"{schedule} out (per-head gate)")
    assert_close(f64(fs), rs, f"{schedule} final_state (per-head gate)")
    # and the per-channel path on the broadcast gate gives the same result
    ob, sb = forward(ref, schedule)
    assert_close(f64(out), f64(ob), f"{schedule} per-head vs broadcast out")
    assert_close(f64(fs), f64(sb), f"{schedule} per-head vs broadcast state")


def test_forward_split_with_workspace_and_fp32_states_matches_kda_fwd():
    inp = synth.workload_inputs("h16", device="cuda")
    ws = torch.empty(kda.kda_workspace_size(inp["T_total"], inp["H"], inp["N"]),
                     dtype=torch.uint8, device="cuda")
    o1, s1 = forward(inp, "split", workspace=ws)
    o2, s2 = kda.kda_fwd(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"],
                         inp["scale"], inp["lower_bound"], inp["initial_state"], None, N=1)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


@pytest.mark.parametrize("lengths,H", [
    ([1] * 48, 2),          # serving step: decode
    ([8192], 2),            # one long sequence, few units: segmented
    ([64] * 80, 4),         # many units: fused
])
def test_auto_schedule(lengths, H):
    inp = to_dev(synth.make_inputs(0, H, lengths=lengths, seed=81, init_std=0.02))
    out, fs = forward(inp, "auto")
    ro, rs = oracle_case(inp)
    assert_close(f64(out), ro, f"auto out {len(lengths)} x {lengths[0]}")
    assert_close(f64(fs), rs, f"auto final_state {len(lengths)} x {lengths[0]}")


@pytest.mark.parametrize("name,units", [
    ("fk96", [(0, 0), (0, 95)]),
    ("fk64", [(0, 7)]),
    ("fk96p", [(5, 40)]),
    ("fk64p", [(7, 63)]),
])
def test_auto_schedule_on_benchmark_row_shapes(name, units):
    # FlashKDA's benchmark row shapes: the automatic choice (segmented for the
    # single sequences, fused for the packed ones) against the oracle
    from kda_testlib import compare_units
    inp = synth.workload_inputs(name, device="cuda")
    out, fs = forward(inp, "auto")
    compare_units(inp, out, fs, units)
