"""GPU parity of the segmented forward pass (kda_fwd_segmented): every
sequence cut into pieces that run at the same time, joined by a scan of their
affine state maps.  Against the fp64 oracle's token-by-token recurrence (small
cases whole, full-size cases on sampled units) and against the one-piece fused
pass on the same inputs."""
import numpy as np
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


def segmented(inp, segments, **kw):
    out, fs = kda.kda_fwd_segmented(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"],
                                    inp["scale"], inp["lower_bound"], inp["initial_state"],
                                    inp["cu_seqlens"], N=inp["N"], segments=segments, **kw)
    assert kda.kda_device_status() == 0
    return out, fs


def fused(inp):
    out, fs = kda.kda_fwd_fused(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"],
                                inp["scale"], inp["lower_bound"], inp["initial_state"],
                                inp["cu_seqlens"], N=inp["N"])
    assert kda.kda_device_status() == 0
    return out, fs


@pytest.mark.parametrize("lengths,H,segments", [
    ([300, 47, 1, 0, 129], 2, 2),
    ([300, 47, 1, 0, 129], 2, 5),   # pieces of one chunk, a ragged tail, empty pieces
    ([17], 1, 5),                   # two chunks in five pieces
    ([1000], 3, 7),
])
@pytest.mark.parametrize("init", [False, True])
def test_segmented_matches_oracle(lengths, H, segments, init):
    inp = to_dev(synth.make_inputs(0, H, lengths=lengths, seed=51 + segments,
                                   init_std=0.02 if init else None))
    out, fs = segmented(inp, segments)
    ro, rs = oracle_case(inp)
    assert_close(f64(out), ro, f"segmented({segments}) out")
    assert_close(f64(fs), rs, f"segmented({segments}) final_state")


def test_segmented_equal_sequences_per_head_gate():
    # N equal sequences (no cu_seqlens), one gate per token and head
    inp = to_dev(synth.make_inputs(3 * 500, 2, 3, seed=57, init_std=0.02, g_mean=-3.0))
    gh = inp["g_raw"][:, :, 0].contiguous()
    out, fs = segmented(dict(inp, g_raw=gh), 4)
    ro, rs = oracle_case(dict(inp, g_raw=gh[:, :, None].expand(-1, -1, 128).contiguous()))
    assert_close(f64(out), ro, "segmented per-head gate out")
    assert_close(f64(fs), rs, "segmented per-head gate final_state")


def test_segmented_one_piece_is_the_fused_pass():
    inp = to_dev(synth.make_inputs(0, 2, lengths=[300, 47, 129], seed=58, init_std=0.02))
    o1, s1 = segmented(inp, 1)
    o2, s2 = fused(inp)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_segmented_slow_decay_against_oracle():
    # slow decay (alpha ~ 0.988): the pieces' transition products stay near the
    # identity, so every piece's output depends on the state handed over by
    # the scan, not only on its own tokens
    inp = to_dev(synth.make_inputs(8192, 4, 1, seed=59, init_std=0.02, g_mean=-6.0))
    ro, rs = oracle_case(inp)
    for segments in (3, 8):
        out, fs = segmented(inp, segments)
        assert_close(f64(out), ro, f"slow decay, {segments} pieces, out")
        assert_close(f64(fs), rs, f"slow decay, {segments} pieces, final_state")


def test_segmented_given_workspace_equals_allocated():
    inp = to_dev(synth.make_inputs(4096, 4, 1, seed=60, init_std=0.02))
    nbytes = kda.kda_segmented_workspace_size(4096, 4, 1, segments=4)
    assert nbytes > 0
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    o1, s1 = segmented(inp, 4, workspace=ws)
    o2, s2 = segmented(inp, 4)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_segmented_deterministic():
    inp = to_dev(synth.make_inputs(0, 2, lengths=[700, 33], seed=61, init_std=0.02))
    o1, s1 = segmented(inp, 3)
    o2, s2 = segmented(inp, 3)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


@pytest.mark.parametrize("name,units", [
    ("long", [(0, 0), (0, 31)]),
    ("slow", [(0, 5)]),
])
def test_segmented_full_size(name, units):
    inp = synth.workload_inputs(name, device="cuda")
    P = kda.kda_segments_auto(inp["T_total"], inp["H"], inp["N"])
    assert P > 1, "the one-sequence workloads are split on this device"
    out, fs = segmented(inp, 0)
    compare_units(inp, out, fs, units)
    of, sf = fused(inp)
    assert_close(f64(out), f64(of), f"{name}: segmented({P}) vs fused out")
    assert_close(f64(fs), f64(sf), f"{name}: segmented({P}) vs fused state")


def test_segmented_empty_input():
    inp = to_dev(synth.make_inputs(0, 2, lengths=[0, 0], seed=62, init_std=0.02))
    out, fs = segmented(inp, 3)
    assert out.numel() == 0
    assert torch.equal(fs, inp["initial_state"])


def test_segmented_through_host_buffers():
    # the host-buffer entry point with the segmented schedule: packed sequences
    # (one empty) in groups, initial states
    inp = synth.make_inputs(0, 2, lengths=[900, 0, 333, 70], seed=63, init_std=0.02)
    pin = {k: (inp[k].pin_memory() if inp[k] is not None else None)
           for k in ("q", "k", "v", "g_raw", "beta_raw", "initial_state", "cu_seqlens")}
    out, fs = kda.kda_forward_host(pin["q"], pin["k"], pin["v"], pin["g_raw"], pin["beta_raw"],
                                   inp["scale"], inp["lower_bound"], pin["initial_state"],
                                   pin["cu_seqlens"], schedule="segmented", groups=2)
    torch.cuda.synchronize()
    assert kda.kda_device_status() == 0
    ro, rs = oracle_case(inp)
    assert_close(f64(out), ro, "segmented host-buffer out")
    assert_close(f64(fs), rs, "segmented host-buffer final_state")


def test_segmented_without_final_state_and_small_workspace():
    inp = to_dev(synth.make_inputs(0, 2, lengths=[500, 200], seed=64, init_std=0.02))
    out, fs = segmented(inp, 3, output_final_state=False)
    assert fs is None
    ro, _ = oracle_case(inp)
    assert_close(f64(out), ro, "segmented out without a final state")
    nbytes = kda.kda_segmented_workspace_size(inp["T_total"], 2, 2, segments=3)
    small = torch.empty(nbytes - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(kda.KdaError) as e:
        segmented(inp, 3, workspace=small)
    assert e.value.status == 3


@pytest.mark.parametrize("per_head", [False, True])
def test_segmented_schedule_options_bf16_states(per_head):
    # kda_forward with the segmented schedule: bf16 initial and final states
    # (the pieces' states stay fp32 inside), per-channel or per-head gate; the
    # automatic count splits 512 chunks of 2 heads into 8 pieces
    inp = to_dev(synth.make_inputs(8192, 2, 1, seed=65, init_std=0.02, g_mean=-3.0))
    assert kda.kda_segments_auto(8192, 2, 1) > 1
    init16 = inp["initial_state"].to(torch.bfloat16)
    g = inp["g_raw"][:, :, 0].contiguous() if per_head else inp["g_raw"]
    out, fs = kda.kda_forward(inp["q"], inp["k"], inp["v"], g, inp["beta_raw"], inp["scale"],
                              inp["lower_bound"], init16, None, N=1, schedule="segmented")
    assert kda.kda_device_status() == 0
    assert fs.dtype == torch.bfloat16
    ref = dict(inp, initial_state=init16.float(),
               g_raw=g[:, :, None].expand(-1, -1, 128).contiguous() if per_head else g)
    ro, rs = oracle_case(ref)
    assert_close(f64(out), ro, "segmented schedule out (bf16 states)")
    assert_close(f64(fs), rs, "segmented schedule final_state (bf16 states)")


@pytest.mark.parametrize("n_seq,H", [(24, 2), (40, 2)])
def test_segmented_many_units(n_seq, H):
    # 48 and 80 (sequence, head) units: the scan runs with 64 and 128 value
    # rows per CTA (one CTA per SM), the shapes few-unit cases never reach
    import random
    rng = random.Random(n_seq)
    lengths = [rng.randint(60, 400) for _ in range(n_seq)]
    inp = to_dev(synth.make_inputs(0, H, lengths=lengths, seed=66, init_std=0.02))
    out, fs = segmented(inp, 2)
    ro, rs = oracle_case(inp)
    assert_close(f64(out), ro, f"segmented, {n_seq * H} units, out")
    assert_close(f64(fs), rs, f"segmented, {n_seq * H} units, final_state")
