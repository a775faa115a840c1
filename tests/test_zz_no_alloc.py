"""kda_fwd_noalloc, the entry point for callers that cannot allocate device
memory (its chunk records live in a fixed 64 MiB array inside libkda), checked
through the C ABI against kda_fwd on two calls in a row.  The second call runs
on other inputs, so it also shows that what the first call left in the shared
array does not leak into the next result.  Collected last on purpose."""
import pytest
import torch

import chunked_gated_delta_11_gb300 as kda
from chunked_gated_delta_11_gb300 import synth
from kda_testlib import assert_close, f64

pytestmark = pytest.mark.gpu


def _dev(inp):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def test_noalloc_matches_kda_fwd_on_two_calls():
    kda.build.build()
    kda.load()
    cases = [
        synth.make_inputs(0, 4, lengths=[300, 17, 1, 64], seed=21, init_std=0.02),
        synth.make_inputs(2 * 400, 8, 2, seed=22),
    ]
    for inp in map(_dev, cases):
        ref_out, ref_fs = kda.kda_fwd(inp["q"], inp["k"], inp["v"], inp["g_raw"],
                                      inp["beta_raw"], inp["scale"], inp["lower_bound"],
                                      inp["initial_state"], inp["cu_seqlens"], N=inp["N"])
        out = torch.full_like(ref_out, float("nan"))
        fs = torch.full_like(ref_fs, float("nan"))
        kda.kda_fwd_noalloc(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"],
                            inp["scale"], inp["lower_bound"], out, fs, inp["initial_state"],
                            inp["cu_seqlens"], N=inp["N"])
        assert kda.kda_device_status() == 0
        assert_close(f64(out), f64(ref_out), "noalloc out")
        assert_close(f64(fs), f64(ref_fs), "noalloc final_state")


def test_noalloc_at_its_size_limit():
    # H = 32, N = 1: T_total = 1248 needs 80 record slots x 32 heads x 26176 B,
    # just under the 64 MiB array; T_total = 1264 needs 81 slots, just over
    H = 32
    assert kda.kda_workspace_size(1248, H, 1) <= kda.NOALLOC_WORKSPACE_BYTES
    assert kda.kda_workspace_size(1264, H, 1) > kda.NOALLOC_WORKSPACE_BYTES
    inp = _dev(synth.make_inputs(1248, H, 1, seed=23, init_std=0.02))
    ref_out, ref_fs = kda.kda_fwd(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"],
                                  inp["scale"], inp["lower_bound"], inp["initial_state"], N=1)
    out = torch.full_like(ref_out, float("nan"))
    fs = torch.full_like(ref_fs, float("nan"))
    kda.kda_fwd_noalloc(inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"],
                        inp["scale"], inp["lower_bound"], out, fs, inp["initial_state"], N=1)
    assert kda.kda_device_status() == 0
    assert_close(f64(out), f64(ref_out), "noalloc out at the limit")
    assert_close(f64(fs), f64(ref_fs), "noalloc final_state at the limit")
    x = torch.zeros((1264, H, 128), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros((1264, H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kda.KdaError) as e:
        kda.kda_fwd_noalloc(x, x, x, x, b, 0.1, -5.0, torch.empty_like(x))
    assert e.value.status == 3


def test_noalloc_rejects_sizes_beyond_its_array():
    kda.load()
    T, H = 4096, 32   # needs (4096/16 + 2) slots x 32 heads x 26176 B > 64 MiB
    assert kda.kda_workspace_size(T, H, 1) > kda.NOALLOC_WORKSPACE_BYTES
    x = torch.zeros((T, H, 128), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kda.KdaError) as e:
        kda.kda_fwd_noalloc(x, x, x, x, b, 0.1, -5.0, torch.empty_like(x))
    assert e.value.status == 3
