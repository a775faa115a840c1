"""Host checks of the seeded input generator (no GPU): the named workloads
have the shapes, dtypes and sequence layouts their descriptions state, and a
(workload, seed) pair always gives the same bits."""
import torch

from chunked_gated_delta_11_gb300 import synth


def test_benchmark_row_workloads_shapes():
    # FlashKDA's benchmark rows: T = 8192, D = 128, H = 96 or 64; one sequence,
    # or 8 x 1024 passed packed with cu_seqlens
    for name, H in (("fk96", 96), ("fk64", 64)):
        w = synth.WORKLOADS[name]
        assert (w.H, w.N, w.T, w.packed) == (H, 1, 8192, False)
    for name, H in (("fk96p", 96), ("fk64p", 64)):
        w = synth.WORKLOADS[name]
        assert (w.H, w.N, w.T, w.packed) == (H, 8, 1024, True)


def test_packed_workload_inputs():
    # a packed workload's inputs carry cu_seqlens of equal lengths (drawn on a
    # small copy of the workload to keep the test light)
    w = synth.Workload("p", H=2, N=4, T=48, init_std=None, seed=3, packed=True)
    saved = synth.WORKLOADS.get("p")
    synth.WORKLOADS["p"] = w
    try:
        inp = synth.workload_inputs("p")
    finally:
        if saved is None:
            del synth.WORKLOADS["p"]
        else:
            synth.WORKLOADS["p"] = saved
    assert inp["cu_seqlens"].dtype == torch.int32
    assert inp["cu_seqlens"].tolist() == [0, 48, 96, 144, 192]
    assert inp["N"] == 4 and inp["T_total"] == 192
    assert inp["q"].shape == (192, 2, 128) and inp["q"].dtype == torch.bfloat16
    assert inp["beta_raw"].shape == (192, 2)


def test_same_seed_same_bits():
    a = synth.make_inputs(64, 2, 2, seed=5, init_std=0.02)
    b = synth.make_inputs(64, 2, 2, seed=5, init_std=0.02)
    for key in ("q", "k", "v", "g_raw", "beta_raw", "initial_state"):
        assert torch.equal(a[key], b[key])
    c = synth.make_inputs(64, 2, 2, seed=6, init_std=0.02)
    assert not torch.equal(a["q"], c["q"])
