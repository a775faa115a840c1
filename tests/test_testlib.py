"""CPU checks of the parity helpers the GPU tests rely on: the streaming
whole-tensor comparison (oracle in time slices with the fp64 state handed
over) reproduces the one-shot oracle exactly, and a planted error in one
element of the output or of the state fails it."""
import numpy as np
import pytest
import torch

from chunked_gated_delta_11_gb300 import synth
from kda_testlib import oracle_case, stream_parity


def _case():
    return synth.make_inputs(0, 2, lengths=[37, 0, 50, 16], seed=71, init_std=0.02)


def test_stream_parity_slices_match_the_one_shot_oracle():
    inp = _case()
    ro, rs = oracle_case(inp)
    res = {"oracle": (torch.from_numpy(ro), torch.from_numpy(rs))}
    rep = stream_parity(inp, res, slice_tokens=16)
    assert rep["oracle"]["out"][1] < 1e-12 and rep["oracle"]["state"][1] < 1e-12


@pytest.mark.parametrize("where", ["out", "state"])
def test_stream_parity_catches_a_planted_error(where):
    inp = _case()
    ro, rs = oracle_case(inp)
    ro, rs = ro.copy(), rs.copy()
    if where == "out":
        ro[60, 1, 7] += 0.05 * np.abs(ro).max()
    else:
        rs[2, 0, 3, 4] += 0.05 * np.abs(rs).max()
    with pytest.raises(AssertionError):
        stream_parity(inp, {"planted": (torch.from_numpy(ro), torch.from_numpy(rs))},
                      slice_tokens=16)
