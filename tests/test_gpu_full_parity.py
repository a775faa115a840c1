"""Whole-tensor parity at full size: every element of `out` and of the final
state of the B = 8 x 8192 (H = 32), varlen (64 packed sequences, H = 32,
initial states) and long (1 x 131072, H = 32) workloads, on each schedule that
serves them, against the fp64 oracle with the method's tolerance (max |err|
<= 1e-2 max |ref| and relative Frobenius <= 5e-3, over the whole tensor).
The oracle streams through each sequence in time slices (kda_testlib.stream_parity),
so the check costs host time but little host memory."""
import pytest

import chunked_gated_delta_11_gb300 as kda
from chunked_gated_delta_11_gb300 import synth
from kda_testlib import stream_parity

pytestmark = pytest.mark.gpu

WORKLOAD_SCHEDULES = {
    "b8": ["fused", "split"],
    "varlen": ["fused", "split"],
    "long": ["segmented", "fused", "split"],
}


@pytest.fixture(scope="module", autouse=True)
def _built():
    kda.build.build()
    kda.load()
    yield
    assert kda.kda_device_status() == 0


@pytest.mark.parametrize("name", list(WORKLOAD_SCHEDULES))
def test_whole_tensor_parity_full_size(name):
    inp = synth.workload_inputs(name, device="cuda")
    a = (inp["q"], inp["k"], inp["v"], inp["g_raw"], inp["beta_raw"], inp["scale"],
         inp["lower_bound"], inp["initial_state"], inp["cu_seqlens"])
    results = {}
    for schedule in WORKLOAD_SCHEDULES[name]:
        results[schedule] = kda.kda_forward(*a, N=inp["N"], schedule=schedule)
        assert kda.kda_device_status() == 0
    stream_parity(inp, results)
