"""Host test of the clamped sequence bounds (csrc/kda_bounds.h) that every
kernel applies to cu_seqlens entries: for any pair of int32 entries the bounds
satisfy 0 <= bos <= eos <= T_total, and a well-formed pair passes unchanged.
The header is plain C++, compiled here with the host compiler."""
import os
import subprocess
import tempfile

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "chunked_gated_delta_11_gb300", "csrc")

DRIVER = r"""
#include <cstdio>
#include "kda_bounds.h"
int main() {
  long long lo, hi, T;
  while (std::scanf("%lld %lld %lld", &lo, &hi, &T) == 3) {
    int64_t bos, eos;
    kda::clamp_seq_bounds(lo, hi, T, bos, eos);
    std::printf("%lld %lld\n", (long long)bos, (long long)eos);
  }
  return 0;
}
"""


@pytest.fixture(scope="module")
def clamp():
    cxx = None
    for cand in ("g++", "c++", "clang++"):
        if subprocess.run(["which", cand], capture_output=True).returncode == 0:
            cxx = cand
            break
    if cxx is None:
        pytest.skip("no host C++ compiler")
    d = tempfile.mkdtemp()
    src, exe = os.path.join(d, "b.cpp"), os.path.join(d, "b")
    open(src, "w").write(DRIVER)
    subprocess.run([cxx, "-O1", "-std=c++17", "-I", CSRC, src, "-o", exe], check=True)

    def run(cases):
        inp = "".join(f"{lo} {hi} {T}\n" for lo, hi, T in cases)
        out = subprocess.run([exe], input=inp, capture_output=True, text=True, check=True).stdout
        return [tuple(int(x) for x in line.split()) for line in out.strip().splitlines()]
    return run


def test_well_formed_bounds_pass_unchanged(clamp):
    cases = [(0, 0, 0), (0, 5, 5), (3, 9, 20), (20, 20, 20), (0, 2 ** 31 - 1, 2 ** 31 - 1)]
    assert clamp(cases) == [(lo, hi) for lo, hi, _ in cases]


def test_malformed_bounds_stay_inside(clamp):
    rng = np.random.default_rng(5)
    cases = [(-7, 4, 10), (4, -7, 10), (12, 30, 10), (8, 3, 10), (-1, -1, 0), (15, 15, 10),
             (-(2 ** 31), 2 ** 31 - 1, 1000)]
    cases += [(int(a), int(b), int(t)) for a, b, t in zip(rng.integers(-2 ** 31, 2 ** 31, 200),
                                                          rng.integers(-2 ** 31, 2 ** 31, 200),
                                                          rng.integers(0, 2 ** 31, 200))]
    for (lo, hi, T), (bos, eos) in zip(cases, clamp(cases)):
        assert 0 <= bos <= eos <= T, (lo, hi, T, bos, eos)
        if 0 <= lo <= T:
            assert bos == lo
        if bos <= hi <= T:
            assert eos == hi
    # the last record slot of a sequence stays below T / 16 + n + 1 (n < N)
    for (lo, hi, T), (bos, eos) in zip(cases, clamp(cases)):
        nch = (eos - bos + 15) // 16
        if nch:
            assert bos // 16 + nch - 1 < T // 16 + 1
