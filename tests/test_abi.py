"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every function include/kda.h declares, sizes its workspace, and rejects bad
arguments with the documented status before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

import chunked_gated_delta_11_gb300 as kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from chunked_gated_delta_11_gb300 import build
    build.build()
    return kda.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "kda_fwd" in names and "kda_workspace_size" in names
    for name in names:
        assert hasattr(lib, name), f"{name} declared in kda.h but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", kda.build.LIB], capture_output=True,
                         text=True).stdout
    for name in names:
        assert re.search(rf"\bT {name}\b", out), name


def test_workspace_size(lib):
    rec = kda.REC_BYTES
    assert kda.kda_workspace_size(65536, 32, 8) == ((65536 // 16 + 8 + 1) * 32 * rec + 255) // 256 * 256
    assert kda.kda_workspace_size(0, 1, 1) >= rec
    assert kda.kda_workspace_size(64, 1, 1, D=64) == 0
    assert kda.kda_workspace_size(-1, 1, 1) == 0
    assert kda.kda_workspace_size(64, 0, 1) == 0


FAKE = 1 << 20  # aligned, never dereferenced: validation fails first


def call_fwd(lib, *, q=FAKE, out=FAKE, T=64, H=1, N=1, D=128, lb=-5.0, scale=0.1, beta=FAKE,
             init=None, final=None, ws=None, ws_bytes=0):
    P = ctypes.c_void_p
    return lib.kda_fwd(P(q), P(FAKE), P(FAKE), P(FAKE), P(beta), scale, lb, P(init) if init else None,
                       None, T, H, N, D, P(out), P(final) if final else None,
                       P(ws) if ws else None, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(D=64), 2),                 # head size other than 128
    (dict(lb=-6.0), 2),              # lower_bound outside [-5, 0]
    (dict(lb=0.5), 2),
    (dict(lb=float("nan")), 2),
    (dict(H=0), 1),
    (dict(N=0), 1),
    (dict(T=-1), 1),
    (dict(T=65, N=2), 1),            # equal split impossible without cu_seqlens
    (dict(T=1 << 31), 1),            # token coordinates of the tensor-map copies are int32
    (dict(q=0), 1),                  # null input
    (dict(q=FAKE + 8), 1),           # misaligned input
    (dict(beta=FAKE + 1), 1),        # misaligned bf16 beta
    (dict(out=0), 1),                # null output
    (dict(init=FAKE + 4), 1),        # misaligned state
    (dict(scale=float("nan")), 1),
    (dict(ws=FAKE, ws_bytes=100), 3),  # workspace too small
])
def test_fwd_rejects_bad_arguments(lib, kw, status):
    assert call_fwd(lib, **kw) == status


def test_stage_entry_points_reject_bad_arguments(lib):
    P = ctypes.c_void_p
    # K1 needs a workspace
    assert lib.kda_chunk_prep(P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 0.1, -5.0, None, 64, 1,
                              1, 128, None, 0, None) == 1
    assert lib.kda_chunk_prep(P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 0.1, -5.0, None, 64, 1,
                              1, 128, P(FAKE), 16, None) == 3
    # K2: size and output checks
    assert lib.kda_chunk_recurrence(P(FAKE), 1 << 30, None, None, 64, 1, 1, 100, P(FAKE), None,
                                    None) == 2
    assert lib.kda_chunk_recurrence(P(FAKE), 1 << 30, None, None, 64, 1, 1, 128, None, None,
                                    None) == 1


def test_status_strings(lib):
    for code in range(6):
        s = kda.kda_status_string(code)
        assert isinstance(s, str) and s
    assert kda.kda_status_string(99) == "unknown status"


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import chunked_gated_delta_11_gb300 as m
    monkeypatch.setattr(m, "_lib", None)
    monkeypatch.setattr(m, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        m.load()


def test_forward_rejects_bad_options(lib):
    P = ctypes.c_void_p
    args = [P(FAKE)] * 5 + [0.1, -5.0, None, None, 64, 1, 1, 128, P(FAKE), P(FAKE), None, 0, None]
    assert lib.kda_forward(None, *args) == 1                      # no options
    for bad in ((5, 0, 0), (1, 2, 0), (1, 0, 2), (-1, 0, 0)):
        opts = kda._Options(*bad)
        assert lib.kda_forward(ctypes.byref(opts), *args) == 1, bad
    opts = kda._Options(1, 0, 0)
    assert lib.kda_forward(ctypes.byref(opts), *args[:9], 64, 1, 1, 64, *args[13:]) == 2  # D


def test_segmented_workspace_size(lib):
    # boundaries and work list (256 B each), X and M states (N P H 64 KiB each), bf16 starting
    # states (N P H 32 KiB), y (T H 256 B)
    assert kda.kda_segmented_workspace_size(4096, 4, 1, segments=4) == (512 + 2 * 4 * 4 * 65536 + 4 * 4 * 32768
                                                                       + 4096 * 4 * 256)
    assert kda.kda_segmented_workspace_size(4096, 4, 1, segments=1) == 0   # plain fused pass
    assert kda.kda_segmented_workspace_size(4096, 4, 1, segments=65) == 0  # more than 64 pieces
    assert kda.kda_segmented_workspace_size(4096, 4, 1, segments=-1) == 0
    assert kda.kda_segmented_workspace_size(4096, 4, 1, segments=4, D=64) == 0
    assert kda.kda_segmented_workspace_size(1 << 31, 1, 1, segments=2) == 0  # int32 boundaries


def test_segmented_rejects_bad_arguments(lib):
    P = ctypes.c_void_p

    def call(T=64, H=1, N=1, D=128, segments=2, gate=0, q=FAKE, lb=-5.0, ws=None, ws_bytes=0):
        return lib.kda_fwd_segmented(P(q), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 0.1, lb, None,
                                     None, T, H, N, D, P(FAKE), None, segments, gate,
                                     P(ws) if ws else None, ws_bytes, None)
    assert call(segments=65) == 1
    assert call(segments=-1) == 1
    assert call(gate=2) == 1
    assert call(D=64) == 2
    assert call(lb=-6.0) == 2
    assert call(q=FAKE + 8) == 1
    assert call(T=65, N=2) == 1
    assert call(T=1 << 31) == 1


def test_validate_cu_seqlens_rejects_bad_arguments(lib):
    P = ctypes.c_void_p
    assert lib.kda_validate_cu_seqlens(None, 2, 10, None) == 1           # null
    assert lib.kda_validate_cu_seqlens(P(FAKE), 0, 10, None) == 1        # no sequences
    assert lib.kda_validate_cu_seqlens(P(FAKE + 2), 2, 10, None) == 1    # misaligned
    assert lib.kda_validate_cu_seqlens(P(FAKE), 2, 1 << 31, None) == 1   # int32 range


def _host_call(lib, cu=None, T=64, H=1, N=1, groups=0, lb=-5.0, schedule=1, sd=0, gate=0, ws=None,
               ws_bytes=0):
    P = ctypes.c_void_p
    opts = kda._Options(schedule, sd, gate)
    buf = (ctypes.c_uint8 * 64)()
    hp = ctypes.cast(buf, P)
    cu_arr = None if cu is None else (ctypes.c_int32 * len(cu))(*cu)
    return lib.kda_fwd_host(ctypes.byref(opts), hp, hp, hp, hp, hp, 0.1, lb, None, cu_arr, T, H, N,
                            128, hp, None, groups, P(ws) if ws else None, ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(cu=[0, 5, 3, 64], N=3), 1),        # decreasing host cu_seqlens
    (dict(cu=[1, 64], N=1), 1),              # does not start at 0
    (dict(cu=[0, 60], N=1), 1),              # does not end at T_total
    (dict(groups=17), 1),                    # more pieces than the pipeline has streams
    (dict(groups=-1), 1),
    (dict(schedule=9), 1),
    (dict(sd=3), 1),
    (dict(lb=0.5), 2),
    (dict(T=63, N=2), 1),                    # T_total not a multiple of N without cu_seqlens
    (dict(ws=FAKE + 16, ws_bytes=1 << 30), 3),  # workspace not 256-byte aligned
])
def test_fwd_host_rejects_bad_arguments_on_the_host(lib, kw, status):
    # all of these are found before any CUDA call (no GPU needed)
    assert _host_call(lib, **kw) == status


def test_fwd_host_workspace_size_is_the_device_layout(lib):
    opts = kda._Options(1, 0, 0)
    r = lambda x: (x + 255) // 256 * 256
    T, H, N = 64, 2, 2
    rows = T * H
    state = N * H * 128 * 128 * 4
    cu_words = N + 2          # the groups' rebased cu_seqlens: 2 groups of 1 sequence
    want = (4 * r(rows * 256) + r(rows * 2) + r(rows * 256) + 2 * r(state) + r(cu_words * 4 + 4))
    got = lib.kda_fwd_host_workspace_size(ctypes.byref(opts), T, H, N, 128, None, 2)
    assert got == want
    assert lib.kda_fwd_host_workspace_size(ctypes.byref(opts), T, H, N, 64, None, 2) == 0
