"""Python binding of libkda, the GB300 (sm_103a) Kimi Delta Attention forward.

Argument marshalling only: every step of the forward pass runs in the CUDA
kernels of ``libkda.so`` (built in-tree by ``build.py``); PyTorch supplies
device memory and streams.  Names follow the C ABI in ``include/kda.h``.
There is no fallback: if the library is missing, every call raises.

Layout: q, k, v, g_raw bf16 [T_total, H, 128]; beta_raw bf16 [T_total, H];
out bf16 [T_total, H, 128]; states fp32 [N, H, 128, 128] (value x key);
cu_seqlens int32 [N + 1] (device) or None for N equal sequences.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB as _LIB_PATH
from .build import build as _build

__all__ = [
    "KdaError", "load", "kda_workspace_size", "kda_fwd", "kda_chunk_prep",
    "kda_chunk_recurrence", "kda_device_status", "kda_status_string", "kda_selftest_tcgen05",
    "kda_selftest_timeout", "kda_fwd_host_workspace_size",
    "kda_forward_host", "kda_fwd_fused", "kda_decode", "kda_forward", "kda_fwd_noalloc",
    "kda_fwd_segmented", "kda_segments_auto", "kda_segmented_workspace_size",
    "kda_validate_cu_seqlens", "REC_BYTES", "CHUNK", "HEAD_DIM",
]

CHUNK = 16
HEAD_DIM = 128
REC_BYTES = 26176

SCHEDULES = {"split": 0, "fused": 1, "decode": 2, "segmented": 3, "auto": 4}


class _Options(ctypes.Structure):
    """kda_options of include/kda.h."""
    _fields_ = [("schedule", ctypes.c_int32), ("state_dtype", ctypes.c_int32),
                ("gate", ctypes.c_int32)]


STATUS = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED",
          3: "KDA_ERR_WORKSPACE", 4: "KDA_ERR_LAUNCH", 5: "KDA_ERR_TIMEOUT"}

_lock = threading.Lock()
_lib = None


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS.get(self.status, self.status)} "
                         f"({kda_status_string(self.status)})")


def load(build_if_missing: bool = False):
    """Load libkda.so (optionally building it first).  Raises if it is absent."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            if not build_if_missing:
                raise RuntimeError(f"libkda is not built ({_LIB_PATH} missing); "
                                   "run chunked_gated_delta_11_gb300.build.build()")
            _build()
        lib = ctypes.CDLL(_LIB_PATH)
        P, i64, i32, f32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                ctypes.c_float, ctypes.c_size_t)
        lib.kda_workspace_size.argtypes = [i64, i32, i32, i32]
        lib.kda_workspace_size.restype = sz
        lib.kda_fwd.argtypes = [P, P, P, P, P, f32, f32, P, P, i64, i32, i32, i32, P, P, P, sz, P]
        lib.kda_fwd.restype = ctypes.c_int
        lib.kda_fwd_fused.argtypes = [P, P, P, P, P, f32, f32, P, P, i64, i32, i32, i32, P, P, P]
        lib.kda_fwd_fused.restype = ctypes.c_int
        lib.kda_decode.argtypes = lib.kda_fwd_fused.argtypes
        lib.kda_decode.restype = ctypes.c_int
        lib.kda_forward.argtypes = [P, P, P, P, P, P, f32, f32, P, P, i64, i32, i32, i32, P, P,
                                    P, sz, P]
        lib.kda_forward.restype = ctypes.c_int
        lib.kda_fwd_noalloc.argtypes = [P, P, P, P, P, f32, f32, P, P, i64, i32, i32, i32, P, P,
                                        P]
        lib.kda_fwd_noalloc.restype = ctypes.c_int
        lib.kda_chunk_prep.argtypes = [P, P, P, P, P, f32, f32, P, i64, i32, i32, i32, P, sz, P]
        lib.kda_chunk_prep.restype = ctypes.c_int
        lib.kda_chunk_recurrence.argtypes = [P, sz, P, P, i64, i32, i32, i32, P, P, P]
        lib.kda_chunk_recurrence.restype = ctypes.c_int
        lib.kda_device_status.argtypes = [P]
        lib.kda_device_status.restype = ctypes.c_int
        lib.kda_status_string.argtypes = [ctypes.c_int]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_fwd_segmented.argtypes = [P, P, P, P, P, f32, f32, P, P, i64, i32, i32, i32, P,
                                          P, i32, i32, P, sz, P]
        lib.kda_fwd_segmented.restype = ctypes.c_int
        lib.kda_segmented_workspace_size.argtypes = [i64, i32, i32, i32, i32]
        lib.kda_segmented_workspace_size.restype = sz
        lib.kda_segments_auto.argtypes = [i64, i32, i32]
        lib.kda_segments_auto.restype = i32
        lib.kda_validate_cu_seqlens.argtypes = [P, i32, i64, P]
        lib.kda_validate_cu_seqlens.restype = ctypes.c_int
        lib.kda_fwd_host.argtypes = [P, P, P, P, P, P, f32, f32, P, P, i64, i32, i32, i32, P, P,
                                     i32, P, sz, P]
        lib.kda_fwd_host.restype = ctypes.c_int
        lib.kda_fwd_host_workspace_size.argtypes = [P, i64, i32, i32, i32, P, i32]
        lib.kda_fwd_host_workspace_size.restype = sz
        lib.kda_profile_phases.argtypes = [i32, P, P, P, P, P, f32, f32, i64, i32, i32, i32, P,
                                           P, P, sz, P, i32, P]
        lib.kda_profile_phases.restype = ctypes.c_int
        lib.kda_piece_workspace_size.argtypes = [i64, i32]
        lib.kda_piece_workspace_size.restype = sz
        lib.kda_piece_forward.argtypes = [P, P, P, P, P, f32, f32, P, i64, i32, i32, P, P, P, P,
                                          i32, P, sz, P]
        lib.kda_piece_forward.restype = ctypes.c_int
        lib.kda_pieces_scan.argtypes = [P, P, i32, i32, i32, P, P]
        lib.kda_pieces_scan.restype = ctypes.c_int
        lib.kda_piece_fixup.argtypes = [P, P, P, i64, i32, i32, P, sz, P]
        lib.kda_piece_fixup.restype = ctypes.c_int
        lib.kda_selftest_timeout.argtypes = [i64, P]
        lib.kda_selftest_timeout.restype = ctypes.c_int
        lib.kda_selftest_tcgen05.argtypes = [P, P, P, P]
        lib.kda_selftest_tcgen05.restype = ctypes.c_int
        _lib = lib
        return lib


def kda_status_string(status: int) -> str:
    return load().kda_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status, where):
    if status != 0:
        raise KdaError(status, where)


def _need(t, name, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def kda_workspace_size(T_total: int, H: int, N: int, D: int = HEAD_DIM) -> int:
    return int(load().kda_workspace_size(int(T_total), int(H), int(N), int(D)))


def _geometry(q, cu_seqlens, N):
    T_total, H, D = q.shape
    if cu_seqlens is not None:
        _need(cu_seqlens, "cu_seqlens", torch.int32)
        N = cu_seqlens.shape[0] - 1
    elif N is None:
        N = 1
    return T_total, H, D, int(N)


def kda_fwd(q, k, v, g_raw, beta_raw, scale, lower_bound, initial_state=None, cu_seqlens=None,
            N=None, out=None, final_state=None, workspace=None, stream=None,
            output_final_state=True):
    """One forward pass (K1 then K2) on device tensors; returns (out, final_state)."""
    T_total, H, D, N = _geometry(q, cu_seqlens, N)
    for name, t in (("q", q), ("k", k), ("v", v), ("g_raw", g_raw)):
        _need(t, name, torch.bfloat16, (T_total, H, D))
    _need(beta_raw, "beta_raw", torch.bfloat16, (T_total, H))
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, (N, H, D, D))
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, (T_total, H, D))
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, D, D), dtype=torch.float32, device=q.device)
    if final_state is not None:
        _need(final_state, "final_state", torch.float32, (N, H, D, D))
    ws_bytes = 0
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8)
        ws_bytes = workspace.numel()
    st = load().kda_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta_raw), float(scale),
                        float(lower_bound), _ptr(initial_state), _ptr(cu_seqlens), T_total, H, N,
                        D, _ptr(out), _ptr(final_state), _ptr(workspace), ws_bytes,
                        _stream(stream))
    _check(st, "kda_fwd")
    return out, final_state


def kda_fwd_fused(q, k, v, g_raw, beta_raw, scale, lower_bound, initial_state=None,
                  cu_seqlens=None, N=None, out=None, final_state=None, stream=None,
                  output_final_state=True):
    """One forward pass in a single kernel (records stay in shared memory);
    returns (out, final_state)."""
    T_total, H, D, N = _geometry(q, cu_seqlens, N)
    for name, t in (("q", q), ("k", k), ("v", v), ("g_raw", g_raw)):
        _need(t, name, torch.bfloat16, (T_total, H, D))
    _need(beta_raw, "beta_raw", torch.bfloat16, (T_total, H))
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, (N, H, D, D))
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, (T_total, H, D))
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, D, D), dtype=torch.float32, device=q.device)
    if final_state is not None:
        _need(final_state, "final_state", torch.float32, (N, H, D, D))
    st = load().kda_fwd_fused(_ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta_raw),
                              float(scale), float(lower_bound), _ptr(initial_state),
                              _ptr(cu_seqlens), T_total, H, N, D, _ptr(out), _ptr(final_state),
                              _stream(stream))
    _check(st, "kda_fwd_fused")
    return out, final_state


NOALLOC_WORKSPACE_BYTES = 64 * 1024 * 1024


def kda_decode(q, k, v, g_raw, beta_raw, scale, lower_bound, initial_state=None,
               cu_seqlens=None, N=None, out=None, final_state=None, stream=None,
               output_final_state=True):
    """The forward pass in the recurrent (decode) schedule: token by token, the
    state slice of each (sequence, head, 32 value rows) in registers.  For a few
    tokens per sequence per call; final_state may be initial_state itself
    (updated in place).  Returns (out, final_state)."""
    T_total, H, D, N = _geometry(q, cu_seqlens, N)
    for name, t in (("q", q), ("k", k), ("v", v), ("g_raw", g_raw)):
        _need(t, name, torch.bfloat16, (T_total, H, D))
    _need(beta_raw, "beta_raw", torch.bfloat16, (T_total, H))
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, (N, H, D, D))
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, (T_total, H, D))
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, D, D), dtype=torch.float32, device=q.device)
    if final_state is not None:
        _need(final_state, "final_state", torch.float32, (N, H, D, D))
    st = load().kda_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta_raw),
                           float(scale), float(lower_bound), _ptr(initial_state),
                           _ptr(cu_seqlens), T_total, H, N, D, _ptr(out), _ptr(final_state),
                           _stream(stream))
    _check(st, "kda_decode")
    return out, final_state


def kda_forward(q, k, v, g_raw, beta_raw, scale, lower_bound, initial_state=None,
                cu_seqlens=None, N=None, out=None, final_state=None, schedule="fused",
                workspace=None, stream=None, output_final_state=True):
    """The forward pass with the options of kda_forward in include/kda.h, read off
    the tensors: states fp32 or bf16 (both the same; the final state is allocated
    with the initial state's dtype), g_raw [T_total, H, 128] (per channel) or
    [T_total, H] (one gate per token and head).  schedule: "fused", "split",
    "decode", "segmented" (automatic piece count) or "auto" (decode for at most
    8 tokens per sequence, segmented when the units are too few for the SMs,
    fused otherwise).  Returns (out, final_state)."""
    T_total, H, D, N = _geometry(q, cu_seqlens, N)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, (T_total, H, D))
    per_head = g_raw.dim() == 2
    _need(g_raw, "g_raw", torch.bfloat16, (T_total, H) if per_head else (T_total, H, D))
    _need(beta_raw, "beta_raw", torch.bfloat16, (T_total, H))
    dtypes = {t.dtype for t in (initial_state, final_state) if t is not None}
    if len(dtypes) > 1:
        raise TypeError("initial_state and final_state must have the same dtype")
    sdt = dtypes.pop() if dtypes else torch.float32
    if sdt not in (torch.float32, torch.bfloat16):
        raise TypeError(f"states must be float32 or bfloat16, got {sdt}")
    if initial_state is not None:
        _need(initial_state, "initial_state", sdt, (N, H, D, D))
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, (T_total, H, D))
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, D, D), dtype=sdt, device=q.device)
    if final_state is not None:
        _need(final_state, "final_state", sdt, (N, H, D, D))
    ws_bytes = 0
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8)
        ws_bytes = workspace.numel()
    opts = _Options(SCHEDULES[schedule], 1 if sdt == torch.bfloat16 else 0, 1 if per_head else 0)
    st = load().kda_forward(ctypes.byref(opts), _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw),
                            _ptr(beta_raw), float(scale), float(lower_bound),
                            _ptr(initial_state), _ptr(cu_seqlens), T_total, H, N, D, _ptr(out),
                            _ptr(final_state), _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "kda_forward")
    return out, final_state


def kda_segments_auto(T_total: int, H: int, N: int) -> int:
    """Pieces per sequence kda_fwd_segmented picks by itself on the current device."""
    return int(load().kda_segments_auto(int(T_total), int(H), int(N)))


def kda_segmented_workspace_size(T_total: int, H: int, N: int, segments: int = 0,
                                 D: int = HEAD_DIM) -> int:
    return int(load().kda_segmented_workspace_size(int(T_total), int(H), int(N), int(D),
                                                   int(segments)))


def kda_fwd_segmented(q, k, v, g_raw, beta_raw, scale, lower_bound, initial_state=None,
                      cu_seqlens=None, N=None, segments=0, out=None, final_state=None,
                      workspace=None, stream=None, output_final_state=True):
    """The forward pass with every sequence cut into `segments` pieces run at
    once and joined by a scan of their state maps (kda_fwd_segmented in
    include/kda.h; 0 = the automatic count).  States fp32; g_raw
    [T_total, H, 128] (per channel) or [T_total, H] (one gate per token and
    head).  Returns (out, final_state)."""
    T_total, H, D, N = _geometry(q, cu_seqlens, N)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need(t, name, torch.bfloat16, (T_total, H, D))
    per_head = g_raw.dim() == 2
    _need(g_raw, "g_raw", torch.bfloat16, (T_total, H) if per_head else (T_total, H, D))
    _need(beta_raw, "beta_raw", torch.bfloat16, (T_total, H))
    if initial_state is not None:
        _need(initial_state, "initial_state", torch.float32, (N, H, D, D))
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16, (T_total, H, D))
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, D, D), dtype=torch.float32, device=q.device)
    if final_state is not None:
        _need(final_state, "final_state", torch.float32, (N, H, D, D))
    ws_bytes = 0
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8)
        ws_bytes = workspace.numel()
    st = load().kda_fwd_segmented(_ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta_raw),
                                  float(scale), float(lower_bound), _ptr(initial_state),
                                  _ptr(cu_seqlens), T_total, H, N, D, _ptr(out),
                                  _ptr(final_state), int(segments), 1 if per_head else 0,
                                  _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "kda_fwd_segmented")
    return out, final_state


def kda_fwd_noalloc(q, k, v, g_raw, beta_raw, scale, lower_bound, out, final_state=None,
                    initial_state=None, cu_seqlens=None, N=None, stream=None):
    """kda_fwd for callers that cannot allocate device memory: the chunk records
    go to a fixed 64 MiB array inside libkda, so the call allocates nothing.
    `out` (and `final_state`, if wanted) must be given.  Sizes whose workspace
    exceeds 64 MiB raise KdaError(KDA_ERR_WORKSPACE).  Calls that overlap on the
    GPU share that array and race."""
    T_total, H, D, N = _geometry(q, cu_seqlens, N)
    st = load().kda_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta_raw),
                                float(scale), float(lower_bound), _ptr(initial_state),
                                _ptr(cu_seqlens), T_total, H, N, D, _ptr(out), _ptr(final_state),
                                _stream(stream))
    _check(st, "kda_fwd_noalloc")
    return out, final_state


def kda_chunk_prep(q, k, v, g_raw, beta_raw, scale, lower_bound, workspace, cu_seqlens=None,
                   N=None, stream=None):
    """K1 alone: writes the chunk records into `workspace` (uint8 device tensor)."""
    T_total, H, D, N = _geometry(q, cu_seqlens, N)
    _need(workspace, "workspace", torch.uint8)
    st = load().kda_chunk_prep(_ptr(q), _ptr(k), _ptr(v), _ptr(g_raw), _ptr(beta_raw),
                               float(scale), float(lower_bound), _ptr(cu_seqlens), T_total, H, N,
                               D, _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "kda_chunk_prep")
    return workspace


def kda_chunk_recurrence(workspace, T_total, H, out, initial_state=None, final_state=None,
                         cu_seqlens=None, N=None, D=HEAD_DIM, stream=None):
    """K2 alone, over records written by kda_chunk_prep."""
    if cu_seqlens is not None:
        N = cu_seqlens.shape[0] - 1
    N = 1 if N is None else int(N)
    _need(workspace, "workspace", torch.uint8)
    st = load().kda_chunk_recurrence(_ptr(workspace), workspace.numel(), _ptr(initial_state),
                                     _ptr(cu_seqlens), int(T_total), int(H), N, int(D), _ptr(out),
                                     _ptr(final_state), _stream(stream))
    _check(st, "kda_chunk_recurrence")
    return out, final_state


def kda_validate_cu_seqlens(cu_seqlens, T_total: int, stream=None):
    """Queue the device check of cu_seqlens (starts at 0, non-decreasing, ends at
    T_total); a violation shows as KDA_ERR_INVALID_ARG from kda_device_status()."""
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    st = load().kda_validate_cu_seqlens(_ptr(cu_seqlens), cu_seqlens.numel() - 1, int(T_total),
                                        _stream(stream))
    _check(st, "kda_validate_cu_seqlens")


def kda_device_status(stream=None) -> int:
    """Synchronise and return (and clear) the device error word: 0 or a status."""
    return int(load().kda_device_status(_stream(stream)))


def kda_selftest_timeout(limit_cycles: int = 100_000, stream=None):
    """Queue the diagnostic whose bounded wait runs out after `limit_cycles`
    SM cycles; kda_device_status() then reports KDA_ERR_TIMEOUT (5) once."""
    _check(load().kda_selftest_timeout(int(limit_cycles), _stream(stream)),
           "kda_selftest_timeout")


def kda_selftest_tcgen05(device="cuda"):
    out1 = torch.zeros((128, 32), dtype=torch.float32, device=device)
    out2 = torch.zeros((128, 144), dtype=torch.float32, device=device)
    status = torch.zeros((1,), dtype=torch.int32, device=device)
    rc = load().kda_selftest_tcgen05(_ptr(out1), _ptr(out2), _ptr(status), _stream(None))
    if rc != 0:
        raise KdaError(rc, "kda_selftest_tcgen05")
    torch.cuda.synchronize()
    return out1, out2, int(status.item())


def kda_fwd_host_workspace_size(T_total: int, H: int, N: int, cu_seqlens=None,
                                schedule: str = "fused", state_bf16: bool = False,
                                per_head_gate: bool = False, groups: int = 8) -> int:
    """Device workspace bytes of kda_fwd_host (cu_seqlens: host int32 tensor or None)."""
    opts = _Options(SCHEDULES[schedule], 1 if state_bf16 else 0, 1 if per_head_gate else 0)
    return int(load().kda_fwd_host_workspace_size(ctypes.byref(opts), int(T_total), int(H),
                                                  int(N), HEAD_DIM, _hptr(cu_seqlens),
                                                  int(groups)))


def _hptr(t):
    if t is None:
        return None
    if t.device.type != "cpu":
        raise ValueError("kda_forward_host takes host tensors")
    if not t.is_contiguous():
        raise ValueError("host tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def kda_forward_host(q, k, v, g_raw, beta_raw, scale, lower_bound, initial_state=None,
                     cu_seqlens=None, N=None, device="cuda", out=None, final_state=None,
                     stream=None, schedule="fused", groups=8, workspace=None):
    """Forward pass on host (CPU, ideally pinned) tensors through kda_fwd_host:
    libkda copies the inputs in, runs the pass and copies the outputs back in a
    pipeline of `groups` pieces (groups of whole sequences, or chunk-aligned
    time slices of few equal sequences).  Returns (out, final_state) as host
    tensors (allocated pinned if not given), complete once `stream` (default:
    the current stream of `device`) is.  The device workspace comes from
    torch's caching allocator on that stream unless `workspace` is given."""
    dev = torch.device(device)
    stream = torch.cuda.current_stream(dev) if stream is None else stream
    T_total, H, D = q.shape
    if cu_seqlens is not None:
        if cu_seqlens.dtype != torch.int32:
            raise TypeError("cu_seqlens must be int32")
        N = cu_seqlens.shape[0] - 1
    elif N is None:
        N = 1
    per_head = g_raw.dim() == 2
    sdt = initial_state.dtype if initial_state is not None else (
        final_state.dtype if final_state is not None else torch.float32)
    if sdt not in (torch.float32, torch.bfloat16):
        raise TypeError(f"states must be float32 or bfloat16, got {sdt}")
    for name, t in (("q", q), ("k", k), ("v", v), ("g_raw", g_raw), ("beta_raw", beta_raw)):
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bfloat16")
    if out is None:
        out = torch.empty((T_total, H, D), dtype=torch.bfloat16, pin_memory=True)
    if final_state is None:
        final_state = torch.empty((N, H, D, D), dtype=sdt, pin_memory=True)
    opts = _Options(SCHEDULES[schedule], 1 if sdt == torch.bfloat16 else 0, 1 if per_head else 0)
    cu = None if cu_seqlens is None else cu_seqlens.cpu().contiguous()
    nbytes = int(load().kda_fwd_host_workspace_size(ctypes.byref(opts), T_total, H, N, D,
                                                    _hptr(cu), int(groups)))
    if nbytes == 0:
        raise KdaError(1, "kda_fwd_host_workspace_size")
    if workspace is None:
        with torch.cuda.stream(stream):
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8)
    with torch.cuda.device(dev):
        st = load().kda_fwd_host(ctypes.byref(opts), _hptr(q), _hptr(k), _hptr(v), _hptr(g_raw),
                                 _hptr(beta_raw), float(scale), float(lower_bound),
                                 _hptr(initial_state), _hptr(cu), T_total, H, N, D, _hptr(out),
                                 _hptr(final_state), int(groups), _ptr(workspace),
                                 workspace.numel(), ctypes.c_void_p(stream.cuda_stream))
    _check(st, "kda_fwd_host")
    return out, final_state
