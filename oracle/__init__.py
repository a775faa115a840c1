"""fp64 CPU oracle for the Kimi Delta Attention forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library in ``chunked_gated_delta_11_gb300`` never imports it
and shares no code with it.

The arithmetic lives in ``kda_oracle.c`` (plain C, double precision); this
module only marshals numpy arrays into it.  What each function computes, and the
passage it follows, is stated in that file:

* ``prepare``        -- L2 norm of q and k, log alpha = lower_bound * sigmoid(g_raw),
                        beta = sigmoid(beta_raw)  ("FlashKDA Delta Attention
                        Algorithm", Core Architecture).
* ``fwd``            -- token-by-token KDA recurrence ("You Could Have Come Up with
                        Kimi Delta Attention", sec. 4) or its chunkwise form (sec. 6).
* ``chunk_factors``  -- per-chunk Akk, Aqk, W, U, Qdec, Kend, dlast (sec. 6.1-6.6).
* ``neumann_inverse`` / ``product_inverse`` / ``trisolve_inverse`` -- three ways
                        to invert a unit lower-triangular matrix (sec. 6.3).

Every function is pinned in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

DEFAULT_EPS = 1e-6


def build(force: bool = False) -> str:
    """Compile kda_oracle.c with gcc into oracle/_build/libkda_oracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
           "-D_POSIX_C_SOURCE=200809L", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.kda_oracle_prepare.argtypes = [P, P, P, P, i64, i32, i32, f64, f64, P, P, P, P]
        lib.kda_oracle_prepare.restype = None
        lib.kda_oracle_fwd.argtypes = [P, P, P, P, P, P, P, i64, i32, i32, i32, i32,
                                       f64, i32, i32, P, P]
        lib.kda_oracle_fwd.restype = ctypes.c_int
        lib.kda_oracle_num_chunks.argtypes = [P, i64, i32, i32]
        lib.kda_oracle_num_chunks.restype = i64
        lib.kda_oracle_chunk_factors.argtypes = [P, P, P, P, P, P, i64, i32, i32, i32, i32,
                                                 f64, i32, P, P, P, P, P, P, P]
        lib.kda_oracle_chunk_factors.restype = i64
        for name in ("kda_oracle_neumann_inverse", "kda_oracle_product_inverse",
                     "kda_oracle_trisolve_inverse"):
            fn = getattr(lib, name)
            fn.argtypes = [P, i32, P]
            fn.restype = ctypes.c_int
        _lib = lib
        return lib


def _f64(a):
    return None if a is None else np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def prepare(q_raw, k_raw, g_raw, beta_raw, lower_bound, eps=DEFAULT_EPS):
    """Return (q_hat, k_hat, log_alpha, beta) in float64.

    q_raw, k_raw, g_raw: [T, H, K]; beta_raw: [T, H]."""
    q_raw, k_raw, g_raw, beta_raw = map(_f64, (q_raw, k_raw, g_raw, beta_raw))
    T, H, K = q_raw.shape
    q_hat, k_hat, la = (np.empty_like(q_raw) for _ in range(3))
    beta = np.empty_like(beta_raw)
    _load().kda_oracle_prepare(_ptr(q_raw), _ptr(k_raw), _ptr(g_raw), _ptr(beta_raw),
                               T, H, K, float(lower_bound), float(eps),
                               _ptr(q_hat), _ptr(k_hat), _ptr(la), _ptr(beta))
    return q_hat, k_hat, la, beta


def fwd(q, k, v, log_alpha, beta, scale, initial_state=None, cu_seqlens=None,
        N=1, chunk=0, nthreads=None):
    """KDA forward on transformed inputs (q, k already normalised as wanted).

    q, k, log_alpha: [T, H, K]; v: [T, H, V]; beta: [T, H];
    initial_state: [N, H, V, K] or None; cu_seqlens: int array [N + 1] or None.
    chunk = 0 runs the token-by-token recurrence, chunk = C > 0 the chunkwise form.
    Returns (out [T, H, V], final_state [N, H, V, K]) in float64."""
    q, k, v, log_alpha, beta = map(_f64, (q, k, v, log_alpha, beta))
    T, H, K = q.shape
    V = v.shape[2]
    cu = None
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        N = cu.shape[0] - 1
    init = _f64(initial_state)
    out = np.zeros((T, H, V), dtype=np.float64)
    fs = np.zeros((N, H, V, K), dtype=np.float64)
    if nthreads is None:
        nthreads = min(os.cpu_count() or 1, max(1, N * H))
    rc = _load().kda_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                _ptr(init), _ptr(cu), T, H, N, K, V, float(scale),
                                int(chunk), int(nthreads), _ptr(out), _ptr(fs))
    if rc != 0:
        raise ValueError("kda_oracle_fwd rejected its arguments")
    return out, fs


def fwd_raw(q_raw, k_raw, v, g_raw, beta_raw, scale, lower_bound, initial_state=None,
            cu_seqlens=None, N=1, chunk=0, eps=DEFAULT_EPS, nthreads=None):
    """prepare() followed by fwd(): the whole forward pass from raw inputs."""
    q, k, la, beta = prepare(q_raw, k_raw, g_raw, beta_raw, lower_bound, eps)
    return fwd(q, k, v, la, beta, scale, initial_state, cu_seqlens, N, chunk, nthreads)


def num_chunks(T_total, N=1, cu_seqlens=None, C=16):
    cu = None
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        N = cu.shape[0] - 1
    n = _load().kda_oracle_num_chunks(_ptr(cu), int(T_total), int(N), int(C))
    if n < 0:
        raise ValueError("bad arguments")
    return int(n)


def chunk_factors(q, k, v, log_alpha, beta, scale, cu_seqlens=None, N=1, C=16):
    """Per-chunk factors of the chunkwise form, records indexed [chunk, h].

    Returns a dict of float64 arrays: Akk, Aqk [nc, H, C, C]; W, Qdec, Kend
    [nc, H, C, K]; U [nc, H, C, V]; dlast [nc, H, K]."""
    q, k, v, log_alpha, beta = map(_f64, (q, k, v, log_alpha, beta))
    T, H, K = q.shape
    V = v.shape[2]
    cu = None
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        N = cu.shape[0] - 1
    nc = num_chunks(T, N, cu, C)
    out = {
        "Akk": np.zeros((nc, H, C, C)), "Aqk": np.zeros((nc, H, C, C)),
        "W": np.zeros((nc, H, C, K)), "U": np.zeros((nc, H, C, V)),
        "Qdec": np.zeros((nc, H, C, K)), "Kend": np.zeros((nc, H, C, K)),
        "dlast": np.zeros((nc, H, K)),
    }
    rc = _load().kda_oracle_chunk_factors(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(cu), T, H, N, K, V,
        float(scale), int(C), _ptr(out["Akk"]), _ptr(out["Aqk"]), _ptr(out["W"]),
        _ptr(out["U"]), _ptr(out["Qdec"]), _ptr(out["Kend"]), _ptr(out["dlast"]))
    if rc < 0:
        raise ValueError("kda_oracle_chunk_factors rejected its arguments")
    return out


def _inverse(name, R):
    R = _f64(R)
    n = R.shape[0]
    out = np.zeros_like(R)
    if getattr(_load(), name)(_ptr(R), n, _ptr(out)) != 0:
        raise ValueError(name)
    return out


def neumann_inverse(R):
    """sum_{m<n} (-R)^m for a strictly lower-triangular n x n R."""
    return _inverse("kda_oracle_neumann_inverse", R)


def product_inverse(R):
    """(I - R)(I + R^2)(I + R^4)... grouped form of the same series."""
    return _inverse("kda_oracle_product_inverse", R)


def trisolve_inverse(R):
    """(I + R)^-1 by forward substitution."""
    return _inverse("kda_oracle_trisolve_inverse", R)
