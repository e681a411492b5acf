"""fp64 CPU oracle of the Kimi Delta Attention (KDA) recurrence.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
benchmark's CPU-baseline leg may import this package.  The CUDA library never
links, loads or calls it, and it shares no code with the CUDA sources.

The arithmetic lives in ``kda_oracle.c`` (plain C, double precision, token by
token); this module compiles it with gcc on first use and marshals numpy
arrays to it.  Every function here takes and returns float64 numpy arrays; the
callers widen bf16/fp32 inputs to float64 first, so the oracle sees exactly the
values the GPU receives.

Parity status: every part of the recurrence is pinned by closed forms and
invariants in ``tests/test_oracle_pins.py`` (pure decay, exact retrieval,
overwrite, geometric convergence, DeltaNet and Gated DeltaNet reductions,
linearity, column permutation, chunked restatement, an exact-rational worked
example); ``l2_normalize`` by a worked 3-4-5 row, its floor, unit norm and
direction.  The pages print no numeric output for the method, so no value here
is compared with a printed number.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile kda_oracle.c into liboracle.so next to it (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC,
                               "-lm", "-lpthread"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            lib.kda_oracle_prefill.restype = ctypes.c_int
            lib.kda_oracle_prefill.argtypes = [_dp, _dp, _dp, _dp, _dp, _ip, ctypes.c_int64,
                                               ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                               _dp, _dp, _dp, ctypes.c_int]
            lib.kda_oracle_decode_step.restype = ctypes.c_int
            lib.kda_oracle_decode_step.argtypes = [_dp, _dp, _dp, _dp, _dp, ctypes.c_int64,
                                                   ctypes.c_int64, ctypes.c_int64,
                                                   ctypes.c_int64, _dp, _dp, ctypes.c_int]
            _lib = lib
    return _lib


def _f64(a, shape=None):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None and a.shape != tuple(shape):
        raise ValueError(f"expected shape {tuple(shape)}, got {a.shape}")
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def prefill(q, k, v, log_alpha, beta, cu_seqlens=None, init_state=None, want_output=True,
            nthreads: int = 0):
    """Token-by-token KDA over packed sequences.

    q, k, log_alpha: [T, H, dk]; v: [T, H, dv]; beta: [T, H];
    cu_seqlens: [N+1] int offsets into T (None = one sequence of length T);
    init_state: [N, H, dk, dv] or None (= zeros).
    Returns (o [T, H, dv] or None, final_state [N, H, dk, dv], threads_used).
    """
    q = _f64(q)
    T, H, dk = q.shape
    k = _f64(k, (T, H, dk))
    la = _f64(log_alpha, (T, H, dk))
    v = _f64(v)
    if v.shape[:2] != (T, H):
        raise ValueError("v must be [T, H, dv]")
    dv = v.shape[2]
    b = _f64(beta, (T, H))
    if cu_seqlens is None:
        cu = np.array([0, T], dtype=np.int64)
    else:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    N = cu.shape[0] - 1
    if N < 0 or cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must start at 0, end at T and be non-decreasing")
    s0 = None if init_state is None else _f64(init_state, (N, H, dk, dv))
    o = np.zeros((T, H, dv), dtype=np.float64) if want_output else None
    fs = np.zeros((N, H, dk, dv), dtype=np.float64)
    lib = _load()
    used = lib.kda_oracle_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(b),
                                  cu.ctypes.data_as(_ip), N, H, dk, dv, _ptr(s0), _ptr(o),
                                  _ptr(fs), int(nthreads))
    if used < 0:
        raise RuntimeError("oracle prefill failed (allocation or thread creation)")
    return o, fs, used


def l2_normalize(x, eps: float = 1e-12):
    """Rows of x (last axis) divided by max(their Euclidean norm, eps), in float64.

    The q / k normalisation that precedes the recurrence in the layer ("K3 attention,
    three-piece set", KDA engineering notes: short causal convolution, then L2
    normalisation; "From 124M to 2.8T", chapter 3 code: normalisation over the channel
    axis).  The floor eps = 1e-12 is the usual library default; the pages state none.
    """
    x = np.asarray(x, dtype=np.float64)
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / np.maximum(n, eps)


def decode_step(q, k, v, log_alpha, beta, state, nthreads: int = 0):
    """One KDA token for B x H independent units; state [B,H,dk,dv] updated IN PLACE.

    q, k, log_alpha: [B, H, dk]; v: [B, H, dv]; beta: [B, H].
    state must be a C-contiguous float64 array.  Returns (o [B, H, dv], threads_used).
    """
    if not (isinstance(state, np.ndarray) and state.dtype == np.float64
            and state.flags["C_CONTIGUOUS"]):
        raise ValueError("state must be a C-contiguous float64 numpy array (updated in place)")
    B, H, dk, dv = state.shape
    q = _f64(q, (B, H, dk))
    k = _f64(k, (B, H, dk))
    la = _f64(log_alpha, (B, H, dk))
    v = _f64(v, (B, H, dv))
    b = _f64(beta, (B, H))
    o = np.zeros((B, H, dv), dtype=np.float64)
    used = _load().kda_oracle_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(la), _ptr(b), B, H,
                                          dk, dv, _ptr(state), _ptr(o), int(nthreads))
    if used < 0:
        raise RuntimeError("oracle decode step failed")
    return o, used
