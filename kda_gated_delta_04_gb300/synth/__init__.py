"""Seeded synthetic inputs for the KDA prefill and decode workloads.

A module of its own: it draws and shapes random numbers (see ``synth.c``) and
knows the workload shapes, but it holds none of the recurrence's arithmetic.
Tests feed the same arrays to the CUDA library and to the fp64 oracle, and the
benchmark uses it to fill device buffers.

Input recipe (every workload, seed 0 unless stated):
  q, k   ~ N(0, 1) per element, then each (token, head) row divided by its L2
           norm over the head dimension, then stored (bf16 or fp32);
  v      ~ N(0, 1), stored (bf16 or fp32);
  log_alpha = -0.05 * softplus(z), z ~ N(0, 1), fp32   (alpha in ~[0.9, 1));
  beta   = sigmoid(z), z ~ N(0, 1), fp32, one per (token, head);
  initial / decode state ~ N(0, 0.02^2) (standard deviation 0.02), fp32;
  varlen lengths uniform integers in [512, 16384].
Every tensor has its own stream, keyed by (seed, workload id, tensor id, step),
and every element is addressable on its own, so a sampled (sequence, head)
unit can be generated without generating the rest.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lib = None
_lock = threading.Lock()

NORMAL, UNIT_ROWS, NEG_SOFTPLUS, SIGMOID = 0, 1, 2, 3
T_Q, T_K, T_V, T_LOG_ALPHA, T_BETA, T_STATE, T_LENGTHS = 1, 2, 3, 4, 5, 6, 7


def build(force: bool = False) -> str:
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
            lib.synth_stream_key.restype = ctypes.c_uint64
            lib.synth_stream_key.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.synth_rows.restype = ctypes.c_int
            lib.synth_rows.argtypes = [ctypes.c_int, ctypes.c_uint64, ctypes.c_int64,
                                       ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p,
                                       ctypes.c_int]
            lib.synth_uniform_ints.restype = None
            lib.synth_uniform_ints.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64,
                                               ctypes.c_int64, ctypes.c_void_p]
            _lib = lib
    return _lib


def stream_key(seed: int, workload_id: int, tensor: int, step: int = 0) -> int:
    stream = (int(workload_id) << 48) | (int(tensor) << 40) | int(step)
    return int(_load().synth_stream_key(int(seed) & 0xFFFFFFFFFFFFFFFF, stream))


def rows(kind: int, key: int, row0: int, row_step: int, nrows: int, D: int, scale: float = 1.0,
         bf16: bool = False):
    """nrows x D values; returns float32 array, or uint16 bf16 bit patterns when bf16."""
    if bf16:
        out = np.empty((nrows, D), dtype=np.uint16)
        rc = _load().synth_rows(kind, key, row0, row_step, nrows, D, scale, None,
                                out.ctypes.data, 0)
    else:
        out = np.empty((nrows, D), dtype=np.float32)
        rc = _load().synth_rows(kind, key, row0, row_step, nrows, D, scale, out.ctypes.data,
                                None, 0)
    if rc != 0:
        raise ValueError("synth_rows: bad row width")
    return out


def uniform_ints(key: int, n: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int64)
    _load().synth_uniform_ints(key, n, lo, hi, out.ctypes.data)
    return out


def bf16_bits_to_tensor(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def to_f64(t) -> np.ndarray:
    """Exact float64 copy of a CPU tensor/array (bf16 and fp32 widen without rounding)."""
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu()
        if t.dtype == torch.bfloat16:
            return t.float().numpy().astype(np.float64)
        return t.numpy().astype(np.float64)
    return np.asarray(t, dtype=np.float64)


# --------------------------------------------------------------------------- workloads
@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    wid: int                 # stream namespace of this workload
    num_heads: int
    d: int                   # d_k == d_v
    dtype: str               # "bf16" or "f32" (q, k, v, o)
    seq_lens: tuple | None   # fixed lengths, or None for drawn varlen lengths
    num_seqs: int
    varlen_range: tuple | None = None
    init_state: bool = False
    raw_qk: bool = False     # q, k as raw N(0, 1) rows (not unit rows), for in-kernel normalisation

    def lengths(self, seed: int = 0) -> np.ndarray:
        if self.seq_lens is not None:
            return np.asarray(self.seq_lens, dtype=np.int64)
        lo, hi = self.varlen_range
        return uniform_ints(stream_key(seed, self.wid, T_LENGTHS), self.num_seqs, lo, hi)


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    wid: int
    batch: int
    num_heads: int
    d: int
    dtype: str
    steps: int
    raw_qk: bool = False     # q, k as raw N(0, 1) rows (not unit rows)


TINY = PrefillWorkload("tiny_f32_T256_H2_d64", 10, 2, 64, "f32", (256,), 1)
PREFILL_4K = PrefillWorkload("prefill_bf16_T4096_H32_d128", 11, 32, 128, "bf16", (4096,), 1)
PREFILL_64K = PrefillWorkload("prefill_bf16_T65536_H32_d128_state", 12, 32, 128, "bf16",
                              (65536,), 1, init_state=True)
VARLEN_16 = PrefillWorkload("varlen16_bf16_T512-16384_H32_d128", 13, 32, 128, "bf16", None, 16,
                            varlen_range=(512, 16384))
DECODE_256 = DecodeWorkload("decode_bf16_B256_H32_d128_1000steps", 14, 256, 32, 128, "bf16", 1000)
PREFILL_WORKLOADS = (TINY, PREFILL_4K, PREFILL_64K, VARLEN_16)


def _qkv_rows(w_dtype, kind, key, row0, row_step, nrows, D):
    if w_dtype == "bf16":
        return bf16_bits_to_tensor(rows(kind, key, row0, row_step, nrows, D, bf16=True))
    return torch.from_numpy(rows(kind, key, row0, row_step, nrows, D))


def prefill_inputs(w: PrefillWorkload, seed: int = 0, heads=None, seqs=None):
    """Inputs of a prefill workload (CPU tensors), optionally restricted to some
    heads and/or sequences (the selected units keep their values in the full
    problem).  Keys: q, k, v [T, Hs, d]; log_alpha [T, Hs, d] f32; beta [T, Hs] f32;
    cu_seqlens int32 [Ns+1]; init_state [Ns, Hs, d, d] f32 or None; heads; seqs."""
    H, D = w.num_heads, w.d
    lens = w.lengths(seed)
    cu_full = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    heads = list(range(H)) if heads is None else [int(h) for h in heads]
    seqs = list(range(len(lens))) if seqs is None else [int(s) for s in seqs]
    sel_lens = lens[seqs]
    T = int(sel_lens.sum())
    Hs = len(heads)
    key = {t: stream_key(seed, w.wid, t) for t in (T_Q, T_K, T_V, T_LOG_ALPHA, T_BETA, T_STATE)}
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    out = {
        "q": torch.empty((T, Hs, D), dtype=tdt), "k": torch.empty((T, Hs, D), dtype=tdt),
        "v": torch.empty((T, Hs, D), dtype=tdt),
        "log_alpha": torch.empty((T, Hs, D), dtype=torch.float32),
        "beta": torch.empty((T, Hs), dtype=torch.float32),
    }
    full_heads = heads == list(range(H))
    all_seqs = seqs == list(range(len(lens)))
    t_out = 0
    # every sequence and head: one contiguous run of global rows (the same values, one call each)
    for s in ([] if (full_heads and all_seqs) else seqs):
        t0, n = int(cu_full[s]), int(lens[s])
        if full_heads:
            # rows t*H + h for t in [t0, t0+n): one contiguous run
            spans = [(slice(None), t0 * H, 1, n * H)]
        else:
            spans = [(j, t0 * H + h, H, n) for j, h in enumerate(heads)]
        for hsel, row0, step, nrows in spans:
            def put(name, val):
                dst = out[name][t_out:t_out + n]
                if hsel == slice(None):
                    dst.copy_(val.reshape(dst.shape))
                else:
                    dst[:, hsel].copy_(val.reshape(dst[:, hsel].shape))
            qk_kind = NORMAL if w.raw_qk else UNIT_ROWS
            put("q", _qkv_rows(w.dtype, qk_kind, key[T_Q], row0, step, nrows, D))
            put("k", _qkv_rows(w.dtype, qk_kind, key[T_K], row0, step, nrows, D))
            put("v", _qkv_rows(w.dtype, NORMAL, key[T_V], row0, step, nrows, D))
            put("log_alpha", torch.from_numpy(
                rows(NEG_SOFTPLUS, key[T_LOG_ALPHA], row0, step, nrows, D, scale=0.05)))
            put("beta", torch.from_numpy(rows(SIGMOID, key[T_BETA], row0, step, nrows, 1)))
        t_out += n
    if full_heads and all_seqs and T > 0:
        qk_kind = NORMAL if w.raw_qk else UNIT_ROWS
        n_rows = T * H
        out["q"].copy_(_qkv_rows(w.dtype, qk_kind, key[T_Q], 0, 1, n_rows, D).reshape(T, H, D))
        out["k"].copy_(_qkv_rows(w.dtype, qk_kind, key[T_K], 0, 1, n_rows, D).reshape(T, H, D))
        out["v"].copy_(_qkv_rows(w.dtype, NORMAL, key[T_V], 0, 1, n_rows, D).reshape(T, H, D))
        out["log_alpha"].copy_(torch.from_numpy(
            rows(NEG_SOFTPLUS, key[T_LOG_ALPHA], 0, 1, n_rows, D, scale=0.05)).reshape(T, H, D))
        out["beta"].copy_(torch.from_numpy(rows(SIGMOID, key[T_BETA], 0, 1, n_rows, 1)).reshape(T, H))
    out["cu_seqlens"] = torch.from_numpy(
        np.concatenate([[0], np.cumsum(sel_lens)]).astype(np.int32))
    if w.init_state and full_heads and all_seqs:  # rows (s * H + h) * D .. in order: one run
        out["init_state"] = torch.from_numpy(
            rows(NORMAL, key[T_STATE], 0, 1, len(seqs) * H * D, D, scale=0.02)).reshape(len(seqs), H, D, D)
    elif w.init_state:
        st = torch.empty((len(seqs), Hs, D, D), dtype=torch.float32)
        for a, s in enumerate(seqs):
            for b, h in enumerate(heads):
                r0 = (s * H + h) * D
                st[a, b].copy_(torch.from_numpy(rows(NORMAL, key[T_STATE], r0, 1, D, D,
                                                     scale=0.02)))
        out["init_state"] = st
    else:
        out["init_state"] = None
    out["heads"], out["seqs"] = heads, seqs
    return out


def decode_state(w: DecodeWorkload, seed: int = 0, batch=None) -> torch.Tensor:
    """Initial decode state [B, H, d, d] fp32 ~ N(0, 0.02^2) (optionally a subset of rows b)."""
    B, H, D = w.batch, w.num_heads, w.d
    key = stream_key(seed, w.wid, T_STATE)
    bs = list(range(B)) if batch is None else [int(b) for b in batch]
    if bs == list(range(B)):
        return torch.from_numpy(rows(NORMAL, key, 0, 1, B * H * D, D, scale=0.02)).view(B, H, D, D)
    st = torch.empty((len(bs), H, D, D), dtype=torch.float32)
    for a, b in enumerate(bs):
        st[a].copy_(torch.from_numpy(rows(NORMAL, key, b * H * D, 1, H * D, D, scale=0.02))
                    .view(H, D, D))
    return st


def decode_inputs(w: DecodeWorkload, step: int, seed: int = 0, batch=None):
    """Per-step decode inputs (CPU tensors): q, k, v [B, H, d]; log_alpha [B, H, d]; beta [B, H]."""
    B, H, D = w.batch, w.num_heads, w.d
    bs = list(range(B)) if batch is None else [int(b) for b in batch]
    key = {t: stream_key(seed, w.wid, t, step + 1) for t in (T_Q, T_K, T_V, T_LOG_ALPHA, T_BETA)}
    contiguous = bs == list(range(B))
    spans = [(slice(None), 0, B * H)] if contiguous else [(a, b * H, H) for a, b in enumerate(bs)]
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    out = {"q": torch.empty((len(bs), H, D), dtype=tdt), "k": torch.empty((len(bs), H, D), dtype=tdt),
           "v": torch.empty((len(bs), H, D), dtype=tdt),
           "log_alpha": torch.empty((len(bs), H, D), dtype=torch.float32),
           "beta": torch.empty((len(bs), H), dtype=torch.float32)}
    for sel, row0, nrows in spans:
        def put(name, val):
            out[name][sel].copy_(val.reshape(out[name][sel].shape))
        qk_kind = NORMAL if w.raw_qk else UNIT_ROWS
        put("q", _qkv_rows(w.dtype, qk_kind, key[T_Q], row0, 1, nrows, D))
        put("k", _qkv_rows(w.dtype, qk_kind, key[T_K], row0, 1, nrows, D))
        put("v", _qkv_rows(w.dtype, NORMAL, key[T_V], row0, 1, nrows, D))
        put("log_alpha", torch.from_numpy(rows(NEG_SOFTPLUS, key[T_LOG_ALPHA], row0, 1, nrows, D,
                                               scale=0.05)))
        put("beta", torch.from_numpy(rows(SIGMOID, key[T_BETA], row0, 1, nrows, 1)))
    return out
