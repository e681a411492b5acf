"""Python binding of libkda (ctypes).  Argument marshalling only.

The raw functions ``kda_prefill``, ``kda_decode_step``,
``kda_prefill_workspace_size``, ``kda_read_device_status`` and
``kda_status_string`` are the C entry points of ``include/kda.h`` with the same
names and arguments (pointers as integers).  ``prefill`` and ``decode_step``
take torch CUDA tensors, allocate outputs with torch when none are given, and
call the same entry points.  Every step of the computation runs in libkda's
kernels; there is no fallback: if ``libkda.so`` is missing or the tensors are
not on a CUDA device, these functions raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libkda.so")

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_TIMEOUT, \
    KDA_ERR_DECAY_RANGE, KDA_ERR_VALUE_RANGE = range(7)
KDA_DTYPE_BF16, KDA_DTYPE_F32 = 0, 1
KDA_FLAG_SCALAR_GATE = 1
KDA_FLAG_QK_L2NORM = 2
KDA_FLAG_NO_SEQ_SPLIT = 4
KDA_FLAG_NO_STREAM = 8
KDA_FLAG_STREAM = 16
KDA_PATH_CUDA_CORE, KDA_PATH_FUSED, KDA_PATH_TWO_KERNEL, KDA_PATH_SEQ_SPLIT, KDA_PATH_SEGMENTED, \
    KDA_PATH_STREAMED = range(6)
CHUNK = 64
KDA_STREAM_RING_MIN = 8

_lib = None
_lock = threading.Lock()

_c = ctypes
_VP = _c.c_void_p
_PREFILL_ARGS = [_VP, _VP, _VP, _VP, _VP, _VP, _c.c_int32, _c.c_int64, _c.c_int32, _c.c_int32,
                 _c.c_int32, _c.c_int, _VP, _VP, _VP, _VP, _c.c_size_t, _VP]
_DECODE_ARGS = [_VP, _VP, _VP, _VP, _VP, _c.c_int32, _c.c_int32, _c.c_int32, _c.c_int32, _c.c_int,
                _VP, _VP, _VP]
EXPORTS = {
    "kda_prefill_workspace_size": (_c.c_size_t, [_c.c_int32, _c.c_int64, _c.c_int32, _c.c_int32,
                                                 _c.c_int32, _c.c_int]),
    "kda_prefill_workspace_size_segmented": (_c.c_size_t, [_c.c_int32, _c.c_int64, _c.c_int32, _c.c_int32,
                                                           _c.c_int32, _c.c_int, _c.c_int64]),
    "kda_prefill_workspace_size_streamed": (_c.c_size_t, [_c.c_int32, _c.c_int64, _c.c_int32, _c.c_int32,
                                                          _c.c_int32, _c.c_int, _c.c_int64]),
    "kda_prefill_path": (_c.c_int32, [_c.c_int32, _c.c_int64, _c.c_int32, _c.c_int32, _c.c_int32, _c.c_int,
                                       _c.c_size_t, _c.c_uint32]),
    "kda_prefill": (_c.c_int, _PREFILL_ARGS),
    "kda_decode_step": (_c.c_int, _DECODE_ARGS),
    "kda_read_device_status": (_c.c_int, [_VP, _VP]),
    "kda_status_string": (_c.c_char_p, [_c.c_int]),
    "kda_prefill_no_alloc": (_c.c_int, _PREFILL_ARGS[:15] + [_VP, _VP]),
    "kda_prefill_events": (_c.c_int, _PREFILL_ARGS + [_c.POINTER(_VP), _c.c_int32]),
    "kda_prefill_events_ex": (_c.c_int, _PREFILL_ARGS + [_c.POINTER(_VP), _c.c_int32, _c.c_uint32]),
    "kda_selftest_bounded_wait": (_c.c_int, [_VP, _c.c_uint64, _VP]),
    "kda_prefill_ex": (_c.c_int, _PREFILL_ARGS + [_c.c_uint32]),
    "kda_diag_tensor_phases": (_c.c_int, [_c.c_int32, _c.c_int32, _VP, _VP, _c.POINTER(_c.c_double)]),
    "kda_prefill_host": (_c.c_int, _PREFILL_ARGS + [_c.c_uint32]),
    "kda_prefill_host_buffer_size": (_c.c_size_t, [_VP, _c.c_int32, _c.c_int64, _c.c_int32, _c.c_int32,
                                                   _c.c_int32, _c.c_int]),
    "kda_prefill_host_segments": (_c.c_int32, [_VP, _c.c_int32, _c.c_int64, _VP, _c.c_int32]),
    "kda_decode_step_ex": (_c.c_int, _DECODE_ARGS + [_c.c_uint32]),
    "kda_decode_step_slots": (_c.c_int, [_VP, _VP, _VP, _VP, _VP, _c.c_int32, _c.c_int32, _c.c_int32,
                                         _c.c_int32, _c.c_int, _VP, _c.c_int32, _VP, _VP, _VP, _VP,
                                         _c.c_uint32]),
    "kda_prefill_slots": (_c.c_int, _PREFILL_ARGS[:12] + [_VP, _c.c_int32, _VP, _VP, _VP, _VP,
                                                          _c.c_size_t, _VP, _c.c_uint32]),
}


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def lib():
    """The loaded libkda (ctypes.CDLL).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libkda.so not found at {LIB_PATH}; build it with "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in EXPORTS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


# ------------------------------------------------------------------ raw C entry points
def kda_prefill_workspace_size(num_seqs, total_tokens, num_heads, d_k, d_v, dtype):
    return lib().kda_prefill_workspace_size(num_seqs, total_tokens, num_heads, d_k, d_v, dtype)


def kda_prefill_workspace_size_segmented(num_seqs, total_tokens, num_heads, d_k, d_v, dtype,
                                         segment_chunks):
    return lib().kda_prefill_workspace_size_segmented(num_seqs, total_tokens, num_heads, d_k, d_v,
                                                      dtype, segment_chunks)


def kda_prefill_workspace_size_streamed(num_seqs, total_tokens, num_heads, d_k, d_v, dtype, ring_chunks):
    return lib().kda_prefill_workspace_size_streamed(num_seqs, total_tokens, num_heads, d_k, d_v, dtype,
                                                     ring_chunks)


def kda_prefill_path(num_seqs, total_tokens, num_heads, d_k, d_v, dtype, workspace_bytes, flags=0):
    return lib().kda_prefill_path(num_seqs, total_tokens, num_heads, d_k, d_v, dtype, workspace_bytes, flags)


def kda_prefill(q, k, v, log_alpha, beta, cu_seqlens, num_seqs, total_tokens, num_heads, d_k,
                d_v, dtype, init_state, o, final_state, workspace, workspace_bytes, stream):
    return lib().kda_prefill(q, k, v, log_alpha, beta, cu_seqlens, num_seqs, total_tokens,
                             num_heads, d_k, d_v, dtype, init_state, o, final_state, workspace,
                             workspace_bytes, stream)


def kda_prefill_ex(q, k, v, log_alpha, beta, cu_seqlens, num_seqs, total_tokens, num_heads, d_k,
                   d_v, dtype, init_state, o, final_state, workspace, workspace_bytes, stream, flags):
    return lib().kda_prefill_ex(q, k, v, log_alpha, beta, cu_seqlens, num_seqs, total_tokens,
                                num_heads, d_k, d_v, dtype, init_state, o, final_state, workspace,
                                workspace_bytes, stream, flags)


def kda_decode_step_ex(q, k, v, log_alpha, beta, batch, num_heads, d_k, d_v, dtype, state, o, stream,
                       flags):
    return lib().kda_decode_step_ex(q, k, v, log_alpha, beta, batch, num_heads, d_k, d_v, dtype,
                                    state, o, stream, flags)


def kda_decode_step(q, k, v, log_alpha, beta, batch, num_heads, d_k, d_v, dtype, state, o, stream):
    return lib().kda_decode_step(q, k, v, log_alpha, beta, batch, num_heads, d_k, d_v, dtype,
                                 state, o, stream)


def kda_prefill_no_alloc(q, k, v, log_alpha, beta, cu_seqlens, num_seqs, total_tokens, num_heads,
                         d_k, d_v, dtype, init_state, o, final_state, device_errors, stream):
    """kda_prefill with its workspace in a fixed array inside libkda, for callers that
    cannot allocate device memory at call time (see include/kda.h)."""
    return lib().kda_prefill_no_alloc(q, k, v, log_alpha, beta, cu_seqlens, num_seqs,
                                      total_tokens, num_heads, d_k, d_v, dtype, init_state, o,
                                      final_state, device_errors, stream)


def kda_prefill_events(q, k, v, log_alpha, beta, cu_seqlens, num_seqs, total_tokens, num_heads,
                       d_k, d_v, dtype, init_state, o, final_state, workspace, workspace_bytes,
                       stream, events):
    """kda_prefill that also records four CUDA events (handles as ints) on `stream` around
    its stages: before the schedule kernel, after it, after the chunk-local kernel, after
    the last kernel (see include/kda.h)."""
    arr = (_VP * len(events))(*events)
    return lib().kda_prefill_events(q, k, v, log_alpha, beta, cu_seqlens, num_seqs, total_tokens,
                                    num_heads, d_k, d_v, dtype, init_state, o, final_state,
                                    workspace, workspace_bytes, stream, arr, len(events))


def kda_prefill_events_ex(q, k, v, log_alpha, beta, cu_seqlens, num_seqs, total_tokens, num_heads,
                          d_k, d_v, dtype, init_state, o, final_state, workspace, workspace_bytes,
                          stream, events, flags):
    """kda_prefill_events with option flags (as kda_prefill_ex)."""
    arr = (_VP * len(events))(*events)
    return lib().kda_prefill_events_ex(q, k, v, log_alpha, beta, cu_seqlens, num_seqs, total_tokens,
                                       num_heads, d_k, d_v, dtype, init_state, o, final_state,
                                       workspace, workspace_bytes, stream, arr, len(events), flags)


def kda_decode_step_slots(q, k, v, log_alpha, beta, batch, num_heads, d_k, d_v, dtype, state_pool,
                          num_slots, slots, o, device_errors, stream, flags):
    return lib().kda_decode_step_slots(q, k, v, log_alpha, beta, batch, num_heads, d_k, d_v, dtype,
                                       state_pool, num_slots, slots, o, device_errors, stream, flags)


def kda_prefill_slots(q, k, v, log_alpha, beta, cu_seqlens, num_seqs, total_tokens, num_heads, d_k,
                      d_v, dtype, state_pool, num_slots, init_slots, final_slots, o, workspace,
                      workspace_bytes, stream, flags):
    return lib().kda_prefill_slots(q, k, v, log_alpha, beta, cu_seqlens, num_seqs, total_tokens,
                                   num_heads, d_k, d_v, dtype, state_pool, num_slots, init_slots,
                                   final_slots, o, workspace, workspace_bytes, stream, flags)


def kda_prefill_host(q, k, v, log_alpha, beta, cu_seqlens, num_seqs, total_tokens, num_heads, d_k, d_v,
                     dtype, init_state, o, final_state, device_buffer, device_bytes, stream, flags):
    return lib().kda_prefill_host(q, k, v, log_alpha, beta, cu_seqlens, num_seqs, total_tokens, num_heads,
                                  d_k, d_v, dtype, init_state, o, final_state, device_buffer, device_bytes,
                                  stream, flags)


def kda_prefill_host_buffer_size(cu_seqlens, num_seqs, total_tokens, num_heads, d_k, d_v, dtype):
    return lib().kda_prefill_host_buffer_size(cu_seqlens, num_seqs, total_tokens, num_heads, d_k, d_v, dtype)


def kda_prefill_host_segments(cu_seqlens, num_seqs, total_tokens, bounds, max_bounds):
    return lib().kda_prefill_host_segments(cu_seqlens, num_seqs, total_tokens, bounds, max_bounds)


def kda_diag_tensor_phases(pass_, reps, workspace, stream, tflops):
    return lib().kda_diag_tensor_phases(pass_, reps, workspace, stream, tflops)


def diag_tensor_phases(pass_, reps, workspace, stream=None):
    """Executed TFLOP/s of the chunk kernel's (pass_ = 0), the state kernel's (pass_ = 1) or
    the streamed kernel's walk (pass_ = 2) tensor-core product groups run on their own (see
    include/kda.h)."""
    out = _c.c_double(0.0)
    st = lib().kda_diag_tensor_phases(pass_, reps, _ptr(workspace, "workspace"),
                                      _stream_handle(stream, workspace.device), _c.byref(out))
    if st != KDA_OK:
        raise KdaError(st, "kda_diag_tensor_phases")
    return out.value


def kda_selftest_bounded_wait(workspace, limit_ns, stream):
    """Runs the device-side bounded-wait self-test (see include/kda.h)."""
    return lib().kda_selftest_bounded_wait(workspace, limit_ns, stream)


def kda_read_device_status(workspace, stream):
    return lib().kda_read_device_status(workspace, stream)


def status_string(status: int) -> str:
    return lib().kda_status_string(int(status)).decode()


kda_status_string = status_string


# ------------------------------------------------------------------ torch convenience
def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return KDA_DTYPE_BF16
    if t.dtype == torch.float32:
        return KDA_DTYPE_F32
    raise TypeError(f"q/k/v must be bf16 or fp32, got {t.dtype}")


def _ptr(t, name, dtype=None):
    torch = _torch()
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _flags(log_alpha, qk_l2norm, seq_split=True, streamed=None):
    """Option bits: a log_alpha without a channel axis is the scalar gate; streamed None leaves
    the streamed form to the library, True asks for it (KDA_FLAG_STREAM), False rules it out
    (KDA_FLAG_NO_STREAM)."""
    return ((KDA_FLAG_SCALAR_GATE if log_alpha.dim() == 2 else 0) |
            (KDA_FLAG_QK_L2NORM if qk_l2norm else 0) | (0 if seq_split else KDA_FLAG_NO_SEQ_SPLIT) |
            (0 if streamed is None else (KDA_FLAG_STREAM if streamed else KDA_FLAG_NO_STREAM)))


def _stream_handle(stream, device):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def workspace_for(num_seqs, total_tokens, num_heads, d, dtype_code, device):
    torch = _torch()
    nbytes = kda_prefill_workspace_size(num_seqs, total_tokens, num_heads, d, d, dtype_code)
    # every byte the kernels read is written first in the same call
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def segmented_workspace_for(num_seqs, total_tokens, num_heads, d, dtype_code, device, segment_chunks):
    """A workspace whose per-chunk records cover at most `segment_chunks` packed chunks: the
    two-kernel prefill then runs segment by segment (kda_prefill_workspace_size_segmented)."""
    torch = _torch()
    nbytes = kda_prefill_workspace_size_segmented(num_seqs, total_tokens, num_heads, d, d, dtype_code,
                                                  segment_chunks)
    if nbytes == 0:
        raise KdaError(KDA_ERR_UNSUPPORTED, "kda_prefill_workspace_size_segmented")
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def streamed_workspace_for(num_seqs, total_tokens, num_heads, d, dtype_code, device, ring_chunks):
    """A workspace whose records cover a ring of `ring_chunks` packed chunks: where the call
    streams, the streamed prefill then reuses their slots (kda_prefill_workspace_size_streamed)."""
    torch = _torch()
    nbytes = kda_prefill_workspace_size_streamed(num_seqs, total_tokens, num_heads, d, d, dtype_code, ring_chunks)
    if nbytes == 0:
        raise KdaError(KDA_ERR_UNSUPPORTED, "kda_prefill_workspace_size_streamed")
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def min_workspace_bytes(num_seqs):
    """KDA_PREFILL_MIN_WORKSPACE(num_seqs): the smallest workspace kda_prefill accepts
    (it then runs the single fused kernel for bf16, d = 128)."""
    return 256 + ((num_seqs * 4 + 1 + 255) // 256) * 256


def prefill(q, k, v, log_alpha, beta, cu_seqlens=None, init_state=None, *, o=None,
            final_state=None, workspace=None, stream=None, check_status=False, outputs=True,
            qk_l2norm=False, seq_split=True, streamed=None):
    """KDA prefill over packed sequences.  q, k: [T, H, d]; v: [T, H, d]; log_alpha: [T, H, d]
    fp32; beta: [T, H] fp32; cu_seqlens: int32 [N+1] CUDA tensor or None (one sequence);
    init_state: [N, H, d, d] fp32 or None.  Returns (o, final_state); with outputs=False
    only the final states are computed and o is None.  A log_alpha of shape [T, H] is the
    scalar-gate (Gated DeltaNet) variant: one decay per token-head for every key channel.
    qk_l2norm=True: q and k are raw and the kernels L2-normalise their rows.  seq_split=False
    keeps each sequence's state pass in one piece (KDA_FLAG_NO_SEQ_SPLIT).  streamed: None (the
    default) leaves it to the library whether the chunk work and the state walk share one launch
    (it does so where that is the faster form); True asks for that whenever the launch holds it
    (KDA_FLAG_STREAM); False runs the chunk kernel and the state pass one after the other
    (KDA_FLAG_NO_STREAM)."""
    torch = _torch()
    T, H, d = q.shape
    dt = _dtype_code(q)
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    if o is None and outputs:
        o = torch.empty((T, H, v.shape[2]), dtype=q.dtype, device=q.device)
    if not outputs:
        o = None
    if final_state is None:
        final_state = torch.empty((N, H, d, v.shape[2]), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = workspace_for(N, T, H, d, dt, q.device)
    flags = _flags(log_alpha, qk_l2norm, seq_split, streamed)
    st = kda_prefill_ex(_ptr(q, "q", q.dtype), _ptr(k, "k", q.dtype), _ptr(v, "v", q.dtype),
                     _ptr(log_alpha, "log_alpha", torch.float32), _ptr(beta, "beta", torch.float32),
                     _ptr(cu_seqlens, "cu_seqlens", torch.int32), N, T, H, d, v.shape[2], dt,
                     _ptr(init_state, "init_state", torch.float32),
                     None if o is None else _ptr(o, "o", q.dtype),
                     _ptr(final_state, "final_state", torch.float32), _ptr(workspace, "workspace"),
                     workspace.numel() * workspace.element_size(),
                     _stream_handle(stream, q.device), flags)
    if st != KDA_OK:
        raise KdaError(st, "kda_prefill")
    if check_status:
        st = kda_read_device_status(workspace.data_ptr(), _stream_handle(stream, q.device))
        if st != KDA_OK:
            raise KdaError(st, "kda_prefill (device)")
    return o, final_state


def prefill_slots(q, k, v, log_alpha, beta, cu_seqlens, state_pool, final_slots, init_slots=None, *,
                  o=None, workspace=None, stream=None, check_status=False, outputs=True,
                  qk_l2norm=False, seq_split=True, streamed=None):
    """Prefill into a paged state cache: sequence n starts from state_pool[init_slots[n]]
    (zero when init_slots is None or the entry is -1) and its final state is written to
    state_pool[final_slots[n]].  state_pool [S, H, d, d] fp32; slots int32 CUDA tensors [N].
    Other arguments as prefill.  Returns o (None with outputs=False)."""
    torch = _torch()
    T, H, d = q.shape
    dt = _dtype_code(q)
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    if o is None and outputs:
        o = torch.empty((T, H, v.shape[2]), dtype=q.dtype, device=q.device)
    if not outputs:
        o = None
    if workspace is None:
        workspace = workspace_for(N, T, H, d, dt, q.device)
    flags = _flags(log_alpha, qk_l2norm, seq_split, streamed)
    st = kda_prefill_slots(_ptr(q, "q", q.dtype), _ptr(k, "k", q.dtype), _ptr(v, "v", q.dtype),
                           _ptr(log_alpha, "log_alpha", torch.float32),
                           _ptr(beta, "beta", torch.float32),
                           _ptr(cu_seqlens, "cu_seqlens", torch.int32), N, T, H, d, v.shape[2], dt,
                           _ptr(state_pool, "state_pool", torch.float32), state_pool.shape[0],
                           _ptr(init_slots, "init_slots", torch.int32),
                           _ptr(final_slots, "final_slots", torch.int32),
                           None if o is None else _ptr(o, "o", q.dtype), _ptr(workspace, "workspace"),
                           workspace.numel() * workspace.element_size(),
                           _stream_handle(stream, q.device), flags)
    if st != KDA_OK:
        raise KdaError(st, "kda_prefill_slots")
    if check_status:
        st = kda_read_device_status(workspace.data_ptr(), _stream_handle(stream, q.device))
        if st != KDA_OK:
            raise KdaError(st, "kda_prefill_slots (device)")
    return o


def _hptr(t, name, dtype=None):
    """Address of a contiguous CPU tensor (None passes through)."""
    torch = _torch()
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError(f"{name} must be a CPU tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def prefill_host(q, k, v, log_alpha, beta, cu_seqlens=None, init_state=None, *, o=None, final_state=None,
                 device_buffer=None, device=None, stream=None, outputs=True, qk_l2norm=False, seq_split=True,
                 streamed=None):
    """kda_prefill_host: q, k, v, log_alpha, beta, cu_seqlens (int32), init_state and the outputs
    in host memory (pin them for the copies to overlap with the prefill).  Returns (o, final_state)
    as host tensors, valid once `stream` has been synchronised."""
    torch = _torch()
    T, H, d = q.shape
    dt = _dtype_code(q)
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    device = device or torch.device("cuda", torch.cuda.current_device())
    if o is None and outputs:
        o = torch.empty((T, H, v.shape[2]), dtype=q.dtype).pin_memory()
    if not outputs:
        o = None
    if final_state is None:
        final_state = torch.empty((N, H, d, v.shape[2]), dtype=torch.float32).pin_memory()
    cu = _hptr(cu_seqlens, "cu_seqlens", torch.int32)
    if device_buffer is None:
        nbytes = kda_prefill_host_buffer_size(cu, N, T, H, d, v.shape[2], dt)
        if nbytes == 0:
            raise KdaError(KDA_ERR_INVALID_ARG, "kda_prefill_host_buffer_size")
        device_buffer = torch.empty(nbytes, dtype=torch.uint8, device=device)
    st = kda_prefill_host(_hptr(q, "q", q.dtype), _hptr(k, "k", q.dtype), _hptr(v, "v", q.dtype),
                          _hptr(log_alpha, "log_alpha", torch.float32), _hptr(beta, "beta", torch.float32),
                          cu, N, T, H, d, v.shape[2], dt, _hptr(init_state, "init_state", torch.float32),
                          _hptr(o, "o", q.dtype), _hptr(final_state, "final_state", torch.float32),
                          _ptr(device_buffer, "device_buffer"),
                          device_buffer.numel() * device_buffer.element_size(),
                          _stream_handle(stream, device_buffer.device),
                          _flags(log_alpha, qk_l2norm, seq_split, streamed))
    if st != KDA_OK:
        raise KdaError(st, "kda_prefill_host")
    return o, final_state


def decode_step_slots(q, k, v, log_alpha, beta, state_pool, slots, *, o=None, errors=None,
                      stream=None, qk_l2norm=False):
    """One decode step on a paged state cache: state_pool [S, H, d, d] fp32 (updated in
    place), slots int32 [B] CUDA tensor of distinct slot indices.  Returns o [B, H, d].
    A log_alpha of shape [B, H] is the scalar-gate variant."""
    torch = _torch()
    B, H, d = q.shape
    dt = _dtype_code(q)
    if o is None:
        o = torch.empty((B, H, v.shape[2]), dtype=q.dtype, device=q.device)
    flags = _flags(log_alpha, qk_l2norm)
    st = kda_decode_step_slots(_ptr(q, "q", q.dtype), _ptr(k, "k", q.dtype), _ptr(v, "v", q.dtype),
                               _ptr(log_alpha, "log_alpha", torch.float32),
                               _ptr(beta, "beta", torch.float32), B, H, d, v.shape[2], dt,
                               _ptr(state_pool, "state_pool", torch.float32), state_pool.shape[0],
                               _ptr(slots, "slots", torch.int32), _ptr(o, "o", q.dtype),
                               None if errors is None else _ptr(errors, "errors", torch.int32),
                               _stream_handle(stream, q.device), flags)
    if st != KDA_OK:
        raise KdaError(st, "kda_decode_step_slots")
    return o


def decode_step(q, k, v, log_alpha, beta, state, *, o=None, stream=None, qk_l2norm=False):
    """One decode step; state [B, H, d, d] fp32 is updated in place.  Returns o [B, H, d].
    A log_alpha of shape [B, H] is the scalar-gate variant."""
    torch = _torch()
    B, H, d = q.shape
    dt = _dtype_code(q)
    if o is None:
        o = torch.empty((B, H, v.shape[2]), dtype=q.dtype, device=q.device)
    flags = _flags(log_alpha, qk_l2norm)
    st = kda_decode_step_ex(_ptr(q, "q", q.dtype), _ptr(k, "k", q.dtype), _ptr(v, "v", q.dtype),
                            _ptr(log_alpha, "log_alpha", torch.float32),
                            _ptr(beta, "beta", torch.float32), B, H, d, v.shape[2], dt,
                            _ptr(state, "state", torch.float32), _ptr(o, "o", q.dtype),
                            _stream_handle(stream, q.device), flags)
    if st != KDA_OK:
        raise KdaError(st, "kda_decode_step")
    return o
