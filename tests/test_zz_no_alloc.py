"""kda_prefill_no_alloc: the prefill for callers that cannot allocate device memory.

Such callers (a serving runtime whose GPU memory all comes from a pool sized at
start-up, or a latency-critical path that must not call cudaMalloc) cannot hand
kda_prefill a workspace; this entry point keeps the workspace in a fixed array
inside libkda instead.  The test calls it through the C ABI twice in a row, on
two different problems, and checks each result against kda_prefill on the same
inputs within the parity tolerances.  It sits in its own file, collected last,
and passes both alone in a fresh process and after the rest of the suite.
"""
import numpy as np
import pytest
import torch

from kda_gated_delta_04_gb300 import kda, synth
from kda_gated_delta_04_gb300.synth import PrefillWorkload
from parity_util import TOL, maxabs, relF, to_device

pytestmark = pytest.mark.gpu

PROBLEMS = [
    PrefillWorkload("no_alloc_varlen", 140, 3, 128, "bf16", (100, 0, 64, 200), 4, init_state=True),
    PrefillWorkload("no_alloc_single", 141, 2, 128, "bf16", (300,), 1),
]


def _buffers(w):
    d = to_device(synth.prefill_inputs(w))
    T, H, D = d["q"].shape
    N = d["cu_seqlens"].numel() - 1
    o = torch.empty((T, H, D), dtype=torch.bfloat16, device="cuda")
    fs = torch.empty((N, H, D, D), dtype=torch.float32, device="cuda")
    return d, o, fs, (N, T, H, D)


def _args(d, o, fs, dims):
    N, T, H, D = dims
    s0 = d["init_state"].data_ptr() if d["init_state"] is not None else None
    return (d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["log_alpha"].data_ptr(),
            d["beta"].data_ptr(), d["cu_seqlens"].data_ptr(), N, T, H, D, D, kda.KDA_DTYPE_BF16,
            s0, o.data_ptr(), fs.data_ptr())


def test_no_alloc_matches_prefill_on_two_calls_in_a_row():
    stream = torch.cuda.current_stream().cuda_stream
    refs, runs = [], []
    for w in PROBLEMS:  # reference results from the workspace entry point
        d, o, fs, dims = _buffers(w)
        ws = kda.workspace_for(dims[0], dims[1], dims[2], dims[3], kda.KDA_DTYPE_BF16, "cuda")
        st = kda.kda_prefill(*_args(d, o, fs, dims), ws.data_ptr(), ws.numel(), stream)
        assert st == kda.KDA_OK
        refs.append((o, fs))
        runs.append((d, dims))
    errors = torch.full((len(PROBLEMS),), 0xFFFF, dtype=torch.int32, device="cuda")
    outs = []
    for i, (d, dims) in enumerate(runs):  # two allocation-free calls back to back
        o = torch.empty_like(refs[i][0])
        fs = torch.empty_like(refs[i][1])
        st = kda.kda_prefill_no_alloc(*_args(d, o, fs, dims), errors[i:].data_ptr(), stream)
        assert st == kda.KDA_OK, kda.status_string(st)
        outs.append((o, fs))
    torch.cuda.synchronize()
    assert errors.tolist() == [0] * len(PROBLEMS)
    for w, (o_ref, fs_ref), (o, fs) in zip(PROBLEMS, refs, outs):
        o_ref, fs_ref = synth.to_f64(o_ref), synth.to_f64(fs_ref)
        o, fs = synth.to_f64(o), synth.to_f64(fs)
        assert maxabs(o, o_ref) <= TOL["bf16"]["o"], w.name
        assert relF(fs, fs_ref) <= TOL["bf16"]["state"], w.name
        assert np.isfinite(o).all() and np.isfinite(fs).all()


def test_no_alloc_reports_device_errors_and_rejects_too_many_sequences():
    stream = torch.cuda.current_stream().cuda_stream
    d, o, fs, dims = _buffers(PROBLEMS[0])
    d["cu_seqlens"] = torch.tensor([0, 100, 50, 164, 364], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = kda.kda_prefill_no_alloc(*_args(d, o, fs, dims), err.data_ptr(), stream)
    assert st == kda.KDA_OK
    torch.cuda.synchronize()
    assert err.item() == 1  # KDA_DEVICE_ERR_SEQLENS
    # the scratch still holds that error; an empty call must report its own (none)
    err.fill_(0xFFFF)
    st = kda.kda_prefill_no_alloc(None, None, None, None, None, d["cu_seqlens"].data_ptr(), 0, 0,
                                  dims[2], dims[3], dims[3], kda.KDA_DTYPE_BF16, None, None,
                                  fs.data_ptr(), err.data_ptr(), stream)
    assert st == kda.KDA_OK
    torch.cuda.synchronize()
    assert err.item() == 0
    too_many = list(_args(d, o, fs, dims))
    too_many[6] = 4097
    assert kda.kda_prefill_no_alloc(*too_many, None, stream) == kda.KDA_ERR_UNSUPPORTED
