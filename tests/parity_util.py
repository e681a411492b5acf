"""Shared helpers of the GPU parity tests: run libkda and the oracle on the same
seeded inputs and measure the agreed error metrics.

Tolerances (the stated bar): for bf16 q/k/v the outputs must agree to a max-abs
error of 2e-2 and the final state to 1e-3 relative Frobenius over the compared
states; for fp32 inputs both are 1e-5.  The bf16 output of the GPU is widened
exactly before the comparison; the oracle stays in float64.
"""
import numpy as np
import torch

import oracle
from kda_gated_delta_04_gb300 import kda
from kda_gated_delta_04_gb300 import synth

TOL = {"bf16": {"o": 2e-2, "state": 1e-3}, "f32": {"o": 1e-5, "state": 1e-5}}


def relF(a, b):
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def maxabs(a, b):
    return float(np.abs(a - b).max()) if a.size else 0.0


def to_device(inp, device="cuda"):
    out = {}
    for key in ("q", "k", "v", "log_alpha", "beta", "cu_seqlens", "init_state"):
        t = inp.get(key)
        out[key] = None if t is None else t.to(device).contiguous()
    return out


def gpu_prefill(inp, device="cuda", init_state_inplace=False, check_status=True, streamed=None):
    d = to_device(inp, device)
    cu = d["cu_seqlens"]
    fs = d["init_state"] if init_state_inplace else None
    o, fs = kda.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], cu_seqlens=cu,
                        init_state=d["init_state"], final_state=fs, check_status=check_status,
                        streamed=streamed)
    torch.cuda.synchronize()
    return synth.to_f64(o), synth.to_f64(fs)


def oracle_prefill(inp):
    f = {k: synth.to_f64(inp[k]) for k in ("q", "k", "v", "log_alpha", "beta")}
    s0 = None if inp["init_state"] is None else synth.to_f64(inp["init_state"])
    o, fs, _ = oracle.prefill(f["q"], f["k"], f["v"], f["log_alpha"], f["beta"],
                              cu_seqlens=inp["cu_seqlens"].numpy().astype(np.int64),
                              init_state=s0)
    return o, fs


def assert_parity(o_gpu, fs_gpu, o_ref, fs_ref, dtype, label=""):
    tol = TOL[dtype]
    eo, es = maxabs(o_gpu, o_ref), relF(fs_gpu, fs_ref)
    print(f"[parity] {label}: max|do| = {eo:.3e} (tol {tol['o']:.0e}), "
          f"relF(state) = {es:.3e} (tol {tol['state']:.0e})")
    assert np.isfinite(o_gpu).all() and np.isfinite(fs_gpu).all()
    assert eo <= tol["o"], f"{label}: output max-abs error {eo:.3e} > {tol['o']}"
    assert es <= tol["state"], f"{label}: final-state relative error {es:.3e} > {tol['state']}"
    return eo, es
