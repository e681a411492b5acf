"""GPU parity of kda_decode_step against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
from kda_gated_delta_04_gb300 import kda, synth
from kda_gated_delta_04_gb300.synth import DecodeWorkload
from parity_util import TOL, maxabs, relF

pytestmark = pytest.mark.gpu

RING = 16  # distinct per-step input sets, cycled (as the benchmark does)


def _run(w, steps, sample_rows, ring=RING):
    """Full batch on the GPU for `steps` steps; oracle on the sampled batch rows.
    Returns the worst output error over all steps and the final-state error."""
    inputs = [synth.decode_inputs(w, s) for s in range(min(ring, steps))]
    dev = [{k: t.cuda() for k, t in x.items()} for x in inputs]
    state = synth.decode_state(w).cuda()
    ref_state = synth.to_f64(synth.decode_state(w, batch=sample_rows))
    ref_in = [{k: synth.to_f64(t[sample_rows]) for k, t in x.items()} for x in inputs]
    worst_o = 0.0
    for s in range(steps):
        x = dev[s % len(dev)]
        o = kda.decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], state)
        r = ref_in[s % len(ref_in)]
        o_ref, _ = oracle.decode_step(r["q"], r["k"], r["v"], r["log_alpha"], r["beta"], ref_state)
        worst_o = max(worst_o, maxabs(synth.to_f64(o[sample_rows]), o_ref))
    torch.cuda.synchronize()
    es = relF(synth.to_f64(state[sample_rows]), ref_state)
    assert torch.isfinite(state).all()
    return worst_o, es


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_small_decode_matches_oracle(d, dtype):
    w = DecodeWorkload(f"decode_small_{dtype}_{d}", 120 + d + (dtype == "f32"), 3, 4, d, dtype, 20)
    eo, es = _run(w, 20, list(range(3)), ring=20)
    print(f"[parity] decode {dtype} d={d}: max|do| {eo:.3e} relF(state) {es:.3e}")
    assert eo <= TOL[dtype]["o"] and es <= TOL[dtype]["state"]


def test_decode_256x32_1000_steps_sampled():
    w = synth.DECODE_256
    eo, es = _run(w, w.steps, [0, 97, 255])
    print(f"[parity] {w.name}: max|do| over 1000 steps {eo:.3e} relF(state) {es:.3e}")
    assert eo <= TOL["bf16"]["o"] and es <= TOL["bf16"]["state"]


def test_empty_batch_is_a_no_op():
    st = kda.kda_decode_step(None, None, None, None, None, 0, 2, 64, 64, kda.KDA_DTYPE_F32, None,
                             None, None)
    assert st == kda.KDA_OK
