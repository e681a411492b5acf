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


def test_decode_256x32_1000_steps_every_unit():
    """The full decode workload, exactly as the benchmark runs it (256 x 32 units, 1000
    in-place steps over a ring of 16 input sets): o of every unit compared element by element
    at every step, and the whole [256, 32, 128, 128] state after step 1000 by relative
    Frobenius.  The oracle's step runs on the host while the GPU's is in flight."""
    w = synth.DECODE_256
    inputs = [synth.decode_inputs(w, s) for s in range(RING)]
    dev = [{k: t.cuda() for k, t in x.items()} for x in inputs]
    ref_in = [{k: synth.to_f64(t) for k, t in x.items()} for x in inputs]
    state = synth.decode_state(w).cuda()
    ref_state = synth.to_f64(synth.decode_state(w))
    unit_o = np.zeros((w.batch, w.num_heads))
    for s in range(w.steps):
        x, r = dev[s % RING], ref_in[s % RING]
        o = kda.decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], state)
        o_ref, _ = oracle.decode_step(r["q"], r["k"], r["v"], r["log_alpha"], r["beta"], ref_state)
        np.maximum(unit_o, np.abs(synth.to_f64(o) - o_ref).max(axis=2), out=unit_o)
    st = synth.to_f64(state)
    assert np.isfinite(st).all()
    es = relF(st, ref_state)
    eo = float(unit_o.max())
    worst = np.unravel_index(np.argmax(unit_o), unit_o.shape)
    print(f"[parity] {w.name}: all {w.batch} x {w.num_heads} units, every step: max|do| {eo:.3e} "
          f"(worst unit b {worst[0]} h {worst[1]}), relF(whole state after {w.steps} steps) {es:.3e}")
    assert eo <= TOL["bf16"]["o"] and es <= TOL["bf16"]["state"]


def test_empty_batch_is_a_no_op():
    st = kda.kda_decode_step(None, None, None, None, None, 0, 2, 64, 64, kda.KDA_DTYPE_F32, None,
                             None, None)
    assert st == kda.KDA_OK


def test_paged_decode_matches_contiguous_decode_and_the_oracle():
    """kda_decode_step_slots on a pool of 7 states x 3 heads, four sequences on slots
    [5, 0, 3, 6], for several steps: bit for bit the contiguous decode of the gathered
    states, within the bar of the oracle, and the slots nobody decodes are untouched."""
    w = DecodeWorkload("decode_paged", 131, 4, 3, 128, "bf16", 6)
    slots_h = [5, 0, 3, 6]
    pool = torch.zeros((7, 3, 128, 128), dtype=torch.float32)
    pool[1] = 1.0  # unused slots must stay as they are
    pool[2] = -2.0
    pool[4] = 3.0
    state0 = synth.decode_state(w)
    pool[slots_h] = state0
    pool_d = pool.cuda()
    slots = torch.tensor(slots_h, dtype=torch.int32, device="cuda")
    contiguous = state0.clone().cuda()
    ref_state = synth.to_f64(state0)
    for s in range(w.steps):
        x = {k: t.cuda() for k, t in synth.decode_inputs(w, s).items()}
        o_paged = kda.decode_step_slots(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], pool_d, slots)
        o_cont = kda.decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], contiguous)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(synth.to_f64(o_paged), synth.to_f64(o_cont))
        r = {k: synth.to_f64(t) for k, t in synth.decode_inputs(w, s).items()}
        o_ref, _ = oracle.decode_step(r["q"], r["k"], r["v"], r["log_alpha"], r["beta"], ref_state)
        assert maxabs(synth.to_f64(o_paged), o_ref) <= TOL["bf16"]["o"]
    np.testing.assert_array_equal(synth.to_f64(pool_d[slots_h].cpu()), synth.to_f64(contiguous.cpu()))
    assert relF(synth.to_f64(pool_d[slots_h].cpu()), ref_state) <= TOL["bf16"]["state"]
    for free, val in ((1, 1.0), (2, -2.0), (4, 3.0)):
        assert bool((pool_d[free] == val).all())


def test_paged_decode_reports_a_bad_slot_and_runs_the_rest():
    w = DecodeWorkload("decode_bad_slot", 132, 3, 2, 64, "f32", 1)
    pool = synth.decode_state(w).cuda()  # slots 0..2
    before = pool.clone()
    x = {k: t.cuda() for k, t in synth.decode_inputs(w, 0).items()}
    slots = torch.tensor([0, 9, 2], dtype=torch.int32, device="cuda")  # 9 is out of range
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    kda.decode_step_slots(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], pool, slots, errors=errors)
    torch.cuda.synchronize()
    assert errors.item() == 16  # KDA_DEVICE_ERR_SLOT
    assert torch.equal(pool[1], before[1])          # slot 1: no sequence decodes it
    assert not torch.equal(pool[0], before[0]) and not torch.equal(pool[2], before[2])



def test_scalar_gate_decode():
    """KDA_FLAG_SCALAR_GATE in decode: log_alpha [B, H]; bit for bit the per-channel call on
    the broadcast gate, and within the bar of the oracle."""
    w = DecodeWorkload("decode_scalar_gate", 133, 3, 4, 128, "bf16", 3)
    st_s = synth.decode_state(w).cuda()
    st_f = st_s.clone()
    ref_state = synth.to_f64(synth.decode_state(w))
    g = torch.Generator().manual_seed(133)
    for s in range(w.steps):
        x = {k: t.cuda() for k, t in synth.decode_inputs(w, s).items()}
        la = (-0.05 * torch.nn.functional.softplus(torch.randn(3, 4, generator=g))).float()
        la_full = la[:, :, None].expand(3, 4, 128).contiguous()
        o_s = kda.decode_step(x["q"], x["k"], x["v"], la.cuda(), x["beta"], st_s)
        o_f = kda.decode_step(x["q"], x["k"], x["v"], la_full.cuda(), x["beta"], st_f)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(synth.to_f64(o_s), synth.to_f64(o_f))
        r = {k: synth.to_f64(t) for k, t in synth.decode_inputs(w, s).items()}
        o_ref, _ = oracle.decode_step(r["q"], r["k"], r["v"], synth.to_f64(la_full), r["beta"], ref_state)
        assert maxabs(synth.to_f64(o_s), o_ref) <= TOL["bf16"]["o"]
    np.testing.assert_array_equal(synth.to_f64(st_s), synth.to_f64(st_f))
    assert relF(synth.to_f64(st_s), ref_state) <= TOL["bf16"]["state"]


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "f32")])
def test_in_kernel_qk_l2_normalisation_decode(d, dtype):
    """KDA_FLAG_QK_L2NORM in decode: raw q, k rows over several steps, within the bar of the
    oracle run on the fp64-normalised rows."""
    w = DecodeWorkload("decode_qk_norm", 134, 3, 4, d, dtype, 4, raw_qk=True)
    state = synth.decode_state(w).cuda()
    ref_state = synth.to_f64(synth.decode_state(w))
    for s in range(w.steps):
        x_h = synth.decode_inputs(w, s)
        x = {k: t.cuda() for k, t in x_h.items()}
        o = kda.decode_step(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], state, qk_l2norm=True)
        torch.cuda.synchronize()
        r = {k: synth.to_f64(t) for k, t in x_h.items()}
        o_ref, _ = oracle.decode_step(oracle.l2_normalize(r["q"]), oracle.l2_normalize(r["k"]), r["v"],
                                      r["log_alpha"], r["beta"], ref_state)
        assert maxabs(synth.to_f64(o), o_ref) <= TOL[dtype]["o"]
    assert relF(synth.to_f64(state), ref_state) <= TOL[dtype]["state"]
