"""GPU parity of kda_prefill against the fp64 oracle (through the C ABI).

Small problems are compared element by element; they span several chunks and
ragged tails.  The full-size workloads run exactly as the benchmark launches
them, and the oracle recomputes every (sequence, head) unit: the whole output
element by element and the whole final-state tensor.
"""
import numpy as np
import pytest
import torch

import oracle
from kda_gated_delta_04_gb300 import kda, synth
from kda_gated_delta_04_gb300.synth import PrefillWorkload
from parity_util import TOL, assert_parity, gpu_prefill, maxabs, oracle_prefill, relF, to_device

pytestmark = pytest.mark.gpu

SMALL = [
    synth.TINY,
    PrefillWorkload("bf16_d128_T200_H3_state", 100, 3, 128, "bf16", (200,), 1, init_state=True),
    PrefillWorkload("bf16_d128_varlen_edges", 101, 2, 128, "bf16", (0, 1, 63, 64, 65, 130), 6),
    PrefillWorkload("f32_d128_T150_H2_state", 102, 2, 128, "f32", (150,), 1, init_state=True),
    PrefillWorkload("bf16_d64_varlen_state", 103, 2, 64, "bf16", (5, 100, 64), 3, init_state=True),
    PrefillWorkload("f32_d64_varlen", 104, 3, 64, "f32", (64, 1, 191), 3),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_problems_match_oracle(w):
    inp = synth.prefill_inputs(w)
    o, fs = gpu_prefill(inp)
    o_ref, fs_ref = oracle_prefill(inp)
    assert_parity(o, fs, o_ref, fs_ref, w.dtype, w.name)


def _whole_tensor_parity(w, group, streamed=None):
    """Run the whole workload on the GPU exactly as the benchmark launches it, then check
    every (sequence, head) unit against the oracle, `group` heads at a time (so host memory
    stays bounded): o element by element (max-abs over the whole output), the final state by
    relative Frobenius over the whole [N, H, d, d] tensor.  Per-unit maxima are printed as
    diagnostics only; the stated bounds gate."""
    full = synth.prefill_inputs(w)
    d = to_device(full)
    o_d, fs_d = kda.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                            cu_seqlens=d["cu_seqlens"], init_state=d["init_state"],
                            check_status=True, streamed=streamed)
    torch.cuda.synchronize()
    o, fs = o_d.cpu(), fs_d.cpu()
    del d, o_d, fs_d
    cu = full["cu_seqlens"].numpy().astype(np.int64)
    N, H = len(cu) - 1, w.num_heads
    unit_o = np.zeros((N, H))
    unit_s = np.zeros((N, H))
    err2 = ref2 = 0.0
    for h0 in range(0, H, group):
        hs = slice(h0, min(H, h0 + group))
        sub = {key: full[key][:, hs].contiguous() for key in ("q", "k", "v", "log_alpha", "beta")}
        sub["cu_seqlens"] = full["cu_seqlens"]
        sub["init_state"] = None if full["init_state"] is None else full["init_state"][:, hs].contiguous()
        o_ref, fs_ref = oracle_prefill(sub)
        diff = np.abs(synth.to_f64(o[:, hs]) - o_ref).max(axis=2)  # [T, heads]
        del o_ref
        for n in range(N):
            if cu[n + 1] > cu[n]:
                unit_o[n, hs] = diff[cu[n]:cu[n + 1]].max(axis=0)
        del diff
        fs_g = synth.to_f64(fs[:, hs])
        assert np.isfinite(fs_g).all()
        e = np.square(fs_g - fs_ref).sum(axis=(2, 3))
        r = np.square(fs_ref).sum(axis=(2, 3))
        unit_s[:, hs] = np.sqrt(e / np.where(r > 0, r, 1.0))
        err2 += float(e.sum())
        ref2 += float(r.sum())
    eo = float(unit_o.max())
    es = float(np.sqrt(err2 / ref2)) if ref2 > 0 else float(np.sqrt(err2))
    wo, ws_ = np.unravel_index(np.argmax(unit_o), unit_o.shape), np.unravel_index(np.argmax(unit_s), unit_s.shape)
    print(f"[parity] {w.name}: all {N} x {H} units; max|do| = {eo:.3e} (tol {TOL[w.dtype]['o']:.0e}, "
          f"worst unit seq {wo[0]} head {wo[1]}), relF(whole final state) = {es:.3e} "
          f"(tol {TOL[w.dtype]['state']:.0e}; worst unit {unit_s.max():.3e} at seq {ws_[0]} head {ws_[1]})")
    assert bool(torch.isfinite(o.float()).all())
    assert eo <= TOL[w.dtype]["o"], f"{w.name}: output max-abs error {eo:.3e}"
    assert es <= TOL[w.dtype]["state"], f"{w.name}: final-state relative error {es:.3e}"


def test_prefill_4k_full_size_every_unit():
    _whole_tensor_parity(synth.PREFILL_4K, group=32)


def test_prefill_4k_two_kernel_form_full_size_every_unit():
    """The same workload with the chunk kernel and the state pass one after the other
    (KDA_FLAG_NO_STREAM): the form of every problem with more (sequence, head) units."""
    _whole_tensor_parity(synth.PREFILL_4K, group=32, streamed=False)


def test_prefill_64k_two_kernel_form_full_size_every_unit():
    _whole_tensor_parity(synth.PREFILL_64K, group=8, streamed=False)


def test_prefill_64k_with_initial_state_full_size_every_unit():
    _whole_tensor_parity(synth.PREFILL_64K, group=8)


def test_varlen16_full_size_every_unit():
    _whole_tensor_parity(synth.VARLEN_16, group=4)


@pytest.mark.parametrize("H", [1, 2], ids=["32_column_slices", "64_column_slices"])
def test_state_pass_slice_widths(H):
    """The state pass takes 32-column value slices while all of them fit in one wave of
    SMs and 64-column slices beyond that: 20 ragged sequences from initial states give
    20 x H x 4 = 80 slices at H = 1 and 160 at H = 2 (a GB300 has 152 SMs).  Every unit
    against the oracle."""
    rng = np.random.default_rng(150 + H)
    lens = tuple(int(x) for x in rng.integers(0, 300, size=20))
    w = PrefillWorkload(f"slices_H{H}", 150 + H, H, 128, "bf16", lens, len(lens), init_state=True)
    inp = synth.prefill_inputs(w)
    o, fs = gpu_prefill(inp)
    o_ref, fs_ref = oracle_prefill(inp)
    assert_parity(o, fs, o_ref, fs_ref, "bf16", w.name)


def _custom(name, wid, lens, H=1, d=128, dtype="bf16", init_state=False, log_alpha=None):
    w = PrefillWorkload(name, wid, H, d, dtype, tuple(lens), len(lens), init_state=init_state)
    inp = synth.prefill_inputs(w)
    if log_alpha is not None:
        inp["log_alpha"] = torch.full_like(inp["log_alpha"], log_alpha)
    return w, inp


def test_strong_decay_near_the_supported_limit():
    # -1.2 per token: a full chunk sums to -76.8, inside the supported range
    w, inp = _custom("strong_decay", 110, [150], H=2, log_alpha=-1.2)
    o, fs = gpu_prefill(inp)
    o_ref, fs_ref = oracle_prefill(inp)
    assert_parity(o, fs, o_ref, fs_ref, "bf16", "strong decay")


def test_no_decay_and_zero_beta():
    w, inp = _custom("no_decay", 111, [130], H=2, log_alpha=0.0, init_state=True)
    inp["beta"][:] = 0.0
    o, fs = gpu_prefill(inp)
    o_ref, fs_ref = oracle_prefill(inp)
    assert_parity(o, fs, o_ref, fs_ref, "bf16", "alpha=1, beta=0")
    # beta = 0 and alpha = 1 leave the initial state untouched
    np.testing.assert_allclose(fs, synth.to_f64(inp["init_state"]), rtol=0, atol=0)


def test_decay_outside_range_is_reported_not_faulted():
    w, inp = _custom("decay_out_of_range", 112, [100], log_alpha=-2.0)
    d = to_device(inp)
    ws = kda.workspace_for(1, 100, 1, 128, kda.KDA_DTYPE_BF16, "cuda")
    kda.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], workspace=ws)
    st = kda.kda_read_device_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == kda.KDA_ERR_DECAY_RANGE
    # the record is cleared by the read
    assert kda.kda_read_device_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0


def test_value_outside_fp16_range_is_reported_not_faulted():
    # the two-kernel path holds v (and the chunk-local products) in fp16
    w, inp = _custom("v_range", 118, [100], H=1)
    inp["v"][37, 0, 5] = 1.0e5
    d = to_device(inp)
    ws = kda.workspace_for(1, 100, 1, 128, kda.KDA_DTYPE_BF16, "cuda")
    kda.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], workspace=ws)
    st = kda.kda_read_device_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == kda.KDA_ERR_VALUE_RANGE


def test_malformed_cu_seqlens_is_reported_not_faulted():
    w, inp = _custom("bad_cu", 113, [100, 50, 50], H=1)
    d = to_device(inp)
    d["cu_seqlens"] = torch.tensor([0, 100, 60, 200], dtype=torch.int32, device="cuda")
    ws = kda.workspace_for(3, 200, 1, 128, kda.KDA_DTYPE_BF16, "cuda")
    kda.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], workspace=ws)
    st = kda.kda_read_device_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == kda.KDA_ERR_INVALID_ARG


def test_final_state_may_alias_initial_state():
    w, inp = _custom("inplace", 114, [90, 200], H=2, init_state=True)
    o1, fs1 = gpu_prefill(inp)
    o2, fs2 = gpu_prefill(inp, init_state_inplace=True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(fs1, fs2)


def test_zero_tokens_keeps_initial_states():
    w, inp = _custom("empty", 115, [0, 0], H=2, init_state=True)
    o, fs = gpu_prefill(inp)
    assert o.size == 0
    np.testing.assert_array_equal(fs, synth.to_f64(inp["init_state"]))


def test_split_prefill_and_decode_continue_the_sequence():
    w, inp = _custom("split", 116, [260], H=2, init_state=True)
    o_all, fs_all = gpu_prefill(inp)
    d = to_device(inp)
    a, b = 130, 255
    sl = lambda t, i, j: t[i:j].contiguous()
    o1, f1 = kda.prefill(sl(d["q"], 0, a), sl(d["k"], 0, a), sl(d["v"], 0, a),
                         sl(d["log_alpha"], 0, a), sl(d["beta"], 0, a), init_state=d["init_state"])
    o2, f2 = kda.prefill(sl(d["q"], a, b), sl(d["k"], a, b), sl(d["v"], a, b),
                         sl(d["log_alpha"], a, b), sl(d["beta"], a, b), init_state=f1)
    state = f2.clone().view(1, 2, 128, 128)
    outs = []
    for t in range(b, 260):
        x = lambda n: d[n][t:t + 1].contiguous()
        outs.append(kda.decode_step(x("q"), x("k"), x("v"), x("log_alpha"), x("beta"), state))
    torch.cuda.synchronize()
    o_split = np.concatenate([synth.to_f64(o1), synth.to_f64(o2)] +
                             [synth.to_f64(x) for x in outs])
    assert np.abs(o_split - o_all).max() < 2e-2
    assert relF(synth.to_f64(state), fs_all) < 1e-3


def test_repeated_runs_are_bitwise_identical():
    w, inp = _custom("determinism", 117, [300, 77], H=3, init_state=True)
    o1, fs1 = gpu_prefill(inp)
    o2, fs2 = gpu_prefill(inp)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(fs1, fs2)


@pytest.mark.parametrize("w", [SMALL[1], SMALL[2], synth.PREFILL_4K], ids=lambda w: w.name)
def test_single_kernel_path_with_minimal_workspace(w):
    """With only KDA_PREFILL_MIN_WORKSPACE bytes the bf16 d=128 prefill runs as one fused
    kernel; it must meet the same bar against the oracle.  The two paths round through
    different factorisations of the chunk update, so they are also compared with each
    other, within the parity bar."""
    heads = None if w.num_heads <= 4 else [0, 17]
    inp = synth.prefill_inputs(w, heads=heads)
    d = to_device(inp)
    N = d["cu_seqlens"].numel() - 1
    ws = torch.empty(kda.min_workspace_bytes(N), dtype=torch.uint8, device="cuda")
    o1, f1 = kda.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"],
                         d["init_state"], workspace=ws, check_status=True)
    o2, f2 = gpu_prefill(inp)  # default (largest) workspace: two-kernel path
    o1, f1 = synth.to_f64(o1), synth.to_f64(f1)
    o_ref, fs_ref = oracle_prefill(inp)
    assert_parity(o1, f1, o_ref, fs_ref, "bf16", w.name + " (single kernel)")
    assert np.abs(o1 - o2).max() < 2e-3 and relF(f1, f2) < 1e-3


def test_stage_events_bracket_the_kernels_and_change_nothing():
    """kda_prefill_events gives the same results as kda_prefill and records its four
    events in order around the stages."""
    w, inp = _custom("events", 119, [300, 77], H=3, init_state=True)
    o_ref, fs_ref = gpu_prefill(inp)
    d = to_device(inp)
    T, H, D = d["q"].shape
    o = torch.empty_like(d["q"])
    fs = torch.empty((2, H, D, D), dtype=torch.float32, device="cuda")
    ws = kda.workspace_for(2, T, H, D, kda.KDA_DTYPE_BF16, "cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    s = torch.cuda.current_stream()
    for e in ev:  # make sure every handle exists before it is passed down
        e.record(s)
    st = kda.kda_prefill_events(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
                                d["log_alpha"].data_ptr(), d["beta"].data_ptr(),
                                d["cu_seqlens"].data_ptr(), 2, T, H, D, D, kda.KDA_DTYPE_BF16,
                                d["init_state"].data_ptr(), o.data_ptr(), fs.data_ptr(),
                                ws.data_ptr(), ws.numel(), s.cuda_stream,
                                [e.cuda_event for e in ev])
    assert st == kda.KDA_OK
    torch.cuda.synchronize()
    np.testing.assert_array_equal(synth.to_f64(o), o_ref)
    np.testing.assert_array_equal(synth.to_f64(fs), fs_ref)
    spans = [ev[i].elapsed_time(ev[i + 1]) for i in range(3)]
    assert all(x >= 0 for x in spans) and spans[1] > 0 and spans[2] > 0
    bad = kda.kda_prefill_events(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
                                 d["log_alpha"].data_ptr(), d["beta"].data_ptr(),
                                 d["cu_seqlens"].data_ptr(), 2, T, H, D, D, kda.KDA_DTYPE_BF16,
                                 None, o.data_ptr(), fs.data_ptr(), ws.data_ptr(), ws.numel(),
                                 s.cuda_stream, [e.cuda_event for e in ev[:3]])
    assert bad == kda.KDA_ERR_INVALID_ARG


def test_bounded_wait_gives_up_and_reports_without_a_fault():
    """The failure path every prefill kernel uses: a wait on a barrier nothing
    completes gives up after its limit (50 ms here), the kernel records
    KDA_ERR_TIMEOUT and returns, and the context keeps working."""
    import time
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    t0 = time.time()
    assert kda.kda_selftest_bounded_wait(ws.data_ptr(), 50_000_000, s) == kda.KDA_OK
    assert kda.kda_read_device_status(ws.data_ptr(), s) == kda.KDA_ERR_TIMEOUT
    assert time.time() - t0 < 10.0
    assert kda.kda_selftest_bounded_wait(ws.data_ptr(), 0, s) == kda.KDA_ERR_INVALID_ARG
    # the context is still usable: a prefill afterwards meets the bar
    w, inp = _custom("after_timeout", 120, [130], H=2, init_state=True)
    o, fs = gpu_prefill(inp)
    o_ref, fs_ref = oracle_prefill(inp)
    assert_parity(o, fs, o_ref, fs_ref, "bf16", "after the timeout self-test")


def test_many_tiny_ragged_sequences():
    """The two-kernel path's schedule with hundreds of sequences, most shorter than one
    chunk, some empty, some spanning a few chunks: every unit is checked against the
    oracle (outputs element by element, states together)."""
    rng = np.random.default_rng(121)
    lens = rng.integers(0, 70, size=300)
    lens[::37] = 0
    lens[5], lens[200] = 190, 129
    w = PrefillWorkload("tiny_ragged", 121, 2, 128, "bf16", tuple(int(x) for x in lens), len(lens),
                        init_state=True)
    inp = synth.prefill_inputs(w)
    o, fs = gpu_prefill(inp)
    o_ref, fs_ref = oracle_prefill(inp)
    assert_parity(o, fs, o_ref, fs_ref, "bf16", "300 tiny ragged sequences")


@pytest.mark.parametrize("case", ["two_kernel", "fused", "fp32"])
def test_state_only_prefill_gives_the_same_final_states(case):
    """o = NULL: only the final states are computed (the two-kernel path also skips the
    output products); they are bit for bit those of the full call."""
    dtype = "f32" if case == "fp32" else "bf16"
    w = PrefillWorkload("state_only_" + case, 122, 2, 128, dtype, (200, 0, 64, 97), 4, init_state=True)
    inp = synth.prefill_inputs(w)
    d = to_device(inp)
    N = 4
    ws = None
    if case == "fused":
        ws = torch.empty(kda.min_workspace_bytes(N), dtype=torch.uint8, device="cuda")
    o_full, fs_full = kda.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"],
                                  d["init_state"], workspace=ws, check_status=True)
    o_none, fs_only = kda.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"],
                                  d["init_state"], workspace=ws, check_status=True, outputs=False)
    torch.cuda.synchronize()
    assert o_none is None
    np.testing.assert_array_equal(synth.to_f64(fs_only), synth.to_f64(fs_full))


def _scalar_gate(inp, seed):
    """Scalar-gate inputs: one log_alpha per token-head ([T, H]) and its broadcast [T, H, d]."""
    g = torch.Generator().manual_seed(seed)
    T, H, d = inp["q"].shape
    la = -0.05 * torch.nn.functional.softplus(torch.randn(T, H, generator=g))
    return la.float().contiguous(), la[:, :, None].expand(T, H, d).float().contiguous()


@pytest.mark.parametrize("case", ["two_kernel", "fp32_d64", "single_kernel"])
def test_scalar_gate_variant(case):
    """KDA_FLAG_SCALAR_GATE (Gated DeltaNet): one decay per token-head.  Within the bar of the
    oracle run on the broadcast gate, and bit for bit the per-channel call on that gate."""
    dtype, d = ("f32", 64) if case == "fp32_d64" else ("bf16", 128)
    w = PrefillWorkload("scalar_gate_" + case, 123, 2, d, dtype, (150, 0, 64, 97), 4, init_state=True)
    inp = synth.prefill_inputs(w)
    la_s, la_full = _scalar_gate(inp, 123)
    d_ = to_device(inp)
    ws = None
    if case == "single_kernel":  # minimal workspace: bf16 d=128 takes the fused tcgen05 kernel
        ws = torch.empty(kda.min_workspace_bytes(4), dtype=torch.uint8, device="cuda")
    o_s, fs_s = kda.prefill(d_["q"], d_["k"], d_["v"], la_s.cuda(), d_["beta"], d_["cu_seqlens"],
                            d_["init_state"], workspace=ws, check_status=True)
    o_f, fs_f = kda.prefill(d_["q"], d_["k"], d_["v"], la_full.cuda(), d_["beta"], d_["cu_seqlens"],
                            d_["init_state"], workspace=ws, check_status=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(synth.to_f64(o_s), synth.to_f64(o_f))
    np.testing.assert_array_equal(synth.to_f64(fs_s), synth.to_f64(fs_f))
    ref = dict(inp)
    ref["log_alpha"] = la_full
    o_ref, fs_ref = oracle_prefill(ref)
    assert_parity(synth.to_f64(o_s), synth.to_f64(fs_s), o_ref, fs_ref, dtype, "scalar gate " + case)


@pytest.mark.parametrize("case", ["two_kernel", "single_kernel", "fp32_d64"])
def test_prefill_into_a_state_pool_then_decode_from_it(case):
    """kda_prefill_slots on a pool of 9 states: sequence 0 continues from its slot in place,
    sequence 1 starts from zero, sequences 2 and 3 move from one slot to another.  The outputs
    and final states are bit for bit those of kda_prefill on the gathered states, slots that no
    sequence writes are untouched, and one decode step on the pool continues every sequence
    within the bar of the oracle."""
    dtype, d = ("f32", 64) if case == "fp32_d64" else ("bf16", 128)
    H = 2
    w = PrefillWorkload("pool_" + case, 124, H, d, dtype, (130, 64, 0, 97), 4, init_state=True)
    inp = synth.prefill_inputs(w)
    init_h, final_h = [3, -1, 5, 7], [3, 2, 6, 0]
    pool = torch.zeros((9, H, d, d), dtype=torch.float32)
    for s in range(9):
        pool[s] = 0.01 * (s + 1)
    for n, s in enumerate(init_h):
        if s >= 0:
            pool[s] = inp["init_state"][n]
    init_dense = inp["init_state"].clone()
    init_dense[1] = 0.0
    pool_before = pool.clone()
    dev = to_device(inp)
    pool_d = pool.cuda()
    ws = None
    if case == "single_kernel":
        ws = torch.empty(kda.min_workspace_bytes(4), dtype=torch.uint8, device="cuda")
    i_slots = torch.tensor(init_h, dtype=torch.int32, device="cuda")
    f_slots = torch.tensor(final_h, dtype=torch.int32, device="cuda")
    o_pool = kda.prefill_slots(dev["q"], dev["k"], dev["v"], dev["log_alpha"], dev["beta"],
                               dev["cu_seqlens"], pool_d, f_slots, i_slots, workspace=ws,
                               check_status=True)
    o_dense, fs_dense = kda.prefill(dev["q"], dev["k"], dev["v"], dev["log_alpha"], dev["beta"],
                                    dev["cu_seqlens"], init_dense.cuda(), workspace=ws, check_status=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(synth.to_f64(o_pool), synth.to_f64(o_dense))
    np.testing.assert_array_equal(synth.to_f64(pool_d[final_h].cpu()), synth.to_f64(fs_dense.cpu()))
    for s in (1, 4, 8):  # read by nobody (slot 5 and 7 are read, not written) or untouched
        assert torch.equal(pool_d[s].cpu(), pool_before[s])
    for s in (5, 7):
        assert torch.equal(pool_d[s].cpu(), pool_before[s])
    # the oracle on the same problem (sequence 1 from zero)
    ref = dict(inp)
    ref["init_state"] = init_dense
    o_ref, fs_ref = oracle_prefill(ref)
    assert_parity(synth.to_f64(o_pool), synth.to_f64(pool_d[final_h].cpu()), o_ref, fs_ref, dtype,
                  "prefill into a pool " + case)
    # decode continues each sequence from its final slot
    g = torch.Generator().manual_seed(125)
    io = torch.float32 if dtype == "f32" else torch.bfloat16
    x = {
        "q": torch.nn.functional.normalize(torch.randn(4, H, d, generator=g), dim=-1).to(io),
        "k": torch.nn.functional.normalize(torch.randn(4, H, d, generator=g), dim=-1).to(io),
        "v": torch.randn(4, H, d, generator=g).to(io),
        "log_alpha": (-0.05 * torch.nn.functional.softplus(torch.randn(4, H, d, generator=g))).float(),
        "beta": torch.sigmoid(torch.randn(4, H, generator=g)).float(),
    }
    o_dec = kda.decode_step_slots(*(x[k].cuda() for k in ("q", "k", "v", "log_alpha", "beta")),
                                  pool_d, f_slots)
    torch.cuda.synchronize()
    r = {k: synth.to_f64(t) for k, t in x.items()}
    od_ref, _ = oracle.decode_step(r["q"], r["k"], r["v"], r["log_alpha"], r["beta"], fs_ref.copy())
    assert maxabs(synth.to_f64(o_dec), od_ref) <= TOL[dtype]["o"]


def test_prefill_into_a_pool_reports_a_bad_slot_and_runs_the_rest():
    """A final slot out of range: KDA_DEVICE_ERR_SLOT is reported (KDA_ERR_INVALID_ARG), that
    sequence's state is written nowhere, and the other sequences are unaffected."""
    w = PrefillWorkload("pool_bad_slot", 126, 2, 128, "bf16", (70, 40), 2)
    inp = synth.prefill_inputs(w)
    dev = to_device(inp)
    pool_d = torch.full((4, 2, 128, 128), 5.0, dtype=torch.float32, device="cuda")
    f_slots = torch.tensor([1, 4], dtype=torch.int32, device="cuda")  # 4 is out of range
    ws = kda.workspace_for(2, 110, 2, 128, kda.KDA_DTYPE_BF16, torch.device("cuda"))
    kda.prefill_slots(dev["q"], dev["k"], dev["v"], dev["log_alpha"], dev["beta"], dev["cu_seqlens"],
                      pool_d, f_slots, workspace=ws)
    st = kda.kda_read_device_status(ws.data_ptr(), kda._stream_handle(None, ws.device))
    assert st == kda.KDA_ERR_INVALID_ARG
    _, fs = kda.prefill(dev["q"], dev["k"], dev["v"], dev["log_alpha"], dev["beta"], dev["cu_seqlens"],
                        check_status=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(synth.to_f64(pool_d[1].cpu()), synth.to_f64(fs[0].cpu()))
    for s in (0, 2, 3):
        assert bool((pool_d[s] == 5.0).all())


@pytest.mark.parametrize("case", ["two_kernel", "single_kernel", "fp32_d64", "bf16_d64"])
def test_in_kernel_qk_l2_normalisation(case):
    """KDA_FLAG_QK_L2NORM: raw N(0, 1) q and k rows (norms near sqrt(d)); the kernels normalise
    them.  Within the bar of the oracle run on the fp64-normalised rows."""
    dtype = "f32" if case == "fp32_d64" else "bf16"
    d = 64 if case in ("fp32_d64", "bf16_d64") else 128
    w = PrefillWorkload("qk_norm_" + case, 127, 2, d, dtype, (150, 0, 64, 97), 4, init_state=True,
                        raw_qk=True)
    inp = synth.prefill_inputs(w)
    dev = to_device(inp)
    ws = None
    if case == "single_kernel":
        ws = torch.empty(kda.min_workspace_bytes(4), dtype=torch.uint8, device="cuda")
    o, fs = kda.prefill(dev["q"], dev["k"], dev["v"], dev["log_alpha"], dev["beta"], dev["cu_seqlens"],
                        dev["init_state"], workspace=ws, check_status=True, qk_l2norm=True)
    torch.cuda.synchronize()
    ref = dict(inp)
    ref["q"] = oracle.l2_normalize(synth.to_f64(inp["q"]))
    ref["k"] = oracle.l2_normalize(synth.to_f64(inp["k"]))
    o_ref, fs_ref = oracle_prefill(ref)
    assert_parity(synth.to_f64(o), synth.to_f64(fs), o_ref, fs_ref, dtype, "q/k L2 norm " + case)


SPLIT_CASES = [  # few (sequence, head) units: the state pass runs in segments
    PrefillWorkload("split_H2_T6000_state", 128, 2, 128, "bf16", (6000,), 1, init_state=True),
    PrefillWorkload("split_H1_varlen_state", 129, 1, 128, "bf16", (10000, 0, 13000, 64, 1), 5,
                    init_state=True),
]


@pytest.mark.parametrize("w", SPLIT_CASES, ids=lambda w: w.name)
def test_sequence_split_state_pass(w):
    """The segmented state pass (transition maps, fp32 chaining, all segments at once) is
    within the bar of the oracle, differs from the unsplit pass only by rounding (so it did
    run), and its state-only and state-pool forms give bit for bit the same final states."""
    inp = synth.prefill_inputs(w)
    d = to_device(inp)
    args = (d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], d["init_state"])
    o_s, fs_s = kda.prefill(*args, check_status=True)
    o_n, fs_n = kda.prefill(*args, check_status=True, seq_split=False)
    _, fs_only = kda.prefill(*args, check_status=True, outputs=False)
    torch.cuda.synchronize()
    o_ref, fs_ref = oracle_prefill(inp)
    assert_parity(synth.to_f64(o_s), synth.to_f64(fs_s), o_ref, fs_ref, "bf16", "split " + w.name)
    assert_parity(synth.to_f64(o_n), synth.to_f64(fs_n), o_ref, fs_ref, "bf16", "unsplit " + w.name)
    # the split did run: the call takes that path, and the outputs differ from the unsplit
    # pass by rounding (the final states may not: with segments of 10 chunks the decay leaves
    # no trace of a start state's rounding by the end of a sequence)
    T = sum(w.seq_lens)
    ws_bytes = kda.kda_prefill_workspace_size(len(w.seq_lens), T, w.num_heads, 128, 128, kda.KDA_DTYPE_BF16)
    assert kda.kda_prefill_path(len(w.seq_lens), T, w.num_heads, 128, 128, kda.KDA_DTYPE_BF16, ws_bytes, 0) == \
        kda.KDA_PATH_SEQ_SPLIT
    assert not np.array_equal(synth.to_f64(o_s), synth.to_f64(o_n))
    np.testing.assert_array_equal(synth.to_f64(fs_only), synth.to_f64(fs_s))
    # the same problem against a state pool: start slots reversed, one sequence from zero
    N, H = len(w.seq_lens), w.num_heads
    pool = torch.zeros((2 * N + 1, H, 128, 128), dtype=torch.float32)
    init_h = [2 * N - n for n in range(N)]
    init_h[0] = -1
    init_dense = inp["init_state"].clone()
    init_dense[0] = 0.0
    for n, s in enumerate(init_h):
        if s >= 0:
            pool[s] = inp["init_state"][n]
    pool_d = pool.cuda()
    final_h = list(range(N))
    o_p = kda.prefill_slots(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], pool_d,
                            torch.tensor(final_h, dtype=torch.int32, device="cuda"),
                            torch.tensor(init_h, dtype=torch.int32, device="cuda"), check_status=True)
    o_d, fs_d = kda.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"],
                            init_dense.cuda(), check_status=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(synth.to_f64(o_p), synth.to_f64(o_d))
    np.testing.assert_array_equal(synth.to_f64(pool_d[final_h].cpu()), synth.to_f64(fs_d.cpu()))


def test_sequence_split_long_context_few_heads_every_unit():
    """T = 65536, H = 4, one sequence (the segmented pass with 5 segments of 205 chunks):
    every head against the oracle, the whole output and the whole final state."""
    w = PrefillWorkload("long_T65536_H4_state", 130, 4, 128, "bf16", (65536,), 1, init_state=True)
    _whole_tensor_parity(w, group=4)


def test_options_together_on_a_split_problem():
    """Scalar gate, in-kernel q/k normalisation, a state pool with a discarded final state
    (slot -1) and the sequence-split pass in one call (H = 2, ragged lengths): the outputs
    are bit for bit those of the same options on a dense call, the discarded sequence's
    slot is untouched, and the stored states are within the bar of the oracle run on the
    broadcast gate and fp64-normalised q, k."""
    H = 2
    w = PrefillWorkload("options_split", 135, H, 128, "bf16", (9000, 5400, 240), 3, init_state=True,
                        raw_qk=True)
    inp = synth.prefill_inputs(w)
    la_s, la_full = _scalar_gate(inp, 135)
    dev = to_device(inp)
    la_d = la_s.cuda()
    pool = torch.full((5, H, 128, 128), 0.25, dtype=torch.float32)
    pool[4] = inp["init_state"][0]
    pool[3] = inp["init_state"][2]
    pool_before = pool.clone()
    pool_d = pool.cuda()
    init_h, final_h = [4, -1, 3], [0, -1, 3]  # sequence 1: from zero, final state discarded
    o_p = kda.prefill_slots(dev["q"], dev["k"], dev["v"], la_d, dev["beta"], dev["cu_seqlens"], pool_d,
                            torch.tensor(final_h, dtype=torch.int32, device="cuda"),
                            torch.tensor(init_h, dtype=torch.int32, device="cuda"), check_status=True,
                            qk_l2norm=True)
    init_dense = inp["init_state"].clone()
    init_dense[1] = 0.0
    o_d, fs_d = kda.prefill(dev["q"], dev["k"], dev["v"], la_d, dev["beta"], dev["cu_seqlens"],
                            init_dense.cuda(), check_status=True, qk_l2norm=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(synth.to_f64(o_p), synth.to_f64(o_d))
    np.testing.assert_array_equal(synth.to_f64(pool_d[0].cpu()), synth.to_f64(fs_d[0].cpu()))
    np.testing.assert_array_equal(synth.to_f64(pool_d[3].cpu()), synth.to_f64(fs_d[2].cpu()))
    for s in (1, 2, 4):
        assert torch.equal(pool_d[s].cpu(), pool_before[s])
    ref = dict(inp)
    ref["log_alpha"] = la_full
    ref["init_state"] = init_dense
    ref["q"] = oracle.l2_normalize(synth.to_f64(inp["q"]))
    ref["k"] = oracle.l2_normalize(synth.to_f64(inp["k"]))
    o_ref, fs_ref = oracle_prefill(ref)
    assert_parity(synth.to_f64(o_p), synth.to_f64(fs_d), o_ref, fs_ref, "bf16", "options together, split")


@pytest.mark.parametrize("scalar,qkn", [(False, False), (True, True)], ids=["plain", "scalar_gate_qk_norm"])
def test_more_items_than_resident_chunk_ctas(scalar, qkn):
    """The chunk kernel keeps two CTAs per SM and each walks several (chunk, head) items:
    8 heads over 3,100 ragged tokens in 7 sequences give 440 items against 304 CTA slots,
    with initial states, and with or without the scalar gate and in-kernel q/k
    normalisation.  Every unit against the oracle."""
    H = 8
    w = PrefillWorkload(f"persistent_{int(scalar)}{int(qkn)}", 160 + 2 * scalar + qkn, H, 128, "bf16",
                        (700, 513, 64, 1, 900, 455, 467), 7, init_state=True, raw_qk=qkn)
    inp = synth.prefill_inputs(w)
    dev = to_device(inp)
    ref = dict(inp)
    la = dev["log_alpha"]
    if scalar:
        la_s, la_full = _scalar_gate(inp, 160)
        la = la_s.cuda()
        ref["log_alpha"] = la_full
    if qkn:
        ref["q"] = oracle.l2_normalize(synth.to_f64(inp["q"]))
        ref["k"] = oracle.l2_normalize(synth.to_f64(inp["k"]))
    o, fs = kda.prefill(dev["q"], dev["k"], dev["v"], la, dev["beta"], dev["cu_seqlens"], dev["init_state"],
                        check_status=True, qk_l2norm=qkn)
    torch.cuda.synchronize()
    o_ref, fs_ref = oracle_prefill(ref)
    assert_parity(synth.to_f64(o), synth.to_f64(fs), o_ref, fs_ref, "bf16", w.name)


@pytest.mark.parametrize("seg_chunks", [1, 3, 17])
def test_bounded_records_run_in_segments(seg_chunks):
    """A workspace whose records cover only `seg_chunks` packed chunks: the chunk and state
    kernels run segment by segment, each sequence cut at a boundary carrying its state in
    the workspace.  Ragged sequences (a zero-length one, one shorter than a chunk, several
    spanning many segments) from initial states, two heads: o and the final states bit for
    bit those of the full workspace in the same two-kernel form (no sequence split, no
    streaming), and within the bar of the oracle; the final state may alias the initial state."""
    w = PrefillWorkload(f"segmented_{seg_chunks}", 170 + seg_chunks, 2, 128, "bf16",
                        (300, 0, 1000, 40, 129, 700), 6, init_state=True)
    inp = synth.prefill_inputs(w)
    d = to_device(inp)
    T, H = inp["q"].shape[:2]
    o_ref_gpu, fs_ref_gpu = kda.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"],
                                        d["init_state"], check_status=True, seq_split=False, streamed=False)
    ws = kda.segmented_workspace_for(6, T, H, 128, kda.KDA_DTYPE_BF16, "cuda", seg_chunks)
    assert ws.numel() < kda.kda_prefill_workspace_size(6, T, H, 128, 128, kda.KDA_DTYPE_BF16)
    o, fs = kda.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], d["init_state"],
                        workspace=ws, check_status=True, streamed=False)
    fs_inplace = d["init_state"].clone()
    o2, _ = kda.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], fs_inplace,
                        final_state=fs_inplace, workspace=ws, check_status=True, streamed=False)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(synth.to_f64(o), synth.to_f64(o_ref_gpu))
    np.testing.assert_array_equal(synth.to_f64(fs), synth.to_f64(fs_ref_gpu))
    np.testing.assert_array_equal(synth.to_f64(o2), synth.to_f64(o_ref_gpu))
    np.testing.assert_array_equal(synth.to_f64(fs_inplace), synth.to_f64(fs_ref_gpu))
    o_ref, fs_ref = oracle_prefill(inp)
    assert_parity(synth.to_f64(o), synth.to_f64(fs), o_ref, fs_ref, "bf16", w.name)


def test_bounded_records_at_full_size():
    """T = 65536, H = 32 from initial states with the records of 128 chunks at a time (8
    segments, 304 MB of records instead of 2.4 GB), in the two-kernel form (KDA_FLAG_NO_STREAM:
    this shape would otherwise stream over a ring of the same records): bit for bit the full
    workspace in the same form."""
    w = synth.PREFILL_64K
    inp = synth.prefill_inputs(w)
    d = to_device(inp)
    T, H = inp["q"].shape[:2]
    o_full, fs_full = kda.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"],
                                  d["init_state"], check_status=True, seq_split=False, streamed=False)
    ws = kda.segmented_workspace_for(1, T, H, 128, kda.KDA_DTYPE_BF16, "cuda", 128)
    o, fs = kda.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], d["init_state"],
                        workspace=ws, check_status=True, streamed=False)
    torch.cuda.synchronize()
    assert torch.equal(o, o_full) and torch.equal(fs, fs_full)


def test_split_prefill_into_a_pool_then_paged_decode():
    """A long prompt with few heads goes through the sequence-split pass straight into a
    state pool; paged decode continues from it within the bar of the oracle."""
    H = 2
    w = PrefillWorkload("handoff_split", 136, H, 128, "bf16", (2500,), 1, init_state=False)
    inp = synth.prefill_inputs(w)
    dev = to_device(inp)
    pool_d = torch.zeros((3, H, 128, 128), dtype=torch.float32, device="cuda")
    f_slots = torch.tensor([2], dtype=torch.int32, device="cuda")
    kda.prefill_slots(dev["q"], dev["k"], dev["v"], dev["log_alpha"], dev["beta"], dev["cu_seqlens"], pool_d,
                      f_slots, check_status=True, outputs=False)
    _, fs_ref = oracle_prefill(inp)
    ref_state = fs_ref.copy()
    dw = synth.DecodeWorkload("handoff_split_decode", 137, 1, H, 128, "bf16", 4)
    for s in range(dw.steps):
        x = synth.decode_inputs(dw, s)
        o = kda.decode_step_slots(*(x[k].cuda() for k in ("q", "k", "v", "log_alpha", "beta")), pool_d, f_slots)
        torch.cuda.synchronize()
        r = {k: synth.to_f64(t) for k, t in x.items()}
        o_ref, _ = oracle.decode_step(r["q"], r["k"], r["v"], r["log_alpha"], r["beta"], ref_state)
        assert maxabs(synth.to_f64(o), o_ref) <= TOL["bf16"]["o"]
    assert relF(synth.to_f64(pool_d[2:3].cpu()), ref_state) <= TOL["bf16"]["state"]


def test_tensor_phase_diagnostic_runs_clean():
    """kda_diag_tensor_phases: both passes finish with a clean status word and a plausible
    executed rate (above zero, below the nominal dense bf16 peak of the GPU with margin)."""
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    for p in (0, 1):
        tf = kda.diag_tensor_phases(p, 50, ws)
        assert 1.0 < tf < 3000.0, (p, tf)


def _pinned(t):
    return None if t is None else t.contiguous().pin_memory()


HOST_CASES = [
    ("bench_shape", synth.PREFILL_4K, True),
    ("varlen_state", PrefillWorkload("host_varlen", 138, 2, 128, "bf16", (700, 0, 2300, 64, 1, 1900), 6,
                                     init_state=True), False),
    ("fp32_d64", PrefillWorkload("host_f32", 139, 2, 64, "f32", (3000, 500), 2, init_state=True), False),
]


@pytest.mark.parametrize("name,w,outputs", HOST_CASES, ids=[c[0] for c in HOST_CASES])
def test_host_buffer_prefill_is_bit_for_bit_kda_prefill(name, w, outputs):
    """kda_prefill_host (pinned host buffers, prompt cut at chunk boundaries into overlapped
    segments) gives bit for bit the o and final states of one kda_prefill, with the sequence
    split off in both (the segments are separate, smaller problems); state-only for varlen."""
    inp = synth.prefill_inputs(w)
    dev = to_device(inp)
    o_d, fs_d = kda.prefill(dev["q"], dev["k"], dev["v"], dev["log_alpha"], dev["beta"], dev["cu_seqlens"],
                            dev["init_state"], check_status=True, seq_split=False)
    host = {k: _pinned(inp[k]) for k in ("q", "k", "v", "log_alpha", "beta", "init_state")}
    buf = torch.empty(kda.kda_prefill_host_buffer_size(inp["cu_seqlens"].data_ptr(), len(w.seq_lens),
                                                       inp["q"].shape[0], w.num_heads, w.d, w.d,
                                                       kda.KDA_DTYPE_BF16 if w.dtype == "bf16" else kda.KDA_DTYPE_F32),
                      dtype=torch.uint8, device="cuda")
    o_h, fs_h = kda.prefill_host(host["q"], host["k"], host["v"], host["log_alpha"], host["beta"],
                                 inp["cu_seqlens"], host["init_state"], device_buffer=buf, seq_split=False,
                                 outputs=outputs)
    torch.cuda.synchronize()
    st = kda.kda_read_device_status(buf.data_ptr(), kda._stream_handle(None, buf.device))
    assert st == kda.KDA_OK
    np.testing.assert_array_equal(synth.to_f64(fs_h), synth.to_f64(fs_d.cpu()))
    if outputs:
        np.testing.assert_array_equal(synth.to_f64(o_h), synth.to_f64(o_d.cpu()))
    else:
        assert o_h is None


def test_maximum_sequence_count():
    """65,535 sequences (the grid limit) of 0, 1 and 2 tokens at H = 1: past the sorted-schedule
    limit, every packed chunk a one- or two-token tail, zero-length sequences in between.  All
    outputs and final states against the oracle."""
    lens = tuple(i % 3 for i in range(65535))
    w = PrefillWorkload("max_seqs", 140, 1, 128, "bf16", lens, len(lens), init_state=True)
    inp = synth.prefill_inputs(w)
    d = to_device(inp)
    o, fs = kda.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], d["init_state"],
                        check_status=True)
    torch.cuda.synchronize()
    o_ref, fs_ref = oracle_prefill(inp)
    assert_parity(synth.to_f64(o), synth.to_f64(fs), o_ref, fs_ref, "bf16", "65,535 sequences")


@pytest.mark.parametrize("seed", range(24))
def test_randomized_problems(seed):
    """Seeded random small problems mixing everything the prefill accepts: 1-3 heads, d = 64 or
    128, bf16 or fp32, 1-6 ragged sequences (zero-length ones included), initial states or
    none, the scalar gate, in-kernel q/k normalisation, state-only calls, the minimal or the
    full workspace, with and without the sequence split.  Each against the oracle."""
    rng = np.random.default_rng(1000 + seed)
    H = int(rng.integers(1, 4))
    d = int(rng.choice([64, 128]))
    dtype = str(rng.choice(["bf16", "f32"]))
    N = int(rng.integers(1, 7))
    lens = tuple(int(x) for x in rng.integers(0, 300, size=N))
    if sum(lens) == 0:
        lens = (1,) + lens[1:]
    scalar, qkn, outputs = bool(rng.integers(2)), bool(rng.integers(2)), bool(rng.integers(2))
    minimal_ws, split = bool(rng.integers(2)), bool(rng.integers(2))
    w = PrefillWorkload(f"random_{seed}", 2000 + seed, H, d, dtype, lens, N, init_state=bool(rng.integers(2)),
                        raw_qk=qkn)
    inp = synth.prefill_inputs(w)
    dev = to_device(inp)
    la = dev["log_alpha"]
    ref = dict(inp)
    if scalar:
        la_s, la_full = _scalar_gate(inp, 3000 + seed)
        la, ref["log_alpha"] = la_s.cuda(), la_full
    if qkn:
        ref["q"] = oracle.l2_normalize(synth.to_f64(inp["q"]))
        ref["k"] = oracle.l2_normalize(synth.to_f64(inp["k"]))
    ws = torch.empty(kda.min_workspace_bytes(N), dtype=torch.uint8, device="cuda") if minimal_ws else None
    o, fs = kda.prefill(dev["q"], dev["k"], dev["v"], la, dev["beta"], dev["cu_seqlens"], dev["init_state"],
                        workspace=ws, check_status=True, outputs=outputs, qk_l2norm=qkn, seq_split=split)
    torch.cuda.synchronize()
    o_ref, fs_ref = oracle_prefill(ref)
    label = f"random {seed}: H={H} d={d} {dtype} lens={lens} scalar={scalar} qkn={qkn} out={outputs} min_ws={minimal_ws}"
    if outputs:
        assert_parity(synth.to_f64(o), synth.to_f64(fs), o_ref, fs_ref, dtype, label)
    else:
        assert o is None
        assert_parity(np.zeros(1), synth.to_f64(fs), np.zeros(1), fs_ref, dtype, label)


def test_concurrent_prefills_on_two_streams_match_sequential_runs():
    """Two prefills of different problems on two streams at once (each with its own workspace)
    give bit for bit what each gives alone: no state is shared between calls."""
    wa = PrefillWorkload("conc_a", 143, 4, 128, "bf16", (900, 130), 2, init_state=True)
    wb = PrefillWorkload("conc_b", 144, 2, 128, "bf16", (2000,), 1)
    da, db = to_device(synth.prefill_inputs(wa)), to_device(synth.prefill_inputs(wb))
    args = lambda d: (d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], d["init_state"])
    oa, fa = kda.prefill(*args(da), check_status=True)
    ob, fb = kda.prefill(*args(db), check_status=True)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(3):
        with torch.cuda.stream(sa):
            ra = kda.prefill(*args(da), stream=sa)
        with torch.cuda.stream(sb):
            rb = kda.prefill(*args(db), stream=sb)
        outs.append((ra, rb))
    torch.cuda.synchronize()
    for (oa2, fa2), (ob2, fb2) in outs:
        assert torch.equal(oa2, oa) and torch.equal(fa2, fa)
        assert torch.equal(ob2, ob) and torch.equal(fb2, fb)


def test_host_buffer_prefill_from_pageable_memory():
    """kda_prefill_host with ordinary (pageable) host tensors: the copies cannot overlap the
    prefill, but the results are the same, bit for bit."""
    w = PrefillWorkload("host_pageable", 145, 2, 128, "bf16", (2500, 300), 2, init_state=True)
    inp = synth.prefill_inputs(w)
    dev = to_device(inp)
    o_d, fs_d = kda.prefill(dev["q"], dev["k"], dev["v"], dev["log_alpha"], dev["beta"], dev["cu_seqlens"],
                            dev["init_state"], check_status=True, seq_split=False)
    o_h = torch.empty_like(inp["v"])
    fs_h = torch.empty_like(inp["init_state"])
    kda.prefill_host(inp["q"], inp["k"], inp["v"], inp["log_alpha"], inp["beta"], inp["cu_seqlens"],
                     inp["init_state"], o=o_h, final_state=fs_h, seq_split=False)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(synth.to_f64(o_h), synth.to_f64(o_d.cpu()))
    np.testing.assert_array_equal(synth.to_f64(fs_h), synth.to_f64(fs_d.cpu()))
