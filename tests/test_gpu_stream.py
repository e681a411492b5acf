"""The streamed prefill (chunk work and state walk in one launch) against the oracle and
against the two-kernel form (KDA_FLAG_NO_STREAM) on the same inputs.

streamed=True asks for the streamed kernel (KDA_FLAG_STREAM; every shape here has at most 32
(sequence, head) units and no sequence split, so the launch holds it), streamed=False runs the
chunk kernel and then the state pass; the default call takes the streamed form only where it
is the faster one.
Both are checked element by element against the fp64 oracle; their difference from each
other is printed (it is rounding only: the walk forms its products transposed)."""
import numpy as np
import pytest
import torch

import oracle
from kda_gated_delta_04_gb300 import kda, synth
from kda_gated_delta_04_gb300.synth import PrefillWorkload
from parity_util import TOL, assert_parity, gpu_prefill, maxabs, oracle_prefill, relF, to_device

pytestmark = pytest.mark.gpu

CASES = [
    PrefillWorkload("stream_T1000_H32", 300, 32, 128, "bf16", (1000,), 1),
    PrefillWorkload("stream_two_seqs_H16_32_units", 301, 16, 128, "bf16", (300, 129), 2, init_state=True),
    PrefillWorkload("stream_varlen_edges_H4_state", 302, 4, 128, "bf16", (0, 1, 63, 64, 65, 130), 6,
                    init_state=True),
    PrefillWorkload("stream_T64_H20", 303, 20, 128, "bf16", (64,), 1, init_state=True),
    PrefillWorkload("stream_T4000_H24_state", 304, 24, 128, "bf16", (4000,), 1, init_state=True),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_streamed_and_two_kernel_forms_match_oracle(w):
    inp = synth.prefill_inputs(w)
    o_s, fs_s = gpu_prefill(inp, streamed=True)
    o_t, fs_t = gpu_prefill(inp, streamed=False)
    o_ref, fs_ref = oracle_prefill(inp)
    print(f"[stream] {w.name}: streamed vs two-kernel max|do| = {maxabs(o_s, o_t):.3e}, "
          f"relF(state) = {relF(fs_s, fs_t):.3e}")
    assert_parity(o_s, fs_s, o_ref, fs_ref, w.dtype, w.name + " (streamed)")
    assert_parity(o_t, fs_t, o_ref, fs_ref, w.dtype, w.name + " (two kernels)")


@pytest.mark.parametrize("variant", ["state_only", "scalar_gate", "qk_l2norm"])
def test_streamed_variants(variant):
    """Final states only (no output products), the scalar gate and in-kernel q/k
    normalisation, each through the streamed kernel and the two-kernel form, against the
    oracle."""
    w = PrefillWorkload(f"stream_{variant}", 310, 16, 128, "bf16", (700, 190), 2, init_state=True,
                        raw_qk=variant == "qk_l2norm")
    inp = synth.prefill_inputs(w)
    d = to_device(inp)
    la = d["log_alpha"]
    ref = dict(inp)
    if variant == "scalar_gate":
        g = torch.Generator().manual_seed(311)
        T, H, dk = inp["q"].shape
        la_s = (-0.05 * torch.nn.functional.softplus(torch.randn(T, H, generator=g))).float().contiguous()
        la = la_s.cuda()
        ref["log_alpha"] = la_s[:, :, None].expand(T, H, dk).contiguous()
    if variant == "qk_l2norm":
        ref["q"] = oracle.l2_normalize(synth.to_f64(inp["q"]))
        ref["k"] = oracle.l2_normalize(synth.to_f64(inp["k"]))
    o_ref, fs_ref = oracle_prefill(ref)
    for streamed in (True, False):
        o, fs = kda.prefill(d["q"], d["k"], d["v"], la, d["beta"], cu_seqlens=d["cu_seqlens"],
                            init_state=d["init_state"], check_status=True, outputs=variant != "state_only",
                            qk_l2norm=variant == "qk_l2norm", streamed=streamed)
        torch.cuda.synchronize()
        label = f"{w.name} ({'streamed' if streamed else 'two kernels'})"
        if variant == "state_only":
            assert o is None
            es = relF(synth.to_f64(fs), fs_ref)
            print(f"[parity] {label}: relF(state) = {es:.3e}")
            assert np.isfinite(synth.to_f64(fs)).all() and es <= TOL["bf16"]["state"]
        else:
            assert_parity(synth.to_f64(o), synth.to_f64(fs), o_ref, fs_ref, "bf16", label)


def test_streamed_prefill_into_state_pool():
    """kda_prefill_slots through the streamed kernel: start states from pool slots (one
    sequence from zero), final states into other slots; untouched slots keep their bytes."""
    w = PrefillWorkload("stream_slots", 320, 8, 128, "bf16", (200, 77, 130), 3, init_state=True)
    inp = synth.prefill_inputs(w)
    d = to_device(inp)
    S = 7
    pool = torch.randn((S, 8, 128, 128), generator=torch.Generator().manual_seed(321)).mul_(0.02).cuda()
    init_slots = torch.tensor([4, -1, 0], dtype=torch.int32, device="cuda")
    final_slots = torch.tensor([1, 5, 6], dtype=torch.int32, device="cuda")
    before = pool.clone()
    o = kda.prefill_slots(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], pool, final_slots,
                          init_slots, check_status=True, streamed=True)
    torch.cuda.synchronize()
    s0 = torch.stack([before[4], torch.zeros_like(before[0]), before[0]]).cpu()
    ref_inp = dict(inp)
    ref_inp["init_state"] = s0
    o_ref, fs_ref = oracle_prefill(ref_inp)
    fs = torch.stack([pool[1], pool[5], pool[6]])
    assert_parity(synth.to_f64(o), synth.to_f64(fs), o_ref, fs_ref, "bf16", w.name)
    for s in (0, 2, 3, 4):
        assert torch.equal(pool[s], before[s])


def test_prefill_path_of_the_benchmark_shapes():
    """kda_prefill_path on the device: the single-sequence H = 32 workloads (32 units) stream
    unless KDA_FLAG_NO_STREAM; a 16-sequence pack (512 units) runs the two kernels; four heads
    over 65,536 tokens take the sequence split, and without it the two kernels (too few units
    for the streamed form to be the faster one) unless KDA_FLAG_STREAM asks for it.  The unit
    count from which the default call streams falls with the sequence length: 31 at 64 chunks,
    27 at 256, 24 at 1024."""
    def path(N, T, H, flags=0):
        ws = kda.kda_prefill_workspace_size(N, T, H, 128, 128, kda.KDA_DTYPE_BF16)
        return kda.kda_prefill_path(N, T, H, 128, 128, kda.KDA_DTYPE_BF16, ws, flags)
    assert path(1, 4096, 32) == kda.KDA_PATH_STREAMED
    assert path(1, 65536, 32) == kda.KDA_PATH_STREAMED
    assert path(1, 4096, 32, kda.KDA_FLAG_NO_STREAM) == kda.KDA_PATH_TWO_KERNEL
    assert path(16, 168023, 32) == kda.KDA_PATH_TWO_KERNEL
    assert path(1, 65536, 4) == kda.KDA_PATH_SEQ_SPLIT
    assert path(1, 65536, 4, kda.KDA_FLAG_NO_SEQ_SPLIT) == kda.KDA_PATH_TWO_KERNEL
    assert path(1, 65536, 4, kda.KDA_FLAG_NO_SEQ_SPLIT | kda.KDA_FLAG_STREAM) == kda.KDA_PATH_STREAMED
    assert path(1, 4096, 16) == kda.KDA_PATH_TWO_KERNEL   # 64 chunks: too short for the split as well
    assert path(1, 4096, 4) == kda.KDA_PATH_TWO_KERNEL
    assert path(1, 4096, 30) == kda.KDA_PATH_TWO_KERNEL
    assert path(1, 4096, 31) == kda.KDA_PATH_STREAMED
    assert path(1, 4096, 24, kda.KDA_FLAG_STREAM) == kda.KDA_PATH_STREAMED
    assert path(1, 16384, 26) == kda.KDA_PATH_TWO_KERNEL
    assert path(1, 16384, 27) == kda.KDA_PATH_STREAMED
    assert path(1, 65536, 23) == kda.KDA_PATH_TWO_KERNEL
    assert path(1, 65536, 24) == kda.KDA_PATH_STREAMED
    assert path(2, 8192, 16) == kda.KDA_PATH_STREAMED       # 32 units of 64 chunks on average
    assert path(1, 4096, 40, kda.KDA_FLAG_STREAM) == kda.KDA_PATH_TWO_KERNEL  # 80 walkers: no room


@pytest.mark.parametrize("case", ["decay", "value", "cu_seqlens"])
def test_streamed_errors_are_reported_not_faulted(case):
    """Device-side errors through the streamed kernel (3 sequences x 8 heads = 24 units): a
    decay outside the supported range (found by a worker), a v value outside the fp16 range
    (found by a walker converting its box) and a cu_seqlens that is not a prefix sum (found by
    the schedule kernel; the workers and walkers still agree on the clamped ranges).  Each is
    recorded in the workspace and the call finishes."""
    lens, H = [100, 50, 50], 8
    w = PrefillWorkload(f"stream_err_{case}", 330, H, 128, "bf16", tuple(lens), len(lens))
    inp = synth.prefill_inputs(w)
    if case == "decay":
        inp["log_alpha"] = torch.full_like(inp["log_alpha"], -2.0)
    if case == "value":
        inp["v"][37, 5, 5] = 1.0e5
    d = to_device(inp)
    if case == "cu_seqlens":
        d["cu_seqlens"] = torch.tensor([0, 100, 60, 200], dtype=torch.int32, device="cuda")
    T = sum(lens)
    ws = kda.workspace_for(len(lens), T, H, 128, kda.KDA_DTYPE_BF16, "cuda")
    assert kda.kda_prefill_path(len(lens), T, H, 128, 128, kda.KDA_DTYPE_BF16, ws.numel(),
                                kda.KDA_FLAG_STREAM) == kda.KDA_PATH_STREAMED
    kda.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], workspace=ws, streamed=True)
    st = kda.kda_read_device_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream)
    expected = {"decay": kda.KDA_ERR_DECAY_RANGE, "value": kda.KDA_ERR_VALUE_RANGE,
                "cu_seqlens": kda.KDA_ERR_INVALID_ARG}[case]
    assert st == expected
    assert kda.kda_read_device_status(ws.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0


def test_streamed_results_do_not_depend_on_timing():
    """The walkers and the workers meet only at the records' flags, and every product and
    rounding is fixed by the data, so repeated calls give the same bits whatever the order in
    which CTAs run.  A record read before its stores were complete, or a buffer refilled
    early, would show up as a difference between calls.  The benchmark workload (T = 4096,
    H = 32: 64 walkers beside 240 workers), with the L2 flushed before every other call so
    that the timing varies; the two-kernel form the same way, and the streamed form over a
    ring of 8 chunks' records (whose slots pass between CTAs as the timing allows)."""
    w = synth.PREFILL_4K
    d = to_device(synth.prefill_inputs(w))
    args = (d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], d["init_state"])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    ring = kda.streamed_workspace_for(1, 4096, 32, 128, kda.KDA_DTYPE_BF16, "cuda", 8)
    for form, kw in (("streamed", dict(streamed=True)), ("two kernels", dict(streamed=False)),
                     ("ring of 8 chunks", dict(workspace=ring))):
        o0, s0 = kda.prefill(*args, check_status=True, **kw)
        o0, s0 = o0.clone(), s0.clone()
        for i in range(16):
            if i % 2:
                flush.zero_()
            o, s = kda.prefill(*args, check_status=True, **kw)
            assert torch.equal(o, o0) and torch.equal(s, s0), f"call {i + 1} differs ({form})"


def test_streamed_form_with_few_units_when_asked():
    """KDA_FLAG_STREAM with few (sequence, head) units, where the default call would not stream:
    four heads, then one, over ragged sequences without the sequence split (two walkers per
    unit, the rest of the grid working), against the oracle."""
    for name, seed, H, lens in (("stream_forced_H4", 340, 4, (1000, 300)), ("stream_forced_H1", 341, 1, (777,))):
        w = PrefillWorkload(name, seed, H, 128, "bf16", lens, len(lens), init_state=True)
        inp = synth.prefill_inputs(w)
        d = to_device(inp)
        T = sum(lens)
        flags = kda.KDA_FLAG_STREAM | kda.KDA_FLAG_NO_SEQ_SPLIT
        ws = kda.kda_prefill_workspace_size(len(lens), T, H, 128, 128, kda.KDA_DTYPE_BF16)
        assert kda.kda_prefill_path(len(lens), T, H, 128, 128, kda.KDA_DTYPE_BF16, ws, flags) == kda.KDA_PATH_STREAMED
        o, fs = kda.prefill(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], d["init_state"],
                            check_status=True, seq_split=False, streamed=True)
        o_ref, fs_ref = oracle_prefill(inp)
        assert_parity(synth.to_f64(o), synth.to_f64(fs), o_ref, fs_ref, w.dtype, name)


def test_streamed_over_a_ring_of_records():
    """A bounded workspace (kda_prefill_workspace_size_streamed) on a call that streams: the
    streamed kernel keeps the records of only `ring` packed chunks, each slot written again
    once both walkers of its previous record have copied it in.  o and the final states are
    bit for bit those of the full workspace: the benchmark shape with rings of 8 and 20
    chunks (of 64); ragged sequences with a zero-length one and initial states (asked to
    stream, four heads), also against the oracle; the state-only form; and a state-pool call
    without outputs in which some sequences store no final state, so that their walkers
    leave at once and only release the slots.  With KDA_FLAG_NO_STREAM the same workspace
    runs the two kernels in segments."""
    def ring_ws(N, T, H, ring):
        ws = kda.streamed_workspace_for(N, T, H, 128, kda.KDA_DTYPE_BF16, "cuda", ring)
        assert ws.numel() < kda.kda_prefill_workspace_size(N, T, H, 128, 128, kda.KDA_DTYPE_BF16)
        return ws

    d = to_device(synth.prefill_inputs(synth.PREFILL_4K))
    args = (d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], d["init_state"])
    o_full, fs_full = kda.prefill(*args, check_status=True)
    _, fs_full_so = kda.prefill(*args, check_status=True, outputs=False)
    for ring in (8, 20):
        ws = ring_ws(1, 4096, 32, ring)
        assert kda.kda_prefill_path(1, 4096, 32, 128, 128, kda.KDA_DTYPE_BF16, ws.numel(), 0) == kda.KDA_PATH_STREAMED
        assert kda.kda_prefill_path(1, 4096, 32, 128, 128, kda.KDA_DTYPE_BF16, ws.numel(),
                                    kda.KDA_FLAG_NO_STREAM) == kda.KDA_PATH_SEGMENTED
        o, fs = kda.prefill(*args, workspace=ws, check_status=True)
        assert torch.equal(o, o_full) and torch.equal(fs, fs_full), f"ring {ring}"
        o_none, fs_so = kda.prefill(*args, workspace=ws, check_status=True, outputs=False)
        assert o_none is None and torch.equal(fs_so, fs_full_so), f"ring {ring}, state only"

    lens = (1000, 0, 300, 2000, 64)
    w = PrefillWorkload("stream_ring_ragged_H4", 350, 4, 128, "bf16", lens, len(lens), init_state=True)
    inp = synth.prefill_inputs(w)
    d = to_device(inp)
    args = (d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], d["init_state"])
    T = sum(lens)
    ws = ring_ws(len(lens), T, 4, 8)
    assert kda.kda_prefill_path(len(lens), T, 4, 128, 128, kda.KDA_DTYPE_BF16, ws.numel(),
                                kda.KDA_FLAG_STREAM) == kda.KDA_PATH_STREAMED
    o_full, fs_full = kda.prefill(*args, check_status=True, seq_split=False, streamed=True)
    o, fs = kda.prefill(*args, workspace=ws, check_status=True, seq_split=False, streamed=True)
    assert torch.equal(o, o_full) and torch.equal(fs, fs_full)
    o_ref, fs_ref = oracle_prefill(inp)
    assert_parity(synth.to_f64(o), synth.to_f64(fs), o_ref, fs_ref, w.dtype, w.name + " (ring of 8 chunks)")

    # the pool: sequences 1 and 3 store no final state (their walkers only release slots)
    pool = torch.zeros(len(lens) + 1, 4, 128, 128, dtype=torch.float32, device="cuda")
    final_slots = torch.tensor([0, -1, 2, -1, 4], dtype=torch.int32, device="cuda")
    init_slots = torch.full((len(lens),), -1, dtype=torch.int32, device="cuda")
    pool_full = pool.clone()
    kda.prefill_slots(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], pool_full, final_slots,
                      init_slots, check_status=True, outputs=False, seq_split=False, streamed=True)
    kda.prefill_slots(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], pool, final_slots,
                      init_slots, workspace=ring_ws(len(lens), T, 4, 8), check_status=True, outputs=False,
                      seq_split=False, streamed=True)
    torch.cuda.synchronize()
    assert torch.equal(pool, pool_full)
    assert not pool[0].eq(0).all() and pool[1].eq(0).all() and pool[3].eq(0).all()


def test_streamed_ring_variants():
    """The ring of records with the kernel variants: raw q, k normalised in the kernels (the
    ring's NORM instantiation), with the channel-wise gate and with a scalar gate ([T, H] log
    decay), each bit for bit the same call with the full workspace."""
    w = PrefillWorkload("stream_ring_variants", 360, 16, 128, "bf16", (1500, 700), 2, init_state=True,
                        raw_qk=True)
    inp = synth.prefill_inputs(w)
    d = to_device(inp)
    T, H = sum(w.seq_lens), w.num_heads
    g = torch.Generator().manual_seed(361)
    la_s = (-0.05 * torch.nn.functional.softplus(torch.randn(T, H, generator=g))).float().contiguous().cuda()
    ws = kda.streamed_workspace_for(2, T, H, 128, kda.KDA_DTYPE_BF16, "cuda", 8)
    for name, la in (("qk_l2norm", d["log_alpha"]), ("qk_l2norm_scalar_gate", la_s)):
        args = (d["q"], d["k"], d["v"], la, d["beta"])
        kw = dict(cu_seqlens=d["cu_seqlens"], init_state=d["init_state"], check_status=True, qk_l2norm=True,
                  seq_split=False, streamed=True)
        o_full, fs_full = kda.prefill(*args, **kw)
        o, fs = kda.prefill(*args, workspace=ws, **kw)
        assert torch.equal(o, o_full) and torch.equal(fs, fs_full), name


def test_streamed_ring_at_full_size():
    """T = 65536, H = 32 from initial states with the records of 16 chunks (each slot
    refilled 64 times, the chunk work held to the walk's pace throughout): o and the final
    states bit for bit those of the full workspace."""
    d = to_device(synth.prefill_inputs(synth.PREFILL_64K))
    T, H = d["q"].shape[:2]
    args = (d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], d["init_state"])
    o_full, fs_full = kda.prefill(*args, check_status=True)
    ws = kda.streamed_workspace_for(1, T, H, 128, kda.KDA_DTYPE_BF16, "cuda", 16)
    assert kda.kda_prefill_path(1, T, H, 128, 128, kda.KDA_DTYPE_BF16, ws.numel(), 0) == kda.KDA_PATH_STREAMED
    o, fs = kda.prefill(*args, workspace=ws, check_status=True)
    assert torch.equal(o, o_full) and torch.equal(fs, fs_full)


def test_streamed_ring_across_many_short_sequences():
    """24 short sequences (0 to 300 tokens, some empty) of one head each, asked to stream over a
    ring of 8 chunks: chunk g's slot is then mostly handed over by another sequence's walkers.
    o and the final states (and the final states alone) bit for bit the full workspace."""
    rng = np.random.default_rng(370)
    lens = tuple(int(x) for x in rng.integers(0, 301, size=24))
    lens = (0,) + lens[1:12] + (0,) + lens[13:]
    w = PrefillWorkload("stream_ring_short_seqs", 371, 1, 128, "bf16", lens, len(lens), init_state=True)
    d = to_device(synth.prefill_inputs(w))
    T = sum(lens)
    args = (d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["cu_seqlens"], d["init_state"])
    ws = kda.streamed_workspace_for(len(lens), T, 1, 128, kda.KDA_DTYPE_BF16, "cuda", 8)
    assert kda.kda_prefill_path(len(lens), T, 1, 128, 128, kda.KDA_DTYPE_BF16, ws.numel(),
                                kda.KDA_FLAG_STREAM | kda.KDA_FLAG_NO_SEQ_SPLIT) == kda.KDA_PATH_STREAMED
    for outputs in (True, False):
        kw = dict(check_status=True, seq_split=False, streamed=True, outputs=outputs)
        o_full, fs_full = kda.prefill(*args, **kw)
        o, fs = kda.prefill(*args, workspace=ws, **kw)
        assert torch.equal(fs, fs_full) and (o is None if not outputs else torch.equal(o, o_full)), outputs
