"""Benchmark of libkda on one GB300 (or N replicas under torchrun).

One step is one kda_prefill over the single-sequence prefill workload
(B=1, H=32, T=4096, d_k=d_v=128, bf16 q/k/v, fp32 gates and state): every
chunkwise row of the path (decay prefix, decayed operands, k-k and q-k
matrices, UT solve, WY factors, output, state propagation).  The decode row is
timed in the same run on its own workload (256 sequences x 32 heads, d=128,
1000 in-place steps) and reported under "decode".  The two larger prefill
workloads are timed in the same run, each with its own roofline and oracle
baseline: one sequence of T=65536 tokens from a nonzero initial state under
"long_prefill" (beside it, "bounded_records": the same call in the two-kernel form with a
workspace whose per-chunk records cover 128 chunks at a time, and "streamed_ring": the
streamed call with records for a ring of 16 chunks), and 16 packed sequences of
512..16384 tokens (168,023 in all) under "varlen_prefill".  A long single sequence with few heads (T=65536, H=4),
where the serial state pass would leave most SMs idle, is timed with and
without the sequence-split state pass under "long_context".

value    prefill tokens/s with inputs resident in HBM (CUDA events, L2 flushed
         between timed steps by writing a 256 MiB buffer, flush not timed);
e2e      the same through the C ABI from pinned host buffers (kda_prefill_host):
         host->device copies of the step's inputs, the prefill and the device->host
         copies of o and the final state, all inside the timed region (the library
         overlaps the copies of later segments with the prefill of earlier ones);
roofline HBM-bound, for the dominant (longest) kernel of the prefill: its share
         of the algorithmic bytes / its event-timed duration (four events that
         kda_prefill_events records around the kernels on the launching stream),
         against the measured copy bandwidth in MEASURED_PEAKS.json; the whole
         call against all algorithmic bytes is reported beside it ("path");
cpu_baseline  the fp64 oracle on the host cores (rank 0, N=1 only); the decode,
         long_prefill and varlen_prefill blocks carry their own, each on a
         bounded sample of its workload that the block states.

`--impl reference` times the oracle itself (the only other implementation of
the method here) on the same workload and prints the same line with
"impl": "reference".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s & decode steps/s (H=32,d=128) and % of roofline"
L2_FLUSH_BYTES = 256 << 20
CASE_STEPS = 5  # timed calls of each further prefill workload (2.5 to 10 ms each)
BOUNDED_CHUNKS = 128  # packed chunks per segment of the bounded-records measurement (T=65536: 8 segments)
RING_CHUNKS = 16      # packed chunks whose records the streamed-ring measurement keeps


def _env_rank():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def prefill_algorithmic_bytes(T, H, d, n_seqs, io_bytes, with_init):
    per_token_head = (3 * d * io_bytes) + d * 4 + 4 + d * io_bytes  # q,k,v + log_alpha + beta + o
    state = n_seqs * H * d * d * 4 * (2 if with_init else 1)
    return T * H * per_token_head + state


def prefill_stage_bytes(T, H, d, n_seqs, io_bytes, with_init):
    """Each kernel's share of the algorithmic bytes: the chunk kernel reads q, k, log_alpha
    and beta; the state kernel reads v (and S0), writes o and the final state.  The
    per-chunk records the first hands to the second are not algorithmic bytes."""
    chunk = T * H * (2 * d * io_bytes + d * 4 + 4)
    state = T * H * (2 * d * io_bytes) + n_seqs * H * d * d * 4 * (2 if with_init else 1)
    return {"prefill_chunk_kernel": chunk, "prefill_state_kernel": state}


def prefill_flops(T, H, d, C=64):
    # dense-tile count per token-head: 5 C x C x d products and 3 C x d x d products per chunk
    return T * H * (10 * C * d + 6 * d * d)


def executed_tensor_flops(T, H, d, C=64):
    """Tensor-core FLOPs the two-kernel path executes on one sequence of T tokens: per (chunk,
    head) the chunk kernel's groups (k-k and q-k, W, P2, three-term P, N, Q'') and, per chunk and
    each of the four 32-column value slices, the state kernel's groups (P V, N S, P2 V, Q' S)."""
    chunks = -(-T // C)
    chunk_groups = 2 * (128 * 64 * 128 + 64 * 128 * 64 + 64 * 64 * 64 + 3 * 128 * 64 * 64
                        + 128 * 128 * 64 + 64 * 128 * 64)
    state_groups = 2 * (128 * 32 * 64 + 128 * 32 * 128 + 64 * 32 * 64 + 64 * 32 * 128) * (d // 32)
    return chunks * H * (chunk_groups + state_groups)


PATH_NAMES = {0: "cuda_core", 1: "fused", 2: "two_kernel", 3: "seq_split", 4: "segmented", 5: "streamed"}
PATH_TWO_KERNEL, PATH_STREAMED = 2, 5


def prefill_roofline(T, H, d, N, with_init, call_ms, stage_ms, peaks, traffic_key, path):
    """Roofline object of one prefill workload: the dominant (longest) kernel against its
    share of the algorithmic bytes, and the whole call against all of them.  call_ms: mean
    event time of one kda_prefill; stage_ms: mean event times of the stages kda_prefill_events
    marks (schedule kernel, chunk kernel, state pass; on the streamed path the schedule
    kernel and the streamed kernel, which moves every algorithmic byte, the third stage
    empty).  path: kda_prefill_path of the call."""
    alg_bytes = prefill_algorithmic_bytes(T, H, d, N, 2, with_init)
    achieved = alg_bytes / (call_ms / 1e3) / 1e9
    if path == PATH_STREAMED:
        names = ("prefill_prep_kernel", "prefill_stream_kernel")
        stage_bytes = {"prefill_stream_kernel": alg_bytes}
    else:
        names = ("prefill_prep_kernel", "prefill_chunk_kernel", "prefill_state_kernel")
        stage_bytes = prefill_stage_bytes(T, H, d, N, 2, with_init)
    kernels = {}
    for name, ms in zip(names, stage_ms):
        kb = stage_bytes.get(name)
        kernels[name] = {"ms_per_launch": ms}
        if kb:
            kernels[name].update({"algorithmic_bytes_per_launch": kb,
                                  "achieved_gbs": kb / (ms / 1e3) / 1e9,
                                  "frac": kb / (ms / 1e3) / 1e9 / peaks["hbm_gbs"]})
    dom = max(stage_bytes, key=lambda n: kernels[n]["ms_per_launch"])
    return {"bound": "hbm", "kernel": dom,
            "achieved": kernels[dom]["achieved_gbs"], "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": kernels[dom]["frac"],
            "traffic": profiled_traffic(dom + "_" + traffic_key),
            "peak_source": peaks["source"],
            "algorithmic_bytes_per_launch": stage_bytes[dom],
            "kernel_path": PATH_NAMES.get(path, str(path)),
            "kernels": kernels,
            "path": {"achieved": achieved, "frac": achieved / peaks["hbm_gbs"],
                     "algorithmic_bytes_per_launch": alg_bytes,
                     "algorithmic_flops_per_call": prefill_flops(T, H, d),
                     "tensor_frac_of_bf16_peak": prefill_flops(T, H, d) /
                     (call_ms / 1e3) / 1e12 / peaks["bf16_tflops"]}}


def decode_algorithmic_bytes(B, H, d, io_bytes):
    return B * H * (2 * d * d * 4 + 3 * d * io_bytes + d * 4 + 4 + d * io_bytes)


def source_sha(files):
    """Hash of the kernel sources a profile was taken on (paths relative to the repo)."""
    h = hashlib.sha256()
    for f in sorted(files):
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary (profiles/traffic.json), if it
    was taken on the kernel's current sources; None otherwise."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("source_sha") != source_sha(e.get("sources", [])):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(v, dist=None, device=None):
    """Slowest replica's time: the job's time under weak scaling."""
    if dist is None:
        return v
    import torch
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_step_per_rank, world, steps, total_ms):
    """Whole-job throughput: units all ranks processed / the max-over-ranks time."""
    return units_per_step_per_rank * world * steps / (total_ms / 1e3)


# ----------------------------------------------------------------------------- GPU arm
class _Gpu:
    """Device buffers and the raw C-ABI calls of one replica."""

    def __init__(self, args, rank, local_rank):
        import torch
        from kda_gated_delta_04_gb300 import kda, synth
        self.torch, self.kda, self.synth = torch, kda, synth
        self.dev = torch.device("cuda", local_rank)
        self.stream = torch.cuda.current_stream(self.dev)
        self.sh = self.stream.cuda_stream
        self.seed = args.seed + rank  # each replica runs its own independent units
        self.flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=self.dev)

    def event(self):
        return self.torch.cuda.Event(enable_timing=True)

    # ------------------------------------------------------------------ prefill
    def setup_prefill(self):
        torch, kda = self.torch, self.kda
        self.w = self.synth.PREFILL_4K
        self.inp = self.synth.prefill_inputs(self.w, seed=self.seed)
        self.T, self.H, self.d = self.inp["q"].shape
        self.x = {k: self.inp[k].to(self.dev)
                  for k in ("q", "k", "v", "log_alpha", "beta", "cu_seqlens")}
        self.o = torch.empty((self.T, self.H, self.d), dtype=torch.bfloat16, device=self.dev)
        self.fs = torch.empty((1, self.H, self.d, self.d), dtype=torch.float32, device=self.dev)
        self.ws = kda.workspace_for(1, self.T, self.H, self.d, kda.KDA_DTYPE_BF16, self.dev)

    def prefill_path(self, flags=0):
        return self.kda.kda_prefill_path(1, self.T, self.H, self.d, self.d, self.kda.KDA_DTYPE_BF16,
                                         self.ws.numel(), flags)

    def prefill_call(self, events=None, flags=0):
        """One kda_prefill through the C ABI; with `events` (four CUDA events) the
        kda_prefill_events(_ex) variant, which also marks the stages; with `flags` kda_prefill_ex."""
        kda, x = self.kda, self.x
        args = (x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(), x["log_alpha"].data_ptr(),
                x["beta"].data_ptr(), x["cu_seqlens"].data_ptr(), 1, self.T, self.H, self.d, self.d,
                kda.KDA_DTYPE_BF16, None, self.o.data_ptr(), self.fs.data_ptr(), self.ws.data_ptr(),
                self.ws.numel(), self.sh)
        if events is not None:
            st = kda.kda_prefill_events_ex(*args, events, flags)
        else:
            st = kda.kda_prefill_ex(*args, flags) if flags else kda.kda_prefill(*args)
        if st != kda.KDA_OK:
            raise kda.KdaError(st, "kda_prefill")

    def time_prefill(self, steps, warmup, barrier):
        """Per-step event times (ms), L2 flushed (untimed) before each step.  `whole`: one
        kda_prefill bracketed by two events (the headline; its kernels overlap their launch
        boundaries).  `stages`: the same number of kda_prefill_events calls, whose four events
        on the launching stream split each call into schedule, chunk and state kernel (the
        events between kernels keep them from overlapping, so these sum slightly higher)."""
        torch = self.torch
        for _ in range(warmup):
            self.flush.zero_()
            self.prefill_call()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        outer = [(self.event(), self.event()) for _ in range(steps)]
        for a, b in outer:
            self.flush.zero_()
            a.record(self.stream)
            self.prefill_call()
            b.record(self.stream)
        torch.cuda.synchronize()
        barrier()
        ev = [[self.event() for _ in range(4)] for _ in range(steps)]
        for e in ev:
            for x in e:  # create the handles before they are passed down
                x.record(self.stream)
        torch.cuda.synchronize()
        for e in ev:
            self.flush.zero_()
            self.prefill_call([x.cuda_event for x in e])
        torch.cuda.synchronize()
        st = self.kda.kda_read_device_status(self.ws.data_ptr(), self.sh)
        if st != self.kda.KDA_OK:
            raise self.kda.KdaError(st, "kda_prefill (device status)")
        whole = [a.elapsed_time(b) for a, b in outer]
        stages = [[e[i].elapsed_time(e[i + 1]) for i in range(3)] for e in ev]
        return whole, stages

    def time_prefill_flags(self, steps, warmup, flags):
        """Per-step event times (ms) of kda_prefill_ex with `flags`, L2 flushed before each, and
        the same number of kda_prefill_events_ex calls split into its stages."""
        torch = self.torch
        for _ in range(warmup):
            self.flush.zero_()
            self.prefill_call(flags=flags)
        torch.cuda.synchronize()
        outer = [(self.event(), self.event()) for _ in range(steps)]
        for a, b in outer:
            self.flush.zero_()
            a.record(self.stream)
            self.prefill_call(flags=flags)
            b.record(self.stream)
        torch.cuda.synchronize()
        ev = [[self.event() for _ in range(4)] for _ in range(steps)]
        for e in ev:
            for x in e:  # create the handles before they are passed down
                x.record(self.stream)
        torch.cuda.synchronize()
        for e in ev:
            self.flush.zero_()
            self.prefill_call([x.cuda_event for x in e], flags=flags)
        torch.cuda.synchronize()
        stages = [[e[i].elapsed_time(e[i + 1]) for i in range(3)] for e in ev]
        return [a.elapsed_time(b) for a, b in outer], stages

    def time_prefill_e2e(self, steps, warmup):
        """Host-to-host through kda_prefill_host: pinned inputs in, o and the final state out,
        the copies of later segments overlapped with the prefill of earlier ones."""
        torch, kda = self.torch, self.kda
        pin = {k: self.inp[k].pin_memory() for k in ("q", "k", "v", "log_alpha", "beta")}
        cu_host = self.inp["cu_seqlens"].contiguous()
        o_host = torch.empty(self.o.shape, dtype=self.o.dtype).pin_memory()
        fs_host = torch.empty(self.fs.shape, dtype=self.fs.dtype).pin_memory()
        self.h2d = sum(t.numel() * t.element_size() for t in pin.values())
        self.d2h = (o_host.numel() * o_host.element_size() +
                    fs_host.numel() * fs_host.element_size())
        nbytes = kda.kda_prefill_host_buffer_size(cu_host.data_ptr(), 1, self.T, self.H, self.d, self.d,
                                                  kda.KDA_DTYPE_BF16)
        dbuf = torch.empty(nbytes, dtype=torch.uint8, device=self.dev)
        bounds = torch.zeros(64, dtype=torch.int64)  # kept alive across the call that fills it
        nseg = kda.kda_prefill_host_segments(cu_host.data_ptr(), 1, self.T, bounds.data_ptr(), 64)
        if nseg < 1:
            raise kda.KdaError(kda.KDA_ERR_INVALID_ARG, "kda_prefill_host_segments")
        # per segment: the schedule kernel, the streamed kernel (or the chunk kernel and the
        # state pass) and the error word
        seg_path = kda.kda_prefill_path(1, max(1, self.T // nseg), self.H, self.d, self.d, kda.KDA_DTYPE_BF16,
                                        kda.kda_prefill_workspace_size(1, max(1, self.T // nseg), self.H,
                                                                       self.d, self.d, kda.KDA_DTYPE_BF16), 0)
        self.e2e_launches = (3 if seg_path == PATH_STREAMED else 4) * nseg

        def step():
            st = kda.kda_prefill_host(pin["q"].data_ptr(), pin["k"].data_ptr(), pin["v"].data_ptr(),
                                      pin["log_alpha"].data_ptr(), pin["beta"].data_ptr(), cu_host.data_ptr(),
                                      1, self.T, self.H, self.d, self.d, kda.KDA_DTYPE_BF16, None,
                                      o_host.data_ptr(), fs_host.data_ptr(), dbuf.data_ptr(), nbytes, self.sh, 0)
            if st != kda.KDA_OK:
                raise kda.KdaError(st, "kda_prefill_host")

        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        out = []
        for _ in range(steps):
            self.flush.zero_()
            a, b = self.event(), self.event()
            a.record(self.stream)
            step()
            b.record(self.stream)
            b.synchronize()
            out.append(a.elapsed_time(b))
        return out

    # ------------------------------------------------------------------ decode
    # ------------------------------------------------------------------ long context
    def setup_long(self):
        torch, kda, synth = self.torch, self.kda, self.synth
        self.lw = lw = synth.PrefillWorkload("prefill_bf16_T65536_H4_d128_state", 15, 4, 128, "bf16",
                                             (65536,), 1, init_state=True)
        inp = synth.prefill_inputs(lw, seed=self.seed)
        self.lx = {k: inp[k].to(self.dev)
                   for k in ("q", "k", "v", "log_alpha", "beta", "cu_seqlens", "init_state")}
        T, H, d = inp["q"].shape
        self.lo = torch.empty((T, H, d), dtype=torch.bfloat16, device=self.dev)
        self.lfs = torch.empty((1, H, d, d), dtype=torch.float32, device=self.dev)
        self.lws = kda.workspace_for(1, T, H, d, kda.KDA_DTYPE_BF16, self.dev)

    def long_call(self, split):
        kda, x = self.kda, self.lx
        T, H, d = x["q"].shape
        st = kda.kda_prefill_ex(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(),
                                x["log_alpha"].data_ptr(), x["beta"].data_ptr(),
                                x["cu_seqlens"].data_ptr(), 1, T, H, d, d, kda.KDA_DTYPE_BF16,
                                x["init_state"].data_ptr(), self.lo.data_ptr(), self.lfs.data_ptr(),
                                self.lws.data_ptr(), self.lws.numel(), self.sh,
                                0 if split else kda.KDA_FLAG_NO_SEQ_SPLIT)
        if st != kda.KDA_OK:
            raise kda.KdaError(st, "kda_prefill_ex")

    def time_long(self, steps, warmup):
        """Event time (ms per call) of the long-context prefill, split and unsplit (its 470 MB
        of inputs exceed L2, so no flush is needed)."""
        torch, out = self.torch, {}
        for split in (True, False):
            for _ in range(warmup):
                self.long_call(split)
            torch.cuda.synchronize()
            a, b = self.event(), self.event()
            a.record(self.stream)
            for _ in range(steps):
                self.long_call(split)
            b.record(self.stream)
            torch.cuda.synchronize()
            out[split] = a.elapsed_time(b) / steps
        st = self.kda.kda_read_device_status(self.lws.data_ptr(), self.sh)
        if st != self.kda.KDA_OK:
            raise self.kda.KdaError(st, "kda_prefill_ex (device status)")
        return out

    # ------------------------------------------------------------------ more prefill workloads
    def setup_case(self, w):
        """Device buffers of one more prefill workload (the long single sequence with an
        initial state, or the 16-sequence varlen pack)."""
        torch, kda = self.torch, self.kda
        inp = self.synth.prefill_inputs(w, seed=self.seed)
        x = {k: (None if inp[k] is None else inp[k].to(self.dev))
             for k in ("q", "k", "v", "log_alpha", "beta", "cu_seqlens", "init_state")}
        T, H, d = inp["q"].shape
        N = inp["cu_seqlens"].numel() - 1
        c = {"w": w, "inp": inp, "x": x, "T": T, "H": H, "d": d, "N": N,
             "o": torch.empty((T, H, d), dtype=torch.bfloat16, device=self.dev),
             "fs": torch.empty((N, H, d, d), dtype=torch.float32, device=self.dev),
             "ws": kda.workspace_for(N, T, H, d, kda.KDA_DTYPE_BF16, self.dev)}
        c["path"] = kda.kda_prefill_path(N, T, H, d, d, kda.KDA_DTYPE_BF16, c["ws"].numel(), 0)
        return c

    def case_call(self, c, events=None, ws=None, flags=0):
        kda, x = self.kda, c["x"]
        ws = c["ws"] if ws is None else ws
        s0 = None if x["init_state"] is None else x["init_state"].data_ptr()
        args = (x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(), x["log_alpha"].data_ptr(),
                x["beta"].data_ptr(), x["cu_seqlens"].data_ptr(), c["N"], c["T"], c["H"], c["d"],
                c["d"], kda.KDA_DTYPE_BF16, s0, c["o"].data_ptr(), c["fs"].data_ptr(),
                ws.data_ptr(), ws.numel(), self.sh)
        if flags:
            st = kda.kda_prefill_ex(*args, flags)
        else:
            st = kda.kda_prefill(*args) if events is None else kda.kda_prefill_events(*args, events)
        if st != kda.KDA_OK:
            raise kda.KdaError(st, "kda_prefill")

    def time_bounded(self, c, chunks, steps, warmup, ring=False):
        """Event time (ms per call) of the same prefill with a workspace whose per-chunk
        records cover only `chunks` packed chunks: the two kernels over segments of that many
        chunks (KDA_FLAG_NO_STREAM), or with ring=True the streamed kernel over a ring of
        them; returns (ms, workspace bytes)."""
        torch = self.torch
        kda = self.kda
        make = kda.streamed_workspace_for if ring else kda.segmented_workspace_for
        ws = make(c["N"], c["T"], c["H"], c["d"], kda.KDA_DTYPE_BF16, self.dev, chunks)
        flags = 0 if ring else kda.KDA_FLAG_NO_STREAM
        for _ in range(warmup):
            self.case_call(c, ws=ws, flags=flags)
        torch.cuda.synchronize()
        a, b = self.event(), self.event()
        a.record(self.stream)
        for _ in range(steps):
            self.case_call(c, ws=ws, flags=flags)
        b.record(self.stream)
        torch.cuda.synchronize()
        st = self.kda.kda_read_device_status(ws.data_ptr(), self.sh)
        if st != self.kda.KDA_OK:
            raise self.kda.KdaError(st, "kda_prefill, bounded records (device status)")
        return a.elapsed_time(b) / steps, ws.numel()

    def time_case(self, c, steps, warmup):
        """Per-call event times (ms) of kda_prefill on one workload, and the per-kernel split
        from the same number of kda_prefill_events calls.  The inputs (over 1 GB) are far
        larger than L2, so no flush runs between calls."""
        torch = self.torch
        for _ in range(warmup):
            self.case_call(c)
        torch.cuda.synchronize()
        outer = [(self.event(), self.event()) for _ in range(steps)]
        for a, b in outer:
            a.record(self.stream)
            self.case_call(c)
            b.record(self.stream)
        torch.cuda.synchronize()
        ev = [[self.event() for _ in range(4)] for _ in range(steps)]
        for e in ev:
            for x in e:
                x.record(self.stream)
        torch.cuda.synchronize()
        for e in ev:
            self.case_call(c, [x.cuda_event for x in e])
        torch.cuda.synchronize()
        st = self.kda.kda_read_device_status(c["ws"].data_ptr(), self.sh)
        if st != self.kda.KDA_OK:
            raise self.kda.KdaError(st, "kda_prefill (device status)")
        return ([a.elapsed_time(b) for a, b in outer],
                [[e[i].elapsed_time(e[i + 1]) for i in range(3)] for e in ev])

    def setup_decode(self):
        torch, synth = self.torch, self.synth
        self.dw = dw = synth.DECODE_256
        self.ring = [{k: t.to(self.dev) for k, t in synth.decode_inputs(dw, s, seed=self.seed).items()}
                     for s in range(16)]
        self.state = synth.decode_state(dw, seed=self.seed).to(self.dev)
        self.o_dec = torch.empty((dw.batch, dw.num_heads, dw.d), dtype=torch.bfloat16,
                                 device=self.dev)

    def decode_call(self, s, stream_handle=None):
        kda, dw, r = self.kda, self.dw, self.ring[s % len(self.ring)]
        st = kda.kda_decode_step(r["q"].data_ptr(), r["k"].data_ptr(), r["v"].data_ptr(),
                                 r["log_alpha"].data_ptr(), r["beta"].data_ptr(), dw.batch,
                                 dw.num_heads, dw.d, dw.d, kda.KDA_DTYPE_BF16,
                                 self.state.data_ptr(), self.o_dec.data_ptr(),
                                 self.sh if stream_handle is None else stream_handle)
        if st != kda.KDA_OK:
            raise kda.KdaError(st, "kda_decode_step")

    def time_decode(self, steps, warmup, barrier):
        """Event time (ms) of `steps` in-place decode steps, captured once as a CUDA graph
        of `steps` kernel launches and replayed (the 537 MB state is larger than L2, so no
        flush is needed between steps)."""
        torch = self.torch
        for s in range(warmup):
            self.decode_call(s)
        torch.cuda.synchronize()
        graph, side = torch.cuda.CUDAGraph(), torch.cuda.Stream(self.dev)
        with torch.cuda.graph(graph, stream=side):
            for s in range(steps):
                self.decode_call(s, side.cuda_stream)
        torch.cuda.synchronize()
        barrier()
        a, b = self.event(), self.event()
        a.record(self.stream)
        graph.replay()
        b.record(self.stream)
        torch.cuda.synchronize()
        barrier()
        return a.elapsed_time(b)


def run_gpu(args):
    import torch

    rank, world, local_rank = _env_rank()
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    barrier = (lambda: dist.barrier()) if dist else (lambda: None)

    def reduce_max(v):
        return max_over_ranks(v, dist, torch.device("cuda", local_rank))

    g = _Gpu(args, rank, local_rank)
    peaks = measured_peaks()
    do_prefill = args.only in ("all", "prefill")
    do_decode = args.only in ("all", "decode")
    do_long = args.only in ("all", "long")
    # the long single sequence with an initial state, and the 16-sequence varlen pack
    case_ws = {"long_prefill": (g.synth.PREFILL_64K, "64k"), "varlen_prefill": (g.synth.VARLEN_16, "varlen16")}
    do_cases = [n for n in case_ws if args.only in ("all", n)]
    if do_prefill:
        g.setup_prefill()
    if do_long:
        g.setup_long()
    if do_decode:
        g.setup_decode()
    clocks = ClockSampler(local_rank)
    line = {"metric": METRIC, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded counter-based generator; no dataset)"}
    case_ms = {}
    with clocks:
        if do_prefill:
            step_ms, stage_ms = g.time_prefill(args.steps, args.warmup, barrier)
            prefill_path = g.prefill_path()
            # the same call with the chunk kernel and the state pass one after the other
            two_kernel_ms = g.time_prefill_flags(args.steps, args.warmup, g.kda.KDA_FLAG_NO_STREAM)
            e2e_ms = g.time_prefill_e2e(args.steps, args.warmup)
            # the prefill kernels' tensor-core product groups on their own (resident operands)
            phase_tflops = {name: g.kda.diag_tensor_phases(i, 2000, g.ws)
                            for i, name in enumerate(("chunk_kernel_products", "state_kernel_products",
                                                      "stream_walk_products"))}
        for name in do_cases:
            # one workload on the device at a time (the varlen pack holds about 20 GB)
            c = g.setup_case(case_ws[name][0])
            barrier()
            case_ms[name] = (c, g.time_case(c, CASE_STEPS, max(3, args.warmup)))
            if name == "long_prefill":  # the same call with records for BOUNDED_CHUNKS chunks at a time
                c["bounded"] = g.time_bounded(c, BOUNDED_CHUNKS, CASE_STEPS, max(3, args.warmup))
                if c["path"] == PATH_STREAMED:  # and with the records of a ring of RING_CHUNKS chunks
                    c["ring"] = g.time_bounded(c, RING_CHUNKS, CASE_STEPS, max(3, args.warmup), ring=True)
                c["full_ws_bytes"] = c["ws"].numel()
            c["with_init"] = c["inp"]["init_state"] is not None
            # the oracle's sample is cut out now; the full host inputs are dropped
            c["cpu_sample"] = case_sample(c["w"], c["inp"])
            for key in ("x", "o", "fs", "ws", "inp"):
                c.pop(key)
            torch.cuda.empty_cache()
        if do_decode:
            dec_ms = g.time_decode(g.dw.steps, max(3, args.warmup), barrier)
        if do_long:
            long_ms = g.time_long(5, max(3, args.warmup))
    if do_prefill:
        total_ms = reduce_max(sum(step_ms))
        e2e_total = reduce_max(sum(e2e_ms))
        mean_step_ms = total_ms / args.steps
        T, H, d = g.T, g.H, g.d
        # per kernel: mean event time (max over ranks) and its share of the algorithmic bytes
        stage_mean = [reduce_max(sum(s[i] for s in stage_ms)) / args.steps for i in range(3)]
        roof = prefill_roofline(T, H, d, 1, False, mean_step_ms, stage_mean, peaks, "4k", prefill_path)
        roof["path"]["executed_tensor_flops_per_call"] = executed_tensor_flops(T, H, d)
        roof["gemm_phases"] = dict(
            {name: {"achieved": tf, "unit": "TFLOP/s", "peak": peaks["bf16_tflops"],
                    "frac": tf / peaks["bf16_tflops"]} for name, tf in phase_tflops.items()},
            note="kda_diag_tensor_phases: each kernel's product groups issued back to back by "
                 "its own issue routines on operands resident in shared memory (executed "
                 "FLOPs, bf16/fp16 inputs, fp32 accumulate), 2000 repetitions per CTA: the "
                 "chunk work's groups (both paths), the state kernel's groups (64-column "
                 "slice, two-kernel path) and the streamed kernel's walk (whole head)")
        tk_whole, tk_stages = two_kernel_ms
        tk_ms = reduce_max(sum(tk_whole)) / args.steps
        tk_stage = [reduce_max(sum(s[i] for s in tk_stages)) / args.steps for i in range(3)]
        tk_roof = prefill_roofline(T, H, d, 1, False, tk_ms, tk_stage, peaks, "4k", PATH_TWO_KERNEL)
        roof["two_kernel_form"] = {
            "ms_per_call": tk_ms, "value": aggregate_rate(T, world, 1, tk_ms),
            "kernel": tk_roof["kernel"], "frac": tk_roof["frac"], "traffic": tk_roof["traffic"],
            "kernels": tk_roof["kernels"], "path_frac": tk_roof["path"]["frac"],
            "note": "the same call with KDA_FLAG_NO_STREAM: the chunk kernel, then the state pass "
                    "(kernel split from kda_prefill_events_ex with the same flag)"}
        roof["note"] = ("kernel durations from the four CUDA events kda_prefill_events records on "
                        "the launching stream around its kernels (a separate timed pass); the "
                        "dominant (longest) kernel is measured against its share of the path's "
                        "algorithmic bytes, the path (one kda_prefill between two events) against "
                        "all of them")
        line.update({
            "value": aggregate_rate(T, world, args.steps, total_ms),
            "ms_per_step": mean_step_ms,
            "config": {"workload": g.w.name, "batch": 1, "num_heads": H, "seq_len": T,
                       "d_k": d, "d_v": d, "chunk": 64, "io_dtype": "bf16",
                       "gate_state_dtype": "f32",
                       "l2": "flushed between timed steps (256 MiB write, untimed)",
                       "parallelism": f"replicas x{world} (independent units, no collective)"},
            "roofline": roof,
            "e2e": {"value": aggregate_rate(T, world, args.steps, e2e_total), "unit": "tokens/s",
                    "h2d_bytes_per_step": g.h2d, "d2h_bytes_per_step": g.d2h,
                    "call": "kda_prefill_host: pinned host buffers, the prompt cut into segments whose "
                            "copies overlap the prefill of the segments before (results bit for bit "
                            "those of kda_prefill)",
                    "link_gbs": (g.h2d + g.d2h) / (e2e_total / args.steps / 1e3) / 1e9,
                    "gpu_launches_per_step": g.e2e_launches},
            # schedule kernel and streamed kernel (or chunk kernel and state pass) per step
            "gpu_launches": (2 if prefill_path == PATH_STREAMED else 3) * args.steps,
        })
    line["clocks"] = clocks.summary()
    for name, (c, (call_ms, stages)) in case_ms.items():
        w, T, H, d, N = c["w"], c["T"], c["H"], c["d"], c["N"]
        ms = reduce_max(sum(call_ms)) / len(call_ms)
        stage_mean = [reduce_max(sum(st[i] for st in stages)) / len(stages) for i in range(3)]
        blk = {"metric": "KDA prefill tokens/s", "workload": w.name, "unit": "tokens/s",
               "value": aggregate_rate(T, world, 1, ms), "ms_per_call": ms, "steps": len(call_ms),
               "num_seqs": N, "total_tokens": T, "num_heads": H, "d_k": d, "d_v": d,
               "init_state": c["with_init"],
               "l2": "inputs larger than L2 (no flush)",
               "gpu_launches": (2 if c["path"] == PATH_STREAMED else 3) * len(call_ms),
               "roofline": prefill_roofline(T, H, d, N, c["with_init"], ms,
                                            stage_mean, peaks, case_ws[name][1], c["path"])}
        if "bounded" in c:
            bms, bws = c["bounded"]
            bms = reduce_max(bms)
            blk["bounded_records"] = {
                "segment_chunks": BOUNDED_CHUNKS, "workspace_bytes": bws, "full_workspace_bytes": c["full_ws_bytes"],
                "value": aggregate_rate(T, world, 1, bms), "ms_per_call": bms, "steps": CASE_STEPS,
                "note": "kda_prefill_ex(KDA_FLAG_NO_STREAM) with a workspace from "
                        "kda_prefill_workspace_size_segmented: the chunk and state kernels run over segments "
                        "of that many packed chunks (results bit for bit those of the full workspace in the "
                        "two-kernel form)"}
        if "ring" in c:
            rms, rws = c["ring"]
            rms = reduce_max(rms)
            blk["streamed_ring"] = {
                "ring_chunks": RING_CHUNKS, "workspace_bytes": rws, "full_workspace_bytes": c["full_ws_bytes"],
                "value": aggregate_rate(T, world, 1, rms), "ms_per_call": rms, "steps": CASE_STEPS,
                # DRAM bytes per launch (ncu) against the path's algorithmic bytes: the records stay in L2
                "traffic": profiled_traffic("prefill_stream_kernel_ring%d_64k" % RING_CHUNKS),
                "algorithmic_bytes_per_launch": blk["roofline"]["algorithmic_bytes_per_launch"],
                "note": "kda_prefill with a workspace from kda_prefill_workspace_size_streamed: the streamed "
                        "kernel keeps the records of that many packed chunks, each slot refilled once both "
                        "walkers have copied its record in (results bit for bit those of the full workspace)"}
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            blk["cpu_baseline"] = cpu_baseline_case(w, c["cpu_sample"])
        line[name] = blk
    if do_decode:
        dw = g.dw
        dec_ms = reduce_max(dec_ms)
        dec_bytes = decode_algorithmic_bytes(dw.batch, dw.num_heads, dw.d, 2)
        dec_step_ms = dec_ms / dw.steps
        dec_achieved = dec_bytes / (dec_step_ms / 1e3) / 1e9
        line["decode"] = {
            "metric": "KDA decode steps/s", "workload": dw.name,
            "value": aggregate_rate(1, world, dw.steps, dec_ms), "unit": "steps/s",
            "ms_per_step": dec_step_ms, "steps": dw.steps, "gpu_launches": dw.steps,
            "timing": "one CUDA graph of the steps' launches, replayed once between two events",
            "tokens_per_s": dw.steps * dw.batch * world / (dec_ms / 1e3),
            "roofline": {"bound": "hbm", "achieved": dec_achieved, "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": dec_achieved / peaks["hbm_gbs"],
                         "traffic": profiled_traffic("decode_256"),
                         "algorithmic_bytes_per_launch": dec_bytes}}
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            line["decode"]["cpu_baseline"] = cpu_baseline_decode(dw, g.seed)
    if do_long:
        T = g.lw.seq_lens[0]
        split_ms, unsplit_ms = reduce_max(long_ms[True]), reduce_max(long_ms[False])
        line["long_context"] = {
            "metric": "KDA prefill tokens/s, one long sequence with few heads",
            "workload": g.lw.name, "unit": "tokens/s",
            "value": aggregate_rate(T, world, 1, split_ms), "ms_per_call": split_ms,
            "unsplit_value": aggregate_rate(T, world, 1, unsplit_ms), "unsplit_ms_per_call": unsplit_ms,
            "speedup_of_sequence_split": unsplit_ms / split_ms, "steps": 5,
            "note": "default call (sequence-split state pass) against KDA_FLAG_NO_SEQ_SPLIT"}
    if do_prefill and rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(g.w, g.inp)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- CPU arm
def _oracle_inputs(inp):
    from kda_gated_delta_04_gb300 import synth
    return {k: synth.to_f64(inp[k]) for k in ("q", "k", "v", "log_alpha", "beta")}


def cpu_baseline(w, inp, heads=None):
    """The oracle as it stands, all host cores, on the whole prefill workload (or the
    given heads); returns the cpu_baseline object (tokens/s of that sample)."""
    import oracle
    f = _oracle_inputs(inp)
    if heads is not None:
        f = {k: np.ascontiguousarray(v[:, heads]) for k, v in f.items()}
    T, H = f["q"].shape[:2]
    # whole passes over the sample until about 12 s of CPU time (cores x wall) have run
    reps, t0 = 0, time.perf_counter()
    while True:
        _, _, used = oracle.prefill(f["q"], f["k"], f["v"], f["log_alpha"], f["beta"])
        reps += 1
        dt = time.perf_counter() - t0
        if dt * used >= 12.0 or reps >= 50:
            break
    return {"value": reps * T * H / w.num_heads / dt, "unit": "tokens/s", "cores": used,
            "kind": "oracle",
            "sample": f"{w.name}: {H} of {w.num_heads} heads x {T} tokens, fp64 token-by-token, "
                      f"{reps} passes in {dt:.2f} s wall on {used} threads (about {dt * used:.0f} s of CPU "
                      f"time); tokens/s counts a token as all {w.num_heads} heads",
            "cpu": _cpu_model(), "nproc": os.cpu_count()}


CASE_SAMPLE_TOKENS = {"prefill_bf16_T65536_H32_d128_state": 2048, "varlen16_bf16_T512-16384_H32_d128": 256}


def case_sample(w, inp):
    """The oracle's bounded sample of a larger prefill workload: every sequence and head,
    each sequence cut to its first few tokens (with its initial state, if any).  The
    oracle's cost per token-head does not depend on the position, so the rate carries over."""
    from kda_gated_delta_04_gb300 import synth
    n = CASE_SAMPLE_TOKENS[w.name]
    cu = inp["cu_seqlens"].numpy().astype(np.int64)
    idx = np.concatenate([np.arange(cu[i], min(cu[i + 1], cu[i] + n)) for i in range(len(cu) - 1)])
    lens = np.minimum(np.diff(cu), n)
    import torch
    sel = torch.from_numpy(idx)
    f = {k: np.ascontiguousarray(synth.to_f64(inp[k].index_select(0, sel)))
         for k in ("q", "k", "v", "log_alpha", "beta")}
    f["cu_seqlens"] = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    f["init_state"] = None if inp["init_state"] is None else synth.to_f64(inp["init_state"])
    f["desc"] = (f"{w.name}: the first {n} tokens of each of its {len(lens)} sequence(s) x all "
                 f"{w.num_heads} heads" + (" from the initial states" if inp["init_state"] is not None else ""))
    return f


def cpu_baseline_case(w, f):
    """The oracle as it stands, all host cores, on the sample case_sample() cut out."""
    import oracle
    T, H = f["q"].shape[:2]
    reps, t0 = 0, time.perf_counter()
    while True:
        _, _, used = oracle.prefill(f["q"], f["k"], f["v"], f["log_alpha"], f["beta"],
                                    cu_seqlens=f["cu_seqlens"], init_state=f["init_state"])
        reps += 1
        dt = time.perf_counter() - t0
        if dt * used >= 12.0 or reps >= 50:
            break
    return {"value": reps * T / dt, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": f"{f['desc']} ({T} tokens), fp64 token-by-token, {reps} passes in {dt:.2f} s "
                      f"wall on {used} threads (about {dt * used:.0f} s of CPU time); tokens/s counts "
                      f"a token as all {H} heads",
            "cpu": _cpu_model(), "nproc": os.cpu_count()}


def cpu_baseline_decode(dw, seed):
    """The oracle's decode step as it stands, all host cores, on the full batch (every
    sequence and head of the decode workload, the same state and per-step inputs), for as
    many of the workload's steps as fit about 12 s of CPU time; steps/s over those steps."""
    import oracle
    from kda_gated_delta_04_gb300 import synth
    state = synth.to_f64(synth.decode_state(dw, seed=seed))
    ring = [{k: synth.to_f64(t) for k, t in synth.decode_inputs(dw, s, seed=seed).items()}
            for s in range(16)]
    steps, t0 = 0, time.perf_counter()
    while True:
        r = ring[steps % len(ring)]
        _, used = oracle.decode_step(r["q"], r["k"], r["v"], r["log_alpha"], r["beta"], state)
        steps += 1
        dt = time.perf_counter() - t0
        if (dt * used >= 12.0 and steps >= 3) or steps >= dw.steps:
            break
    return {"value": steps / dt, "unit": "steps/s", "cores": used, "kind": "oracle",
            "sample": f"{dw.name}: the first {steps} of its {dw.steps} steps over all {dw.batch} x "
                      f"{dw.num_heads} units (fp64 state, in place), {dt:.2f} s wall on {used} threads "
                      f"(about {dt * used:.0f} s of CPU time); measured over those steps, not extrapolated",
            "cpu": _cpu_model(), "nproc": os.cpu_count()}


def _cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part", "hardware")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def run_reference(args):
    rank, world, _ = _env_rank()
    if rank != 0:
        return
    from kda_gated_delta_04_gb300 import synth
    import oracle
    w = synth.PREFILL_4K
    inp = synth.prefill_inputs(w, seed=args.seed)
    f = _oracle_inputs(inp)
    # each step: the oracle on the whole workload (32 heads x 4096 tokens, ~1-2 s on
    # 8-16 cores), so K steps stay within a few minutes
    heads = list(range(w.num_heads))
    fs = {k: np.ascontiguousarray(v[:, heads]) for k, v in f.items()}
    T = fs["q"].shape[0]
    used = 0
    for _ in range(args.warmup):
        oracle.prefill(fs["q"], fs["k"], fs["v"], fs["log_alpha"], fs["beta"])
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _, _, used = oracle.prefill(fs["q"], fs["k"], fs["v"], fs["log_alpha"], fs["beta"])
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = T * len(heads) / w.num_heads * args.steps / total
    sample = (f"{w.name}: all {len(heads)} heads x {T} tokens per step, fp64 token-by-token "
              f"oracle on {used} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded counter-based generator)",
        "config": {"workload": w.name, "batch": 1, "num_heads": w.num_heads, "seq_len": T,
                   "d_k": w.d, "d_v": w.d, "chunk": 64, "io_dtype": "bf16",
                   "gate_state_dtype": "f32"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
                         "sample": sample, "cpu": _cpu_model(), "nproc": os.cpu_count()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["all", "prefill", "decode", "long", "long_prefill",
                                       "varlen_prefill"], default="all",
                    help="profiling aid: run only one part (the printed line is then partial)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
