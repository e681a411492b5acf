"""The C-ABI library: builds, loads, exports every declared entry point, and
rejects bad arguments on the host before touching any GPU."""
import ctypes
import os
import pathlib
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def kda():
    from kda_gated_delta_04_gb300 import build
    build.build()
    from kda_gated_delta_04_gb300 import kda as binding
    return binding


def declared_functions():
    src = pathlib.Path(HEADER).read_text()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("kda_prefill", "kda_decode_step", "kda_prefill_workspace_size",
                     "kda_read_device_status", "kda_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(kda):
    lib = ctypes.CDLL(kda.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"libkda.so does not export {name}"
    assert set(declared_functions()) == set(kda.EXPORTS)


def test_binding_constants_match_the_header(kda):
    """Every integer constant the binding restates (status codes, dtypes, option flags, path
    codes, the ring minimum, device error bits) has the header's value: the header's integer
    #defines and enumerators, parsed from its text."""
    src = re.sub(r"/\*.*?\*/", "", pathlib.Path(HEADER).read_text(), flags=re.S)
    consts = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define\s+(KDA_[A-Z0-9_]+)\s+(\d+)u?\s*$", src, re.M)}
    consts.update({m.group(1): int(m.group(2)) for m in re.finditer(r"\b(KDA_[A-Z0-9_]+)\s*=\s*(\d+)\b", src)})
    shared = sorted(n for n in consts if hasattr(kda, n))
    for n in shared:
        assert getattr(kda, n) == consts[n], n
    for required in ("KDA_OK", "KDA_ERR_VALUE_RANGE", "KDA_DTYPE_F32", "KDA_FLAG_STREAM", "KDA_PATH_STREAMED",
                     "KDA_STREAM_RING_MIN"):
        assert required in shared, required

def test_status_strings(kda):
    for code in range(7):
        s = kda.status_string(code)
        assert s.startswith("KDA_")
    assert "unknown" in kda.status_string(99)


def test_workspace_size(kda):
    a = kda.kda_prefill_workspace_size(1, 4096, 32, 128, 128, 0)
    b = kda.kda_prefill_workspace_size(16, 10, 32, 128, 128, 0)
    assert a >= 256 + 4 and a % 256 == 0
    assert b >= 256 + 64 and b % 256 == 0
    assert kda.kda_prefill_workspace_size(-1, 0, 1, 64, 64, 1) == 0


def test_segmented_workspace_size(kda):
    """Bounded records: a fixed part (schedule, chunk numbering, descriptors and two carried
    [H, 128, 128] fp32 states) plus one 74,240-byte record per (chunk, head) of a segment,
    never more than the full two-kernel workspace without the sequence split."""
    H, T, N = 32, 65536, 1
    one = kda.kda_prefill_workspace_size_segmented(N, T, H, 128, 128, 0, 1)
    two = kda.kda_prefill_workspace_size_segmented(N, T, H, 128, 128, 0, 2)
    assert one > 2 * H * 128 * 128 * 4 and one % 256 == 0
    assert two - one == H * 74240
    bound = T // 64 + N
    full_seg = kda.kda_prefill_workspace_size_segmented(N, T, H, 128, 128, 0, bound)
    assert kda.kda_prefill_workspace_size_segmented(N, T, H, 128, 128, 0, 10 * bound) == full_seg
    assert full_seg - one == (bound - 1) * H * 74240
    # the records of every chunk, as in the full workspace (this shape has no sequence split),
    # plus the two carried states, less the full workspace's ready flag and copy count per
    # chunk-head record (and its item counter)
    flags = -(-(2 * bound * H + 1) * 4 // 256) * 256
    assert full_seg - kda.kda_prefill_workspace_size(N, T, H, 128, 128, 0) == 2 * H * 128 * 128 * 4 - flags
    for bad in (dict(seg=0), dict(dtype=1), dict(d=64), dict(T=0), dict(H=0)):
        a = dict(N=N, T=T, H=H, d=128, dtype=0, seg=4)
        a.update(bad)
        assert kda.kda_prefill_workspace_size_segmented(a["N"], a["T"], a["H"], a["d"], a["d"], a["dtype"],
                                                        a["seg"]) == 0


def test_streamed_workspace_size(kda):
    """kda_prefill_workspace_size_streamed: the streamed prefill's fixed part plus the records
    of ring_chunks packed chunks.  One more chunk adds one chunk's records (the step of the
    segmented size); clamped to every chunk it is the full workspace of a shape without the
    sequence split; 0 below KDA_STREAM_RING_MIN chunks and for shapes the tensor-core path
    does not run; at T = 65536, H = 32 a ring of 16 chunks is under 40 MB."""
    N, T, H = 1, 4096, 32
    bound = T // 64 + N
    size = lambda ring, d=128, dt=0, T=T: kda.kda_prefill_workspace_size_streamed(N, T, H, d, d, dt, ring)
    seg = lambda c: kda.kda_prefill_workspace_size_segmented(N, T, H, 128, 128, 0, c)
    assert size(9) - size(8) == seg(2) - seg(1) > 0
    full = kda.kda_prefill_workspace_size(N, T, H, 128, 128, 0)
    assert size(bound) == size(10 * bound) == full
    assert size(kda.KDA_STREAM_RING_MIN) > 0 and size(kda.KDA_STREAM_RING_MIN - 1) == 0
    assert size(8, dt=1) == 0 and size(8, d=64) == 0 and size(8, T=0) == 0
    assert 0 < kda.kda_prefill_workspace_size_streamed(1, 65536, 32, 128, 128, 0, 16) < 40e6

def test_prefill_path_query(kda):
    """kda_prefill_path, on the shapes and workspaces that decide it without the device (the
    streamed choice is checked on the GPU, the sequence split below): fp32 and d = 64 take the
    CUDA-core kernel, a bf16 d = 128 call with the minimal workspace the fused kernel, with a
    bounded-records workspace the segmented pass, and with the full workspace the two kernels
    when streaming and the sequence split are turned off.  Rejected arguments give the
    negated status kda_prefill_ex returns."""
    N, T, H = 1, 4096, 32
    full = kda.kda_prefill_workspace_size(N, T, H, 128, 128, 0)
    seg = kda.kda_prefill_workspace_size_segmented(N, T, H, 128, 128, 0, 4)
    minimal = kda.min_workspace_bytes(N)
    off = kda.KDA_FLAG_NO_STREAM | kda.KDA_FLAG_NO_SEQ_SPLIT
    assert kda.kda_prefill_path(N, T, H, 128, 128, 1, full, 0) == kda.KDA_PATH_CUDA_CORE
    assert kda.kda_prefill_path(N, T, H, 64, 64, 0, full, 0) == kda.KDA_PATH_CUDA_CORE
    assert kda.kda_prefill_path(N, T, H, 128, 128, 0, minimal, 0) == kda.KDA_PATH_FUSED
    assert kda.kda_prefill_path(N, T, H, 128, 128, 0, seg, 0) == kda.KDA_PATH_SEGMENTED
    assert kda.kda_prefill_path(N, T, H, 128, 128, 0, full, off) == kda.KDA_PATH_TWO_KERNEL
    assert kda.kda_prefill_path(N, T, H, 128, 128, 0, minimal - 1, 0) == -kda.KDA_ERR_INVALID_ARG
    assert kda.kda_prefill_path(N, T, H, 128, 128, 0, full, 1 << 9) == -kda.KDA_ERR_INVALID_ARG
    both = kda.KDA_FLAG_STREAM | kda.KDA_FLAG_NO_STREAM  # asking for and ruling out the streamed form
    assert kda.kda_prefill_path(N, T, H, 128, 128, 0, full, both) == -kda.KDA_ERR_INVALID_ARG
    assert kda.kda_prefill_path(N, T, H, 96, 96, 0, full, 0) == -kda.KDA_ERR_UNSUPPORTED



def test_sequence_split_choice(kda):
    """Which bf16 d = 128 calls with the full workspace take the sequence-split state pass
    (decided without the device; KDA_FLAG_NO_STREAM keeps the streamed form out of the
    answer).  Only up to 19 (sequence, head) units, so that the transition pass fits one
    wave, and only for sequences long enough for the split to pay, a bound that grows with
    the unit count.  The cases follow the timings the rule was set from: at 64 chunks per
    sequence the two kernels are faster at every unit count, at 96 the split is faster with
    4 and 8 units but not with 16 or 19, at 256 it is faster at every count up to 19."""
    def path(N, T, H, flags=0):
        ws = kda.kda_prefill_workspace_size(N, T, H, 128, 128, 0)
        return kda.kda_prefill_path(N, T, H, 128, 128, 0, ws, flags | kda.KDA_FLAG_NO_STREAM)
    split, two = kda.KDA_PATH_SEQ_SPLIT, kda.KDA_PATH_TWO_KERNEL
    for H in (1, 4, 8, 16, 19):
        assert path(1, 4096, H) == two, H
        assert path(1, 16384, H) == split, H
    for H, want in ((4, split), (8, split), (16, two), (19, two)):
        assert path(1, 6144, H) == want, H
    assert path(2, 16384, 4) == split            # two sequences of 128 chunks: 8 units
    assert path(4, 16384, 4) == two              # four of 64 chunks: too short
    assert path(1, 65536, 20) == two             # 20 units: the transition pass needs two waves
    assert path(1, 65536, 4, kda.KDA_FLAG_NO_SEQ_SPLIT) == two
    assert path(1, 256, 1) == two                # 4 chunks: no room for three segments

FAKE = 1 << 20  # 16-byte aligned dummy address; never dereferenced (rejected first)


def _prefill_args(**over):
    a = dict(q=FAKE, k=FAKE, v=FAKE, log_alpha=FAKE, beta=FAKE, cu_seqlens=None, num_seqs=1,
             total_tokens=64, num_heads=2, d_k=64, d_v=64, dtype=1, init_state=None, o=FAKE,
             final_state=FAKE, workspace=FAKE, workspace_bytes=1 << 16, stream=None)
    a.update(over)
    return a


@pytest.mark.parametrize("over,expected", [
    (dict(q=None), 1), (dict(o=FAKE + 8), 1), (dict(final_state=None), 1), (dict(workspace=None), 1),
    (dict(q=FAKE + 4), 1), (dict(workspace=FAKE + 16), 1), (dict(workspace_bytes=8), 1),
    (dict(num_seqs=2), 1),                     # cu_seqlens required for several sequences
    (dict(num_heads=0), 1), (dict(total_tokens=-1), 1), (dict(dtype=7), 1),
    (dict(num_seqs=0, total_tokens=5, cu_seqlens=FAKE), 1),
    (dict(d_k=96, d_v=96), 2), (dict(d_k=128, d_v=64), 2), (dict(d_k=256, d_v=256), 2),
])
def test_prefill_rejects_bad_arguments_on_host(kda, over, expected):
    a = _prefill_args(**over)
    assert kda.kda_prefill(*a.values()) == expected


@pytest.mark.parametrize("over,expected", [
    (dict(state=None), 1), (dict(beta=None), 1), (dict(o=FAKE + 8), 1), (dict(num_heads=0), 1),
    (dict(batch=-1), 1), (dict(d_k=32, d_v=32), 2), (dict(dtype=3), 1),
])
def test_decode_rejects_bad_arguments_on_host(kda, over, expected):
    a = dict(q=FAKE, k=FAKE, v=FAKE, log_alpha=FAKE, beta=FAKE, batch=4, num_heads=2, d_k=128,
             d_v=128, dtype=0, state=FAKE, o=FAKE, stream=None)
    a.update(over)
    assert kda.kda_decode_step(*a.values()) == expected


def test_binding_refuses_cpu_tensors(kda):
    import torch
    x = torch.zeros(4, 1, 64)
    with pytest.raises(TypeError):
        kda.decode_step(x, x, x, x, torch.zeros(4, 1), torch.zeros(4, 1, 64, 64))


def test_product_path_does_not_import_the_oracle():
    """The package and its native sources never reach the oracle or its sources."""
    pkg = os.path.join(ROOT, "kda_gated_delta_04_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".c", ".h")):
                text = pathlib.Path(dirpath, f).read_text()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "kda_oracle" not in text, f


def test_unknown_flags_are_rejected_on_host(kda):
    a = _prefill_args()
    assert kda.kda_prefill_ex(*a.values(), 1 << 7) == 1
    assert kda.kda_decode_step_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 128, 128, 0, FAKE, FAKE, None,
                                  1 << 7) == 1


def test_slot_calls_reject_bad_arguments_on_host(kda):
    head = list(_prefill_args().values())[:12]

    def prefill_slots(pool=FAKE, num_slots=4, init_slots=None, final_slots=FAKE, flags=1):
        return kda.kda_prefill_slots(*head, pool, num_slots, init_slots, final_slots, FAKE, FAKE,
                                     1 << 16, None, flags)
    assert prefill_slots(pool=None) == 1
    assert prefill_slots(final_slots=None) == 1
    assert prefill_slots(num_slots=-1) == 1
    assert prefill_slots(init_slots=FAKE + 2) == 1      # misaligned
    assert prefill_slots(flags=1 << 7) == 1             # unknown flag
    dec = [FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2, 128, 128, 0, FAKE, 8, FAKE, FAKE, None, None]
    assert kda.kda_decode_step_slots(*dec, 1 << 7) == 1  # unknown flag


def test_diag_tensor_phases_rejects_bad_arguments_on_host(kda):
    import ctypes
    out = ctypes.c_double(0.0)
    assert kda.kda_diag_tensor_phases(3, 10, FAKE, None, ctypes.byref(out)) == 1    # no such pass
    assert kda.kda_diag_tensor_phases(0, 0, FAKE, None, ctypes.byref(out)) == 1     # no repetition
    assert kda.kda_diag_tensor_phases(0, 10, FAKE + 16, None, ctypes.byref(out)) == 1  # misaligned
    assert kda.kda_diag_tensor_phases(1, 10, None, None, ctypes.byref(out)) == 1    # no workspace
    assert kda.kda_diag_tensor_phases(0, 10, FAKE, None, None) == 1                 # no result


def _segments(kda, cu, N, T):
    import ctypes
    bounds = (ctypes.c_int64 * 8)()
    arr = None if cu is None else (ctypes.c_int32 * len(cu))(*cu)
    n = kda.kda_prefill_host_segments(None if arr is None else ctypes.addressof(arr), N, T,
                                      ctypes.addressof(bounds), 8)
    return n, [bounds[i] for i in range(max(n, 0) + 1)]


@pytest.mark.parametrize("cu,T", [
    (None, 4096), (None, 1500), (None, 2048), (None, 100000),
    ([0, 700, 700, 3000, 3064, 3065, 9000], 9000), ([0, 5000], 5000), ([0, 1, 2, 3, 4096], 4096),
])
def test_host_prefill_segments_fall_on_chunk_boundaries(kda, cu, T):
    """kda_prefill_host's cuts: at most four segments, strictly increasing from 0 to T, prompts
    under 2,048 tokens uncut, and every cut a 64-token multiple from the start of the
    sequence it falls in (so every chunk is the one a single kda_prefill runs)."""
    N = 1 if cu is None else len(cu) - 1
    n, b = _segments(kda, cu, N, T)
    assert 1 <= n <= 4 and b[0] == 0 and b[n] == T
    assert all(b[i] < b[i + 1] for i in range(n))
    if T < 2048:
        assert n == 1
    starts = [0] if cu is None else cu[:-1]
    for cut in b[1:n]:
        start = max(s for s in starts if s <= cut)
        assert (cut - start) % 64 == 0, (cut, start)


def test_host_prefill_sizes_and_host_side_checks(kda):
    import ctypes
    assert kda.kda_prefill_host_buffer_size(None, 1, 4096, 32, 128, 128, 0) > 4096 * 32 * 128 * 2
    assert kda.kda_prefill_host_buffer_size(None, 2, 4096, 32, 128, 128, 0) == 0    # cu_seqlens needed
    assert kda.kda_prefill_host_buffer_size(None, 1, 4096, 32, 128, 64, 0) == 0     # d_k != d_v
    n, _ = _segments(kda, None, 1, 0)
    assert n == 0
    bad_cu = (ctypes.c_int32 * 3)(0, 10, 9)                                           # not a prefix sum
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.addressof(bad_cu), 2, 9, 2, 128, 128, 0, None, FAKE,
            FAKE, FAKE, 1 << 30, None, 0]
    assert kda.kda_prefill_host(*args) == 1
    good_cu = (ctypes.c_int32 * 3)(0, 4, 9)
    args[5] = ctypes.addressof(good_cu)
    args[15] = FAKE + 16                                                              # misaligned buffer
    assert kda.kda_prefill_host(*args) == 1
    args[15] = FAKE
    args[9], args[10] = 96, 96                                                        # unsupported d
    assert kda.kda_prefill_host(*args) == 2
