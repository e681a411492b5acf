// kda_api.cu -- the extern "C" boundary of libkda: argument validation, workspace
// layout and kernel launches.  No compute happens here.
#include <stdint.h>
#include <string.h>

#include "common.cuh"

namespace {

constexpr int kMaxDevices = 64;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Device check, cached per device (the only global state of the library):
// 1 = supported (compute capability 10.3), -1 = not supported, 0 = unknown.
int g_device_ok[kMaxDevices];

kda_status_t check_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
    if (g_device_ok[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return KDA_ERR_CUDA;
        g_device_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    return g_device_ok[dev] == 1 ? KDA_OK : KDA_ERR_UNSUPPORTED;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace layout: status header | sequence order | first chunk of each sequence
// | per-chunk descriptors | per chunk-head ready flags | per chunk-head records (the last
// four only for the two-kernel tensor-core path; the bounded-records layout carries two
// states per head instead of the flags, and records for a segment of chunks).
size_t ws_order_bytes(int32_t num_seqs) { return round_up((size_t)num_seqs * sizeof(int32_t) + 1, 256); }
size_t ws_min_bytes(int32_t num_seqs) { return kda::kWorkspaceHeader + ws_order_bytes(num_seqs); }
size_t ws_cc_bytes(int32_t num_seqs) { return round_up(((size_t)num_seqs + 1) * sizeof(int32_t), 256); }
// one (first token, rows) pair per packed chunk, bounded by total_tokens / 64 + num_seqs
int64_t chunk_bound(int32_t num_seqs, int64_t total_tokens) { return total_tokens / kda::kChunk + num_seqs; }
size_t ws_desc_bytes(int32_t num_seqs, int64_t total_tokens)
{
    return round_up((size_t)chunk_bound(num_seqs, total_tokens) * 2 * sizeof(int32_t), 256);
}
bool split_shape(int32_t num_seqs, int64_t total_tokens, int32_t num_heads, int32_t d_k, int32_t d_v,
                 kda_dtype_t dtype)
{
    // the chunk kernel's one-dimensional grid holds (chunks + sequences) x heads CTAs
    return dtype == KDA_DTYPE_BF16 && d_k == 128 && d_v == 128 && total_tokens > 0 &&
           total_tokens <= 0x7fffffffll &&
           (total_tokens / KDA_CHUNK + num_seqs) * (int64_t)num_heads <= 0x7fffffffll;
}
// a ready flag and a copy count (int32 each) per chunk-head record and an item counter, for
// the streamed prefill
size_t ws_flags_bytes(int32_t num_seqs, int64_t total_tokens, int32_t num_heads)
{
    return round_up((2 * (size_t)chunk_bound(num_seqs, total_tokens) * (size_t)num_heads + 1) * sizeof(int32_t),
                    256);
}
// the two-kernel path: schedule, chunk numbering, descriptors, ready flags and records
size_t ws_records_bytes(int32_t num_seqs, int64_t total_tokens, int32_t num_heads)
{
    return ws_min_bytes(num_seqs) + ws_cc_bytes(num_seqs) + ws_desc_bytes(num_seqs, total_tokens) +
           ws_flags_bytes(num_seqs, total_tokens, num_heads) +
           kda::prefill_split_records_bytes(total_tokens, num_seqs, num_heads);
}
// the streamed prefill over a ring of records: schedule, chunk numbering, descriptors,
// flags and counts; the records of as many packed chunks as the rest holds follow
size_t ws_stream_fixed(int32_t num_seqs, int64_t total_tokens, int32_t num_heads)
{
    return ws_min_bytes(num_seqs) + ws_cc_bytes(num_seqs) + ws_desc_bytes(num_seqs, total_tokens) +
           ws_flags_bytes(num_seqs, total_tokens, num_heads);
}
// packed chunks whose records a workspace of that size holds after the streamed prefill's
// fixed part, up to all of them; 0 when fewer than kStreamRingMin (and not all)
int64_t stream_ring_chunks(int32_t num_seqs, int64_t total_tokens, int32_t num_heads, size_t workspace_bytes)
{
    const size_t fixed = ws_stream_fixed(num_seqs, total_tokens, num_heads);
    if (workspace_bytes <= fixed) return 0;
    const int64_t fit = (int64_t)((workspace_bytes - fixed) / ((size_t)num_heads * kda::prefill_split_record_bytes()));
    const int64_t all = chunk_bound(num_seqs, total_tokens);
    const int64_t ring = fit < all ? fit : all;
    return ring >= kda::kStreamRingMin || ring == all ? ring : 0;
}
// ... plus the sequence-split state pass where the shape calls for it
size_t ws_split_bytes(int32_t num_seqs, int64_t total_tokens, int32_t num_heads)
{
    return ws_records_bytes(num_seqs, total_tokens, num_heads) +
           kda::seqsplit_bytes(num_seqs, total_tokens, num_heads);
}
// the two-kernel path with bounded records: schedule, chunk numbering, descriptors, two
// carried states per head ([num_heads, 128, 128] fp32 each) and records for seg_chunks chunks
size_t ws_carry_bytes(int32_t num_heads) { return round_up((size_t)2 * num_heads * 128 * 128 * sizeof(float), 256); }
size_t ws_segmented_fixed(int32_t num_seqs, int64_t total_tokens, int32_t num_heads)
{
    return ws_min_bytes(num_seqs) + ws_cc_bytes(num_seqs) + ws_desc_bytes(num_seqs, total_tokens) +
           ws_carry_bytes(num_heads);
}

// The path kda_prefill_ex takes for a call with these arguments (kda_prefill_path_t): the
// decisions of prefill_impl below, in the same order.
int32_t path_for(int32_t num_seqs, int64_t total_tokens, int32_t num_heads, int32_t d_k, int32_t d_v,
                 kda_dtype_t dtype, size_t workspace_bytes, uint32_t flags)
{
    const bool split_ok = split_shape(num_seqs, total_tokens, num_heads, d_k, d_v, dtype);
    const bool full = split_ok && workspace_bytes >= ws_records_bytes(num_seqs, total_tokens, num_heads);
    if (full) {
        if (!(flags & KDA_FLAG_NO_SEQ_SPLIT) && workspace_bytes >= ws_split_bytes(num_seqs, total_tokens, num_heads) &&
            kda::seqsplit_lseg(num_seqs, total_tokens, num_heads) > 0)
            return KDA_PATH_SEQ_SPLIT;
        if (!(flags & KDA_FLAG_NO_STREAM) &&
            kda::prefill_stream_fits((int64_t)num_seqs * num_heads, kda::mean_chunks_per_sequence(num_seqs, total_tokens),
                                     (flags & KDA_FLAG_STREAM) != 0))
            return KDA_PATH_STREAMED;
        return KDA_PATH_TWO_KERNEL;
    }
    // a bounded workspace: the streamed prefill over a ring of records where the call would
    // stream, else the two kernels in segments
    if (split_ok && !(flags & KDA_FLAG_NO_STREAM) &&
        stream_ring_chunks(num_seqs, total_tokens, num_heads, workspace_bytes) > 0 &&
        kda::prefill_stream_fits((int64_t)num_seqs * num_heads, kda::mean_chunks_per_sequence(num_seqs, total_tokens),
                                 (flags & KDA_FLAG_STREAM) != 0))
        return KDA_PATH_STREAMED;
    const size_t rec_chunk = (size_t)num_heads * kda::prefill_split_record_bytes();
    if (split_ok && workspace_bytes >= ws_segmented_fixed(num_seqs, total_tokens, num_heads) + rec_chunk)
        return KDA_PATH_SEGMENTED;
    const bool tc = dtype == KDA_DTYPE_BF16 && d_k == 128 && total_tokens > 0 && total_tokens <= 0x7fffffffll;
    return tc ? KDA_PATH_FUSED : KDA_PATH_CUDA_CORE;
}

kda_status_t check_shape(int32_t d_k, int32_t d_v, kda_dtype_t dtype)
{
    if (dtype != KDA_DTYPE_BF16 && dtype != KDA_DTYPE_F32) return KDA_ERR_INVALID_ARG;
    if (d_k <= 0 || d_v <= 0) return KDA_ERR_INVALID_ARG;
    if (d_k != d_v || (d_k != 64 && d_k != 128)) return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

}  // namespace

// every option bit of the _ex / _slots calls
constexpr uint32_t kKnownFlags =
    KDA_FLAG_SCALAR_GATE | KDA_FLAG_QK_L2NORM | KDA_FLAG_NO_SEQ_SPLIT | KDA_FLAG_NO_STREAM | KDA_FLAG_STREAM;
// flags valid for a call: known bits, and not both streaming choices
inline bool flags_valid(uint32_t flags)
{
    return !(flags & ~kKnownFlags) && (flags & (KDA_FLAG_STREAM | KDA_FLAG_NO_STREAM)) != (KDA_FLAG_STREAM | KDA_FLAG_NO_STREAM);
}

extern "C" {

size_t kda_prefill_workspace_size(int32_t num_seqs, int64_t total_tokens, int32_t num_heads,
                                  int32_t d_k, int32_t d_v, kda_dtype_t dtype)
{
    if (num_seqs < 0 || total_tokens < 0 || num_heads < 0) return 0;
    if (split_shape(num_seqs, total_tokens, num_heads, d_k, d_v, dtype))
        return ws_split_bytes(num_seqs, total_tokens, num_heads);
    return ws_min_bytes(num_seqs);
}

size_t kda_prefill_workspace_size_segmented(int32_t num_seqs, int64_t total_tokens, int32_t num_heads,
                                            int32_t d_k, int32_t d_v, kda_dtype_t dtype,
                                            int64_t segment_chunks)
{
    if (num_seqs < 0 || total_tokens < 0 || num_heads <= 0 || segment_chunks < 1) return 0;
    if (!split_shape(num_seqs, total_tokens, num_heads, d_k, d_v, dtype)) return 0;
    const int64_t bound = chunk_bound(num_seqs, total_tokens);
    const int64_t seg = segment_chunks < bound ? segment_chunks : bound;
    return ws_segmented_fixed(num_seqs, total_tokens, num_heads) +
           (size_t)seg * (size_t)num_heads * kda::prefill_split_record_bytes();
}

size_t kda_prefill_workspace_size_streamed(int32_t num_seqs, int64_t total_tokens, int32_t num_heads,
                                           int32_t d_k, int32_t d_v, kda_dtype_t dtype, int64_t ring_chunks)
{
    if (num_seqs < 0 || total_tokens < 0 || num_heads <= 0 || ring_chunks < kda::kStreamRingMin) return 0;
    if (!split_shape(num_seqs, total_tokens, num_heads, d_k, d_v, dtype)) return 0;
    const int64_t bound = chunk_bound(num_seqs, total_tokens);
    const int64_t ring = ring_chunks < bound ? ring_chunks : bound;
    return ws_stream_fixed(num_seqs, total_tokens, num_heads) +
           (size_t)ring * (size_t)num_heads * kda::prefill_split_record_bytes();
}

int32_t kda_prefill_path(int32_t num_seqs, int64_t total_tokens, int32_t num_heads, int32_t d_k,
                         int32_t d_v, kda_dtype_t dtype, size_t workspace_bytes, uint32_t flags)
{
    if (!flags_valid(flags)) return -(int32_t)KDA_ERR_INVALID_ARG;
    const kda_status_t st = check_shape(d_k, d_v, dtype);
    if (st != KDA_OK) return -(int32_t)st;
    if (num_seqs < 0 || total_tokens < 0 || num_heads <= 0 || (num_seqs == 0 && total_tokens != 0))
        return -(int32_t)KDA_ERR_INVALID_ARG;
    if (num_seqs > 65535 || num_heads > 65535) return -(int32_t)KDA_ERR_UNSUPPORTED;
    if (workspace_bytes < ws_min_bytes(num_seqs)) return -(int32_t)KDA_ERR_INVALID_ARG;
    return path_for(num_seqs, total_tokens, num_heads, d_k, d_v, dtype, workspace_bytes, flags);
}

namespace {

// The prefill behind both entry points; ev (four events, or NULL) marks the stages.
kda_status_t prefill_impl(const void *q, const void *k, const void *v, const float *log_alpha,
                          const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                          int64_t total_tokens, int32_t num_heads, int32_t d_k, int32_t d_v,
                          kda_dtype_t dtype, const float *init_state, void *o, float *final_state,
                          void *workspace, size_t workspace_bytes, void *stream, const cudaEvent_t *ev,
                          uint32_t flags, const kda::StateSlots *slots = nullptr)
{
    if (!flags_valid(flags)) return KDA_ERR_INVALID_ARG;
    const bool scalar_gate = (flags & KDA_FLAG_SCALAR_GATE) != 0;
    kda_status_t st = check_shape(d_k, d_v, dtype);
    if (st != KDA_OK) return st;
    if (num_seqs < 0 || total_tokens < 0 || num_heads <= 0) return KDA_ERR_INVALID_ARG;
    if (num_seqs == 0 && total_tokens != 0) return KDA_ERR_INVALID_ARG;
    if (!cu_seqlens && num_seqs != 1) return KDA_ERR_INVALID_ARG;
    if (num_seqs > 65535) return KDA_ERR_UNSUPPORTED;  // grid z extent
    if (num_heads > 65535) return KDA_ERR_UNSUPPORTED;  // grid y extent
    // token tensors may be NULL only when there are no tokens; o may be NULL (final states only)
    if (total_tokens > 0 && (!q || !k || !v || !log_alpha || !beta))
        return KDA_ERR_INVALID_ARG;
    if (!final_state || !workspace) return KDA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(log_alpha, scalar_gate ? 4 : 16) ||
        !aligned(o, 16) || !aligned(final_state, 16) || !aligned(beta, 4) ||
        (init_state && !aligned(init_state, 16)) || (cu_seqlens && !aligned(cu_seqlens, 4)) ||
        !aligned(workspace, 256))
        return KDA_ERR_INVALID_ARG;
    if (workspace_bytes < ws_min_bytes(num_seqs)) return KDA_ERR_INVALID_ARG;
    st = check_device();
    if (st != KDA_OK) return st;
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    auto mark = [&](int i) { return !ev || cudaEventRecord(ev[i], strm) == cudaSuccess; };
    if (num_seqs == 0) return mark(0) && mark(1) && mark(2) && mark(3) ? KDA_OK : KDA_ERR_CUDA;

    kda::PrefillProblem p;
    p.q = q; p.k = k; p.v = v; p.log_alpha = log_alpha; p.beta = beta;
    p.cu_seqlens = cu_seqlens; p.num_seqs = num_seqs; p.total_tokens = total_tokens;
    p.num_heads = num_heads; p.d = d_k; p.dtype = dtype; p.init_state = init_state;
    p.o = o; p.final_state = final_state;
    p.scalar_gate = scalar_gate;
    p.qk_l2norm = (flags & KDA_FLAG_QK_L2NORM) != 0;
    if (slots) p.slots = *slots;
    p.status = static_cast<uint32_t *>(workspace);
    char *ws = static_cast<char *>(workspace);
    p.order = reinterpret_cast<int32_t *>(ws + kda::kWorkspaceHeader);
    p.stream = strm;
    // bf16 at d = 128 runs on the tensor cores: as the chunk / state kernel pair when the
    // workspace holds the per-chunk records (all of them, or those of a bounded number of
    // chunks at a time, the pass then run in segments), else as the single fused kernel.
    // fp32 I/O (the exact path) and d = 64 run the CUDA-core chunk kernel.
    const bool split_ok = split_shape(num_seqs, total_tokens, num_heads, d_k, d_v, dtype);
    const bool full = split_ok && workspace_bytes >= ws_records_bytes(num_seqs, total_tokens, num_heads);
    const size_t rec_chunk = (size_t)num_heads * kda::prefill_split_record_bytes();
    const size_t seg_fixed = split_ok ? ws_segmented_fixed(num_seqs, total_tokens, num_heads) : 0;
    // a bounded workspace: the streamed prefill over a ring of records where the call would
    // stream (the same choice as kda_prefill_path), else the two kernels in segments
    const int64_t ring = split_ok && !full && !(flags & KDA_FLAG_NO_STREAM)
                             ? stream_ring_chunks(num_seqs, total_tokens, num_heads, workspace_bytes)
                             : 0;
    const bool ring_stream =
        ring > 0 && kda::prefill_stream_fits((int64_t)num_seqs * num_heads,
                                             kda::mean_chunks_per_sequence(num_seqs, total_tokens),
                                             (flags & KDA_FLAG_STREAM) != 0);
    const bool segmented = split_ok && !full && !ring_stream && workspace_bytes >= seg_fixed + rec_chunk;
    const bool split = full || ring_stream || segmented;
    p.cc = split ? reinterpret_cast<int32_t *>(ws + ws_min_bytes(num_seqs)) : nullptr;
    p.desc = split ? reinterpret_cast<int2 *>(ws + ws_min_bytes(num_seqs) + ws_cc_bytes(num_seqs)) : nullptr;
    p.chunk_bound = split ? (int)chunk_bound(num_seqs, total_tokens) : 0;
    const size_t after_desc = ws_min_bytes(num_seqs) + ws_cc_bytes(num_seqs) + ws_desc_bytes(num_seqs, total_tokens);
    if (full) {
        if (!(flags & KDA_FLAG_NO_STREAM)) p.flags = reinterpret_cast<int *>(ws + after_desc);
        p.stream_force = (flags & KDA_FLAG_STREAM) != 0;
        p.records = ws + after_desc + ws_flags_bytes(num_seqs, total_tokens, num_heads);
    } else if (ring_stream) {
        p.flags = reinterpret_cast<int *>(ws + after_desc);
        p.stream_force = (flags & KDA_FLAG_STREAM) != 0;
        p.records = ws + after_desc + ws_flags_bytes(num_seqs, total_tokens, num_heads);
        p.ring_chunks = (int)ring;
    } else if (segmented) {
        p.carry = reinterpret_cast<float *>(ws + after_desc);
        p.records = ws + seg_fixed;
        const size_t fit = (workspace_bytes - seg_fixed) / rec_chunk;
        p.seg_chunks = fit < (size_t)p.chunk_bound ? (int)fit : p.chunk_bound;
    } else {
        p.records = nullptr;
    }
    // few (sequence, head) units: the state pass runs each sequence in segments
    if (full && !(flags & KDA_FLAG_NO_SEQ_SPLIT) &&
        workspace_bytes >= ws_split_bytes(num_seqs, total_tokens, num_heads))
        kda::seqsplit_carve(p.split, num_seqs, total_tokens, num_heads,
                            static_cast<char *>(p.records) +
                                kda::prefill_split_records_bytes(total_tokens, num_seqs, num_heads));

    if (!mark(0)) return KDA_ERR_CUDA;
    if (kda::launch_prefill_prep(p) != cudaSuccess) return KDA_ERR_CUDA;
    if (!mark(1)) return KDA_ERR_CUDA;
    cudaError_t err;
    if (split) {
        err = kda::launch_prefill_split(p, p.cc, p.records, ev ? ev[2] : nullptr);
    } else {
        if (!mark(2)) return KDA_ERR_CUDA;
        err = kda::prefill_tc_supported(p) ? kda::launch_prefill_tc(p) : kda::launch_prefill_simt(p);
    }
    if (err != cudaSuccess) return KDA_ERR_CUDA;
    if (!mark(3)) return KDA_ERR_CUDA;
    return KDA_OK;
}

}  // namespace

kda_status_t kda_prefill(const void *q, const void *k, const void *v, const float *log_alpha,
                         const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                         int64_t total_tokens, int32_t num_heads, int32_t d_k, int32_t d_v,
                         kda_dtype_t dtype, const float *init_state, void *o, float *final_state,
                         void *workspace, size_t workspace_bytes, void *stream)
{
    return prefill_impl(q, k, v, log_alpha, beta, cu_seqlens, num_seqs, total_tokens, num_heads, d_k,
                        d_v, dtype, init_state, o, final_state, workspace, workspace_bytes, stream,
                        nullptr, 0u);
}

kda_status_t kda_prefill_ex(const void *q, const void *k, const void *v, const float *log_alpha,
                            const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                            int64_t total_tokens, int32_t num_heads, int32_t d_k, int32_t d_v,
                            kda_dtype_t dtype, const float *init_state, void *o, float *final_state,
                            void *workspace, size_t workspace_bytes, void *stream, uint32_t flags)
{
    return prefill_impl(q, k, v, log_alpha, beta, cu_seqlens, num_seqs, total_tokens, num_heads, d_k,
                        d_v, dtype, init_state, o, final_state, workspace, workspace_bytes, stream,
                        nullptr, flags);
}

kda_status_t kda_prefill_slots(const void *q, const void *k, const void *v, const float *log_alpha,
                               const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                               int64_t total_tokens, int32_t num_heads, int32_t d_k, int32_t d_v,
                               kda_dtype_t dtype, float *state_pool, int32_t num_slots,
                               const int32_t *init_slots, const int32_t *final_slots, void *o,
                               void *workspace, size_t workspace_bytes, void *stream, uint32_t flags)
{
    if (num_slots < 0 || !state_pool || !final_slots || !aligned(init_slots, 4) || !aligned(final_slots, 4))
        return KDA_ERR_INVALID_ARG;
    kda::StateSlots slots;
    slots.init = init_slots;
    slots.fin = final_slots;
    slots.num = num_slots;
    return prefill_impl(q, k, v, log_alpha, beta, cu_seqlens, num_seqs, total_tokens, num_heads, d_k,
                        d_v, dtype, init_slots ? state_pool : nullptr, o, state_pool, workspace,
                        workspace_bytes, stream, nullptr, flags, &slots);
}

kda_status_t kda_prefill_events_ex(const void *q, const void *k, const void *v, const float *log_alpha,
                                   const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                                   int64_t total_tokens, int32_t num_heads, int32_t d_k, int32_t d_v,
                                   kda_dtype_t dtype, const float *init_state, void *o,
                                   float *final_state, void *workspace, size_t workspace_bytes,
                                   void *stream, void *const *events, int32_t num_events, uint32_t flags)
{
    if (!events || num_events != 4) return KDA_ERR_INVALID_ARG;
    cudaEvent_t ev[4];
    for (int i = 0; i < 4; ++i) {
        if (!events[i]) return KDA_ERR_INVALID_ARG;
        ev[i] = static_cast<cudaEvent_t>(events[i]);
    }
    return prefill_impl(q, k, v, log_alpha, beta, cu_seqlens, num_seqs, total_tokens, num_heads, d_k,
                        d_v, dtype, init_state, o, final_state, workspace, workspace_bytes, stream, ev, flags);
}

kda_status_t kda_prefill_events(const void *q, const void *k, const void *v, const float *log_alpha,
                                const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                                int64_t total_tokens, int32_t num_heads, int32_t d_k, int32_t d_v,
                                kda_dtype_t dtype, const float *init_state, void *o,
                                float *final_state, void *workspace, size_t workspace_bytes,
                                void *stream, void *const *events, int32_t num_events)
{
    return kda_prefill_events_ex(q, k, v, log_alpha, beta, cu_seqlens, num_seqs, total_tokens, num_heads, d_k,
                                 d_v, dtype, init_state, o, final_state, workspace, workspace_bytes, stream,
                                 events, num_events, 0u);
}

kda_status_t kda_decode_step_slots(const void *q, const void *k, const void *v, const float *log_alpha,
                                   const float *beta, int32_t batch, int32_t num_heads, int32_t d_k,
                                   int32_t d_v, kda_dtype_t dtype, float *state_pool, int32_t num_slots,
                                   const int32_t *slots, void *o, uint32_t *device_errors, void *stream,
                                   uint32_t flags)
{
    if (!flags_valid(flags)) return KDA_ERR_INVALID_ARG;
    const bool scalar_gate = (flags & KDA_FLAG_SCALAR_GATE) != 0;
    kda_status_t st = check_shape(d_k, d_v, dtype);
    if (st != KDA_OK) return st;
    if (batch < 0 || num_heads <= 0 || num_slots < 0) return KDA_ERR_INVALID_ARG;
    if ((int64_t)batch * num_heads > INT32_MAX || (int64_t)num_slots * num_heads > INT32_MAX)
        return KDA_ERR_UNSUPPORTED;
    if (batch == 0) return KDA_OK;
    if (!q || !k || !v || !log_alpha || !beta || !state_pool || !slots || !o) return KDA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(log_alpha, scalar_gate ? 4 : 16) ||
        !aligned(o, 16) || !aligned(state_pool, 16) || !aligned(beta, 4) || !aligned(slots, 4) ||
        (device_errors && !aligned(device_errors, 4)))
        return KDA_ERR_INVALID_ARG;
    st = check_device();
    if (st != KDA_OK) return st;
    kda::DecodeProblem p;
    p.q = q; p.k = k; p.v = v; p.log_alpha = log_alpha; p.beta = beta;
    p.batch = batch; p.num_heads = num_heads; p.d = d_k; p.dtype = dtype;
    p.state = state_pool; p.o = o; p.stream = static_cast<cudaStream_t>(stream);
    p.slots = slots; p.num_slots = num_slots; p.errors = device_errors;
    p.scalar_gate = scalar_gate;
    p.qk_l2norm = (flags & KDA_FLAG_QK_L2NORM) != 0;
    return kda::launch_decode(p) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_decode_step_ex(const void *q, const void *k, const void *v, const float *log_alpha,
                                const float *beta, int32_t batch, int32_t num_heads, int32_t d_k,
                                int32_t d_v, kda_dtype_t dtype, float *state, void *o, void *stream,
                                uint32_t flags)
{
    if (!flags_valid(flags)) return KDA_ERR_INVALID_ARG;
    const bool scalar_gate = (flags & KDA_FLAG_SCALAR_GATE) != 0;
    kda_status_t st = check_shape(d_k, d_v, dtype);
    if (st != KDA_OK) return st;
    if (batch < 0 || num_heads <= 0) return KDA_ERR_INVALID_ARG;
    if ((int64_t)batch * num_heads > INT32_MAX) return KDA_ERR_UNSUPPORTED;
    if (batch == 0) return KDA_OK;  // nothing to read or write; pointers may be NULL
    if (!q || !k || !v || !log_alpha || !beta || !state || !o) return KDA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(log_alpha, scalar_gate ? 4 : 16) ||
        !aligned(o, 16) || !aligned(state, 16) || !aligned(beta, 4))
        return KDA_ERR_INVALID_ARG;
    st = check_device();
    if (st != KDA_OK) return st;
    kda::DecodeProblem p;
    p.q = q; p.k = k; p.v = v; p.log_alpha = log_alpha; p.beta = beta;
    p.batch = batch; p.num_heads = num_heads; p.d = d_k; p.dtype = dtype;
    p.state = state; p.o = o; p.stream = static_cast<cudaStream_t>(stream);
    p.scalar_gate = scalar_gate;
    p.qk_l2norm = (flags & KDA_FLAG_QK_L2NORM) != 0;
    return kda::launch_decode(p) == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

kda_status_t kda_decode_step(const void *q, const void *k, const void *v, const float *log_alpha,
                             const float *beta, int32_t batch, int32_t num_heads, int32_t d_k,
                             int32_t d_v, kda_dtype_t dtype, float *state, void *o, void *stream)
{
    return kda_decode_step_ex(q, k, v, log_alpha, beta, batch, num_heads, d_k, d_v, dtype, state, o,
                              stream, 0u);
}

kda_status_t kda_read_device_status(void *workspace, void *stream)
{
    if (!workspace || !aligned(workspace, 256)) return KDA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (cudaMemsetAsync(workspace, 0, sizeof(word), s) != cudaSuccess) return KDA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KDA_ERR_CUDA;
    if (word & (kda::DEV_ERR_SEQLENS | kda::DEV_ERR_SLOT)) return KDA_ERR_INVALID_ARG;
    if (word & kda::DEV_ERR_TIMEOUT) return KDA_ERR_TIMEOUT;
    if (word & kda::DEV_ERR_DECAY) return KDA_ERR_DECAY_RANGE;
    if (word & kda::DEV_ERR_RANGE) return KDA_ERR_VALUE_RANGE;
    return KDA_OK;
}

const char *kda_status_string(kda_status_t status)
{
    switch (status) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: unsupported shape, dtype or device";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA: CUDA runtime or launch failure";
    case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT: a bounded device-side wait expired";
    case KDA_ERR_DECAY_RANGE:
        return "KDA_ERR_DECAY_RANGE: in-chunk cumulative log-decay outside the supported range";
    case KDA_ERR_VALUE_RANGE:
        return "KDA_ERR_VALUE_RANGE: a value held in fp16 left the fp16 range";
    }
    return "KDA: unknown status";
}

}  // extern "C"
