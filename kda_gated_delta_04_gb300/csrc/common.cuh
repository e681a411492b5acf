// common.cuh -- internal definitions shared by libkda's CUDA translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

// Bits of the device-side error word at the head of the prefill workspace.
enum : uint32_t {
    DEV_ERR_SEQLENS = 1u,  // cu_seqlens is not a prefix sum ending at total_tokens
    DEV_ERR_TIMEOUT = 2u,  // a bounded mbarrier / flag wait gave up
    DEV_ERR_DECAY = 4u,    // |in-chunk cumulative log-decay| exceeded the supported range
    DEV_ERR_RANGE = 8u,    // a value kept in fp16 left the fp16 range
    DEV_ERR_SLOT = 16u,    // a state-slot index outside [0, num_slots)
};

constexpr int kChunk = KDA_CHUNK;
constexpr size_t kWorkspaceHeader = 256;  // status word, padded
constexpr float kQkNormEps = 1e-12f;       // floor of the q / k row norm (KDA_FLAG_QK_L2NORM)

// Everything a prefill launch needs, already validated on the host.
// Where each sequence's states live.  Dense (fin == null): entry n of init_state and of
// final_state.  A state pool of num entries: init[n] (-1, or init == null: start from zero)
// and fin[n] (-1: not stored).
struct StateSlots {
    const int32_t *init = nullptr, *fin = nullptr;
    int64_t num = 0;
};

// Sequence-split state pass (bf16, d = 128, few (sequence, head) units): every sequence's
// chunks are cut into segments of lseg chunks, each a "virtual sequence" v.  A transition
// pass gives each segment but the last its affine map S_end = M_v S_start + R_v, a combine
// kernel chains the maps into every segment's true start state, and the state pass then
// runs all segments at once.  lseg == 0: no split.  Every pointer is workspace.
struct SeqSplit {
    int lseg = 0;                // chunks per segment
    int nv_max = 0;              // bound on the number of segments (grid extent)
    int32_t *vcu = nullptr;      // [nv_max + 2] token start of each segment (then the end)
    int32_t *vcc = nullptr;      // [nv_max + 2] first global chunk of each segment
    int32_t *vorder = nullptr;   // [nv_max]     segment processed by grid index z
    int32_t *seg_first = nullptr;  // [num_seqs + 1] first segment of each sequence
    int32_t *init_src = nullptr;   // [num_seqs]   the sequence's initial-state entry, -1 = zero
    int32_t *fin_a = nullptr;    // [nv_max + 1] transition-pass store slot (-1: last segment)
    int32_t *init_c = nullptr;   // [nv_max + 1] state-pass start slot in `start`
    int32_t *fin_c = nullptr;    // [nv_max + 1] state-pass final slot (the sequence's, last segment only)
    float *R = nullptr, *M = nullptr, *start = nullptr;  // [nv_max, H, d, d] fp32 each
    void *vzero = nullptr;       // [H, d] bf16 zeros: the value rows of the transition pass
};

struct PrefillProblem {
    const void *q, *k, *v;
    const float *log_alpha, *beta;
    const int32_t *cu_seqlens;  // may be null: one sequence of total_tokens tokens
    int num_seqs;
    int64_t total_tokens;
    int num_heads, d;           // d = d_k = d_v
    kda_dtype_t dtype;
    const float *init_state;    // may be null
    void *o;
    float *final_state;
    uint32_t *status;           // workspace word
    int32_t *order;             // workspace: sequence processing order (longest first)
    int32_t *cc;                // workspace: first chunk of each sequence [num_seqs + 1], or null
    int2 *desc = nullptr;       // workspace: per packed chunk g < chunk_bound, (first token, rows); or null
    int chunk_bound = 0;        // total_tokens / 64 + num_seqs, a bound on the packed chunk count
    void *records;              // workspace: per chunk-head records of the two-kernel path, or null
    bool scalar_gate = false;   // log_alpha is [T, H]: one decay per token-head for every key channel
    StateSlots slots;           // state pool indices, or none (dense states)
    SeqSplit split;             // sequence-split state pass, or none
    bool qk_l2norm = false;     // q, k rows are normalised in the kernels
    // bounded records (two-kernel path): records for seg_chunks packed chunks at a time, the
    // pass run segment by segment; a sequence cut at a segment boundary carries its state in
    // carry (two [num_heads, d, d] fp32 buffers, alternating by segment).  0: unsegmented.
    int seg_chunks = 0;
    float *carry = nullptr;
    // a ready flag and a copy count per chunk-head record ([chunk_bound, num_heads] each) and
    // one item counter after them, zeroed by the schedule kernel: the streamed prefill
    // publishes each record through its flag and frees its slot through its count.  Null:
    // no streaming.
    int *flags = nullptr;
    // streamed prefill: records kept for ring_chunks packed chunks (slot g mod ring_chunks);
    // 0 or chunk_bound: one slot per chunk (a workspace that holds every record)
    int ring_chunks = 0;
    // stream whenever the launch holds the walkers (KDA_FLAG_STREAM), not only where the
    // streamed form is the faster one
    bool stream_force = false;
    cudaStream_t stream;
};

// The part of the packed chunk range one launch of the state pass walks: chunks
// [g_lo, g_hi) (records indexed from g_lo); a sequence that began in an earlier segment
// starts from carry_in[head], one that goes on past g_hi ends in carry_out[head].
struct StateSegment {
    int g_lo = 0, g_hi = 0x7fffffff;
    const float *carry_in = nullptr;
    float *carry_out = nullptr;
};

struct DecodeProblem {
    const void *q, *k, *v;
    const float *log_alpha, *beta;
    int batch, num_heads, d;
    kda_dtype_t dtype;
    float *state;
    void *o;
    cudaStream_t stream;
    // paged state (optional): sequence b's state is slot slots[b] of `state`, which then
    // holds num_slots x num_heads states; out-of-range slots are skipped and reported in *errors
    const int32_t *slots = nullptr;
    int num_slots = 0;
    uint32_t *errors = nullptr;
    bool scalar_gate = false;   // log_alpha is [B, H]: one decay per sequence-head for every key channel
    bool qk_l2norm = false;     // q, k rows are normalised in the kernel
};

// Launchers (each returns the launch error, cudaSuccess when enqueued).
cudaError_t launch_prefill_prep(const PrefillProblem &p);
cudaError_t launch_prefill_simt(const PrefillProblem &p);
bool prefill_tc_supported(const PrefillProblem &p);  // bf16, d = 128, 0 < total_tokens < 2^31
cudaError_t launch_prefill_tc(const PrefillProblem &p);
// Two-kernel tensor-core prefill (needs p.cc and p.records).
size_t prefill_split_records_bytes(int64_t total_tokens, int num_seqs, int num_heads);
// bytes of one (chunk, head) record of the two-kernel path
size_t prefill_split_record_bytes();
// `mid` (may be null) is recorded on p.stream between the chunk kernel and the state kernel
// (after the streamed kernel, when that one runs).
cudaError_t launch_prefill_split(const PrefillProblem &p, const int32_t *cc, void *records,
                                 cudaEvent_t mid = nullptr);
// Whether launch_prefill_split runs the streamed kernel (chunk work and state walk in one
// grid) for p: ready flags given, no sequence split, no segments, and prefill_stream_fits.
bool prefill_stream_eligible(const PrefillProblem &p);
// Whether the streamed kernel takes a problem of `units` (sequence, head) units of about
// `chunks_per_unit` chunks each on the current device: the launch holds two walker CTAs per
// unit beside at least one worker CTA per SM, and (unless `force`) there are enough units
// for the streamed form to be the faster one at that length.
bool prefill_stream_fits(int64_t units, int64_t chunks_per_unit, bool force);
// Fewest packed chunks whose records a bounded workspace must hold for the streamed prefill
// to run over a ring of them (fewer: the two kernels in segments).
constexpr int kStreamRingMin = KDA_STREAM_RING_MIN;
// The mean chunk count of a sequence, ceil(ceil(total_tokens / num_seqs) / 64) (0 with no
// sequences).
int64_t mean_chunks_per_sequence(int32_t num_seqs, int64_t total_tokens);
cudaError_t launch_decode(const DecodeProblem &p);
// Measurement only: the tensor-core product groups of the chunk kernel (pass 0) or the state
// kernel (pass 1) back to back on resident operands; synchronises `stream`; executed TFLOP/s.
cudaError_t diag_tensor_phases(int pass, int reps, uint32_t *status, cudaStream_t stream, double *tflops);
// Sequence-split state pass: segment length for a problem shape (0: no split), the bound on
// its segment count, the workspace it needs, and its two small kernels (segment tables after
// the schedule kernel; start states after the transition pass).
int seqsplit_lseg(int num_seqs, int64_t total_tokens, int num_heads);
int seqsplit_nv_max(int lseg, int num_seqs, int64_t total_tokens);
size_t seqsplit_bytes(int num_seqs, int64_t total_tokens, int num_heads);
void seqsplit_carve(SeqSplit &s, int num_seqs, int64_t total_tokens, int num_heads, char *ws);
cudaError_t launch_seqsplit_plan(const PrefillProblem &p);
cudaError_t launch_seqsplit_combine(const PrefillProblem &p);

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ float load_io(const float *p) { return *p; }
__device__ __forceinline__ float load_io(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store_io(float *p, float x) { *p = x; }
__device__ __forceinline__ void store_io(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }
// four consecutive values (p 16-byte aligned for fp32, 8-byte aligned for bf16)
__device__ __forceinline__ void load_io4(const float *p, float (&x)[4])
{
    const float4 a = *reinterpret_cast<const float4 *>(p);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
}
__device__ __forceinline__ void load_io4(const __nv_bfloat16 *p, float (&x)[4])
{
    const uint2 a = *reinterpret_cast<const uint2 *>(p);
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&a.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&a.y));
    x[0] = lo.x; x[1] = lo.y; x[2] = hi.x; x[3] = hi.y;
}
__device__ __forceinline__ void store_io4(float *p, const float (&x)[4])
{
    *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
}
__device__ __forceinline__ void store_io4(__nv_bfloat16 *p, const float (&x)[4])
{
    __nv_bfloat162 lo = __floats2bfloat162_rn(x[0], x[1]), hi = __floats2bfloat162_rn(x[2], x[3]);
    *reinterpret_cast<uint2 *>(p) = make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
}

// Four consecutive elements (16-byte aligned for fp32, 8-byte for bf16).
__device__ __forceinline__ float4 load4_io(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 load4_io(const __nv_bfloat16 *p)
{
    const uint2 raw = *reinterpret_cast<const uint2 *>(p);
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&raw.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&raw.y);
    const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    return make_float4(fa.x, fa.y, fb.x, fb.y);
}
__device__ __forceinline__ void store4_io(float *p, float4 x) { *reinterpret_cast<float4 *>(p) = x; }
__device__ __forceinline__ void store4_io(__nv_bfloat16 *p, float4 x)
{
    __nv_bfloat162 a = __floats2bfloat162_rn(x.x, x.y), b = __floats2bfloat162_rn(x.z, x.w);
    uint2 raw;
    raw.x = *reinterpret_cast<uint32_t *>(&a);
    raw.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = raw;
}

// Token range [t0, t1) of sequence n, clamped to [0, total] so that a malformed
// cu_seqlens can never send a kernel outside the buffers.
__device__ __forceinline__ void seq_range(const int32_t *cu, int n, int64_t total, int64_t &t0,
                                          int64_t &t1)
{
    if (!cu) { t0 = 0; t1 = total; return; }
    int64_t a = cu[n], b = cu[n + 1];
    a = a < 0 ? 0 : (a > total ? total : a);
    b = b < a ? a : (b > total ? total : b);
    t0 = a;
    t1 = b;
}

// Sequence n's initial-state entry si (-1: zero) and final-state entry sf (-1: not stored).
// Returns false for a pool slot out of range; the sequence then starts from zero and its final
// state is not written.
__device__ __forceinline__ bool state_entries(const StateSlots &s, int n, bool has_init, int64_t &si,
                                              int64_t &sf)
{
    if (!s.fin) {
        si = has_init ? n : -1;
        sf = n;
        return true;
    }
    si = s.init ? s.init[n] : -1;
    sf = s.fin[n];
    if (si >= -1 && si < s.num && sf >= -1 && sf < s.num) return true;
    si = sf = -1;
    return false;
}

}  // namespace kda
