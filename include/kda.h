/*
 * kda.h -- C ABI of libkda: the Kimi Delta Attention (KDA) recurrence on one GPU.
 *
 * The operation (per sequence n, head h; key channel i < d_k, value channel j < d_v):
 *
 *     decayed   = Diag(alpha_t) S_{t-1}                 alpha_t = exp(log_alpha[t,h,:])
 *     S_t       = decayed + beta_t k_t (v_t - decayed^T k_t)^T
 *     o_t       = S_t^T q_t / sqrt(d_k)
 *
 * Sources: "Day 19, linear attention & KDA" (ai.air7.fun, k3-course-30), section 3:
 * the update decays the state per channel first, then writes back only the
 * prediction error scaled by beta_t; "K3 attention, three-piece set"
 * (yeyulingfeng.com), KDA paragraphs: the (I - beta_t k_t k_t^T) factor, the
 * per-key-channel gate Diag(alpha_t), a fixed-size d_k x d_v state per head,
 * and the chunkwise-parallel deployment form; "From 124M to 2.8T"
 * (ciyuanerhao.com), chapter 4: the gate has one value per key channel and
 * scales the key rows of S.  The 1/sqrt(d_k) output scale is this library's
 * definition (the pages state none).  q and k are expected to be L2-normalised
 * by the caller (the pages normalise them inside the layer, before this step),
 * unless KDA_FLAG_QK_L2NORM asks the kernels to do it.
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller, row-major and
 *    contiguous (last dimension has stride 1), 16-byte aligned; kda_prefill_host
 *    alone takes host buffers.  The library allocates no device memory; its only
 *    global state is cached device attributes and, for kda_prefill_host, two
 *    streams and a few events per device.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*, NULL =
 *    the legacy default stream) and never synchronise, except
 *    kda_read_device_status.
 *  - Argument errors are reported synchronously, before anything is enqueued.
 *    A failed kernel launch returns KDA_ERR_CUDA.  Errors detected on the device
 *    (see kda_prefill) are recorded in the workspace and read back with
 *    kda_read_device_status.  Nothing aborts or throws across the ABI.
 *  - Supported shapes: d_k == d_v == 64 or 128, with q/k/v/o stored as bf16 or
 *    fp32 (kda_dtype_t); log_alpha, beta and every state are fp32.  Other shapes
 *    return KDA_ERR_UNSUPPORTED.
 */
#ifndef LIBKDA_KDA_H
#define LIBKDA_KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misalignment, bad cu_seqlens  */
    KDA_ERR_UNSUPPORTED = 2,  /* valid but not implemented shape / dtype / device       */
    KDA_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed            */
    KDA_ERR_TIMEOUT = 4,      /* a bounded device-side wait expired (no hang, no trap)  */
    KDA_ERR_DECAY_RANGE = 5,  /* a chunk's cumulative log-decay left the supported range */
    KDA_ERR_VALUE_RANGE = 6   /* a value the bf16 d = 128 fast path holds in fp16 left    */
                              /* the fp16 range (|x| > 65504, or not finite)            */
} kda_status_t;

typedef enum { KDA_DTYPE_BF16 = 0, KDA_DTYPE_F32 = 1 } kda_dtype_t;

/* Chunk length of the chunkwise prefill (tokens). */
#define KDA_CHUNK 64
/* Lower bound on sum(log_alpha) over any 64-token chunk, per key channel, that
 * kda_prefill supports: its chunk factorisation forms exp(-g) for the in-chunk
 * cumulative log-decay g, which must stay finite in fp32. */
#define KDA_MIN_CHUNK_LOG_DECAY (-80.0f)

/*
 * Bytes of device workspace for the fastest kda_prefill path on this problem.
 * For bf16 q/k/v at d_k = d_v = 128 that is the tensor-core path with per-chunk
 * records: a status word, a sequence schedule, the first chunk of each sequence,
 * one 8-byte descriptor per chunk, a 4-byte ready flag per record (for the streamed
 * form, KDA_FLAG_NO_STREAM) and one item counter, and one 74,240-byte record per
 * (64-token chunk, head), at most (total_tokens / 64 + num_seqs) * num_heads
 * records (about 1.2 KB per token per head); when the problem has so few
 * (sequence, head) units that the
 * state pass runs in segments (KDA_FLAG_NO_SEQ_SPLIT), also three fp32 states
 * per segment and head.  For other shapes it equals
 * KDA_PREFILL_MIN_WORKSPACE(num_seqs).
 * Pure host arithmetic; returns 0 only for negative sizes.
 */
#define KDA_PREFILL_MIN_WORKSPACE(num_seqs) \
    (256u + ((((size_t)(num_seqs)) * 4u + 1u + 255u) / 256u) * 256u)
size_t kda_prefill_workspace_size(int32_t num_seqs, int64_t total_tokens, int32_t num_heads,
                                  int32_t d_k, int32_t d_v, kda_dtype_t dtype);

/*
 * Workspace bytes for the two-kernel prefill with its per-chunk records bounded (the
 * chunkwise form of "From 124M to 2.8T", chapter 3, run over a bounded window of chunks
 * at a time).  kda_prefill_workspace_size covers the records of every packed 64-token
 * chunk, about 1.16 KB per token-head (a one-million-token, 32-head prompt would need
 * about 39 GB).  With this size instead the records cover at most segment_chunks packed
 * chunks: kda_prefill then runs the chunk kernel and the state pass one segment of
 * packed chunks after the other, and a sequence cut at a segment boundary carries its
 * fp32 state to the next segment in the workspace (two [num_heads, 128, 128] fp32
 * buffers).  The results are bit for bit those of the full workspace without the
 * sequence split (KDA_FLAG_NO_SEQ_SPLIT); each extra segment costs two more launches.
 * Any workspace between this size for segment_chunks = 1 and kda_prefill_workspace_size
 * runs segmented, with as many chunks per segment as its records fit, when the call runs
 * the two kernels (KDA_FLAG_NO_STREAM, or too few (sequence, head) units to stream); where
 * the call would stream, a bounded workspace runs the streamed prefill over a ring of
 * records instead (kda_prefill_workspace_size_streamed), if it holds those of at least
 * KDA_STREAM_RING_MIN chunks.
 *
 *  segment_chunks  >= 1; values past the packed chunk bound (total_tokens / 64 +
 *                  num_seqs) are clamped to it.
 *  Returns 0 for invalid arguments and for shapes the two-kernel path does not run
 *  (anything but bf16, d_k = d_v = 128, total_tokens > 0).
 */
size_t kda_prefill_workspace_size_segmented(int32_t num_seqs, int64_t total_tokens, int32_t num_heads,
                                            int32_t d_k, int32_t d_v, kda_dtype_t dtype,
                                            int64_t segment_chunks);

/*
 * Workspace bytes for the streamed prefill (chunk work and state walk in one launch, see
 * KDA_FLAG_NO_STREAM) with its records kept in a ring of ring_chunks packed chunks: the
 * record of chunk g (all heads) goes to slot g mod ring_chunks, written only once both
 * walking CTAs of chunk g - ring_chunks have copied that slot's previous record in.  The
 * chunk work then leads the walk by at most ring_chunks chunks, and the workspace no
 * longer grows with the records of every chunk (T = 65536, H = 32: about 39 MB for 16
 * chunks against 2.44 GB).  The results are bit for bit those of the streamed prefill
 * with the full workspace.  It is not faster than that: held to the walk's pace, the
 * chunk work shares the SMs with it to the end.  Any workspace between this size for
 * KDA_STREAM_RING_MIN chunks and kda_prefill_workspace_size runs this way where the call
 * streams (kda_prefill_path says so), with as many chunks as its records fit.
 *
 *  ring_chunks  >= KDA_STREAM_RING_MIN; values past the packed chunk bound
 *               (total_tokens / 64 + num_seqs) are clamped to it.
 *  Returns 0 for invalid arguments and for shapes the streamed prefill does not run
 *  (anything but bf16, d_k = d_v = 128, total_tokens > 0).
 */
#define KDA_STREAM_RING_MIN 8
size_t kda_prefill_workspace_size_streamed(int32_t num_seqs, int64_t total_tokens, int32_t num_heads,
                                           int32_t d_k, int32_t d_v, kda_dtype_t dtype, int64_t ring_chunks);

/*
 * The kernels a kda_prefill_ex call with these arguments runs (the path it takes).
 *  KDA_PATH_CUDA_CORE  fp32 I/O or d = 64: the exact CUDA-core chunk kernel
 *  KDA_PATH_FUSED      bf16, d = 128, workspace below the bounded-records size: one
 *                      tensor-core kernel per (sequence, head, value slice)
 *  KDA_PATH_TWO_KERNEL the chunk kernel, then the state pass
 *  KDA_PATH_SEQ_SPLIT  the chunk kernel, then the sequence-split state pass
 *  KDA_PATH_SEGMENTED  the chunk kernel and the state pass over segments of records
 *  KDA_PATH_STREAMED   chunk work and state walk in one launch (see KDA_FLAG_NO_STREAM),
 *                      with a bounded workspace over a ring of records
 *                      (kda_prefill_workspace_size_streamed)
 * Host arithmetic plus one device-attribute query (the SM count of the current
 * device); returns a negative kda_status_t for arguments kda_prefill_ex rejects on
 * the host.  Each path also runs the schedule kernel first.
 */
typedef enum {
    KDA_PATH_CUDA_CORE = 0,
    KDA_PATH_FUSED = 1,
    KDA_PATH_TWO_KERNEL = 2,
    KDA_PATH_SEQ_SPLIT = 3,
    KDA_PATH_SEGMENTED = 4,
    KDA_PATH_STREAMED = 5
} kda_prefill_path_t;
int32_t kda_prefill_path(int32_t num_seqs, int64_t total_tokens, int32_t num_heads, int32_t d_k,
                         int32_t d_v, kda_dtype_t dtype, size_t workspace_bytes, uint32_t flags);

/*
 * Chunkwise prefill over packed variable-length sequences ("K3 attention,
 * three-piece set": chunkwise-parallel form with WY representation and UT
 * transform; "From 124M to 2.8T", chapter 3: parallel inside a chunk, serial
 * across chunks).  Chunks of KDA_CHUNK tokens never cross a sequence boundary.
 *
 *  q, k        [total_tokens, num_heads, d_k]  dtype
 *  v           [total_tokens, num_heads, d_v]  dtype
 *  log_alpha   [total_tokens, num_heads, d_k]  fp32, finite, <= 0; per chunk and
 *              channel its sum must be >= KDA_MIN_CHUNK_LOG_DECAY
 *  beta        [total_tokens, num_heads]       fp32
 *  cu_seqlens  [num_seqs + 1] int32 device offsets: 0 = cu[0] <= ... <= cu[num_seqs]
 *              = total_tokens; NULL means one sequence of total_tokens tokens
 *              (num_seqs must then be 1)
 *  init_state  [num_seqs, num_heads, d_k, d_v] fp32, or NULL for zero states
 *  o           [total_tokens, num_heads, d_v]  dtype (written for every token), or NULL
 *              for a state-only prefill (final states only; the two-kernel path then
 *              also skips the output products)
 *  final_state [num_seqs, num_heads, d_k, d_v] fp32; may equal init_state
 *              (in-place update); a zero-length sequence gets its initial state
 *  workspace   device buffer owned by the caller, 256-byte aligned, reused by every
 *              call.  With kda_prefill_workspace_size(...) bytes or more the bf16,
 *              d = 128 prefill runs as two kernels (chunk-local products for all
 *              chunks at once, then the serial state pass; with few (sequence, head)
 *              units both in one launch, see KDA_FLAG_NO_STREAM; kda_prefill_path tells
 *              which); with less, but at least
 *              kda_prefill_workspace_size_segmented(..., 1) bytes, as the same two
 *              kernels over segments of chunks (bounded records, identical results);
 *              with at least KDA_PREFILL_MIN_WORKSPACE(num_seqs) bytes as one fused
 *              kernel (same results up to rounding order, slower).  Smaller
 *              workspaces are rejected.
 *  q, k, v, log_alpha and beta may be NULL when total_tokens == 0.
 *
 * Device-side errors (timeout of a bounded wait, a cu_seqlens array that is not
 * a valid prefix sum, a decay outside the supported range, and on the two-kernel
 * path a v value or a chunk-local product outside the fp16 range, which that
 * path keeps in fp16) do not fault: the
 * kernels clamp every access to the buffers, finish, and record the error in the
 * workspace.  Each call clears the record first; read it with
 * kda_read_device_status.  Calls that share a workspace must be ordered (same
 * stream or synchronised).
 */
kda_status_t kda_prefill(const void *q, const void *k, const void *v, const float *log_alpha,
                         const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                         int64_t total_tokens, int32_t num_heads, int32_t d_k, int32_t d_v,
                         kda_dtype_t dtype, const float *init_state, void *o, float *final_state,
                         void *workspace, size_t workspace_bytes, void *stream);

/*
 * kda_decode_step on a paged state cache: sequence b's state is slot slots[b] of
 * state_pool ([num_slots, num_heads, d_k, d_v] fp32, read and overwritten in place),
 * so a serving runtime can keep every live sequence's state in one pool and decode
 * any subset of them in one call ("Day 19", section 2: constant memory per sequence).
 *  slots          [batch] int32 device indices in [0, num_slots); they must be
 *                 distinct within a call (two sequences on one slot race)
 *  device_errors  NULL or a device uint32 that receives KDA_DEVICE_ERR_SLOT (or-ed)
 *                 when a slot is out of range; that sequence is then skipped (its o
 *                 and every pool slot are left untouched) and the others run
 *  flags          as kda_decode_step_ex (KDA_FLAG_SCALAR_GATE below)
 * Other arguments, layouts and errors as kda_decode_step.
 */
kda_status_t kda_decode_step_slots(const void *q, const void *k, const void *v, const float *log_alpha,
                                   const float *beta, int32_t batch, int32_t num_heads, int32_t d_k,
                                   int32_t d_v, kda_dtype_t dtype, float *state_pool, int32_t num_slots,
                                   const int32_t *slots, void *o, uint32_t *device_errors, void *stream,
                                   uint32_t flags);

/*
 * kda_prefill with its stages marked, for measuring them: the same arguments and
 * results, plus four CUDA events (cudaEvent_t handles passed as void*, created by
 * the caller) recorded on `stream`:
 *   events[0]  before the schedule kernel (cu_seqlens check, sequence order),
 *   events[1]  after it,
 *   events[2]  after the chunk-local kernel of the two-kernel path (on the
 *              single-kernel paths, the streamed one included, after that kernel),
 *   events[3]  after the last kernel.
 * All four are recorded even when no kernel runs.  num_events must be 4 and no
 * handle NULL, else KDA_ERR_INVALID_ARG before anything is enqueued.
 */
kda_status_t kda_prefill_events(const void *q, const void *k, const void *v, const float *log_alpha,
                                const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                                int64_t total_tokens, int32_t num_heads, int32_t d_k, int32_t d_v,
                                kda_dtype_t dtype, const float *init_state, void *o,
                                float *final_state, void *workspace, size_t workspace_bytes,
                                void *stream, void *const *events, int32_t num_events);

/* kda_prefill_events with option flags (as kda_prefill_ex); flags = 0 is kda_prefill_events. */
kda_status_t kda_prefill_events_ex(const void *q, const void *k, const void *v, const float *log_alpha,
                                   const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                                   int64_t total_tokens, int32_t num_heads, int32_t d_k, int32_t d_v,
                                   kda_dtype_t dtype, const float *init_state, void *o,
                                   float *final_state, void *workspace, size_t workspace_bytes,
                                   void *stream, void *const *events, int32_t num_events, uint32_t flags);

/*
 * Options of kda_prefill_ex / kda_decode_step_ex (bitwise or; other bits are
 * rejected with KDA_ERR_INVALID_ARG).
 *  KDA_FLAG_SCALAR_GATE  scalar-gate (Gated DeltaNet) variant: log_alpha holds one
 *                        value per token-head, [total_tokens, num_heads] fp32 (4-byte
 *                        aligned; decode: [batch, num_heads]), the decay of every key
 *                        channel ("From 124M to 2.8T", chapter 3: the scalar gate of
 *                        Gated DeltaNet; "K3 attention, three-piece set": KDA makes the
 *                        gate channel-wise).  Its chunk-prefix bound is the same.
 */
#define KDA_FLAG_SCALAR_GATE 1u
/*  KDA_FLAG_QK_L2NORM    q and k are raw (the layer's activations before their L2
 *                        normalisation): the kernels normalise every q and k row over
 *                        d_k in fp32, x / max(||x||_2, 1e-12), before the recurrence
 *                        ("K3 attention, three-piece set", KDA engineering notes: q and
 *                        k pass a short causal convolution and then L2 normalisation;
 *                        "From 124M to 2.8T", chapter 3 code: the normalisation over the
 *                        channel axis).  The 1/sqrt(d_k) output scale is unchanged. */
#define KDA_FLAG_QK_L2NORM 2u
/*  KDA_FLAG_NO_SEQ_SPLIT  keep each sequence's serial state pass in one piece.  By
 *                        default, when a bf16 d = 128 problem has so few (sequence,
 *                        head) units that the state pass would leave most SMs idle (at
 *                        most 19), sequences long enough for the split to pay (on average
 *                        at least 72 chunks of 64 tokens with up to 8 units, 15 per unit
 *                        less 50 beyond), and the workspace was sized by
 *                        kda_prefill_workspace_size for that shape, every sequence is cut
 *                        into segments of whole chunks: a
 *                        transition pass gives each segment its affine map (the
 *                        chunkwise form makes every chunk's update affine in its start
 *                        state), the maps are chained in fp32 into each segment's start
 *                        state, and the segments then run at once.  The results agree
 *                        with the unsplit pass to within rounding, not bit for bit. */
#define KDA_FLAG_NO_SEQ_SPLIT 4u
/*  KDA_FLAG_NO_STREAM     run the chunk kernel and the state pass one after the other.
 *                        By default, when a bf16 d = 128 problem has no sequence split, a
 *                        workspace that holds every record, and enough (sequence, head)
 *                        units for it to be the faster form (at most 32; at least 31 when
 *                        the sequences average up to 96 chunks of 64 tokens, 27 up to 384,
 *                        24 beyond), both run in one launch: two CTAs walk the state of
 *                        each unit (64 value columns each) while the others do the chunk
 *                        work, and each record is handed over through a ready flag in the
 *                        workspace as soon as its stores are complete.  The two forms
 *                        agree to within rounding, not bit for bit (the walk forms its
 *                        products transposed).  The walking CTAs wait for records that
 *                        the others produce (and, over a ring of records, those wait for
 *                        the walk to free a slot), so the launch needs SM slots for both:
 *                        if kernels on other streams hold all but a few slots for longer
 *                        than the device-side wait limit (2 s), the call gives up with
 *                        KDA_ERR_TIMEOUT instead of hanging.  The two-kernel form has no
 *                        such dependence; pass this flag where the GPU is shared that way
 *                        (with a bounded workspace it then runs the two kernels in
 *                        segments). */
#define KDA_FLAG_NO_STREAM 8u
/*  KDA_FLAG_STREAM        run both in one launch whenever the launch holds the walking CTAs
 *                        (1 to 32 units on a 152-SM GB300; same conditions otherwise),
 *                        however few the units.  Passing it with KDA_FLAG_NO_STREAM is
 *                        KDA_ERR_INVALID_ARG. */
#define KDA_FLAG_STREAM 16u

/* kda_prefill with options (flags above); flags = 0 is kda_prefill. */
kda_status_t kda_prefill_ex(const void *q, const void *k, const void *v, const float *log_alpha,
                            const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                            int64_t total_tokens, int32_t num_heads, int32_t d_k, int32_t d_v,
                            kda_dtype_t dtype, const float *init_state, void *o, float *final_state,
                            void *workspace, size_t workspace_bytes, void *stream, uint32_t flags);

/*
 * kda_prefill against the paged state cache of kda_decode_step_slots: sequence n
 * starts from slot init_slots[n] of state_pool and its final state is written to
 * slot final_slots[n], so a prompt is prefilled straight into the pool that decode
 * then continues from ("Day 19", section 2: a fixed-size state per sequence carried
 * from the prompt into generation).
 *  state_pool   [num_slots, num_heads, d_k, d_v] fp32, 16-byte aligned
 *  init_slots   [num_seqs] int32 device, or NULL (every sequence starts from zero);
 *               an entry -1 starts that sequence from zero
 *  final_slots  [num_seqs] int32 device, required; an entry -1 stores no final
 *               state for that sequence
 * A sequence may read and write the same slot (it is updated in place).  Final
 * slots must be distinct, and no sequence may start from another sequence's final
 * slot (the two would race).  A slot outside [0, num_slots) (init: also -1) is a
 * device-side error (KDA_DEVICE_ERR_SLOT; kda_read_device_status returns
 * KDA_ERR_INVALID_ARG): that sequence starts from zero, its outputs are computed
 * and its final state is not written; the other sequences are not affected.
 * Other arguments (flags included), layouts and errors as kda_prefill_ex.
 */
kda_status_t kda_prefill_slots(const void *q, const void *k, const void *v, const float *log_alpha,
                               const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                               int64_t total_tokens, int32_t num_heads, int32_t d_k, int32_t d_v,
                               kda_dtype_t dtype, float *state_pool, int32_t num_slots,
                               const int32_t *init_slots, const int32_t *final_slots, void *o,
                               void *workspace, size_t workspace_bytes, void *stream, uint32_t flags);

/*
 * One decode step for `batch` sequences x num_heads heads: the recurrence for a
 * single new token per sequence, applied to the caller's state in place
 * ("Day 19", section 2: constant memory and O(1) work per generated token;
 * "K3 attention, three-piece set": fixed-size d_k x d_v state per KDA head).
 *
 *  q, k, log_alpha  [batch, num_heads, d_k]  (q, k dtype; log_alpha fp32)
 *  v                [batch, num_heads, d_v]  dtype
 *  beta             [batch, num_heads]       fp32
 *  state            [batch, num_heads, d_k, d_v] fp32, read and overwritten
 *  o                [batch, num_heads, d_v]  dtype
 * No workspace; no device-side error conditions.  batch == 0 is a no-op that
 * enqueues nothing (every pointer may then be NULL).
 */
kda_status_t kda_decode_step(const void *q, const void *k, const void *v, const float *log_alpha,
                             const float *beta, int32_t batch, int32_t num_heads, int32_t d_k,
                             int32_t d_v, kda_dtype_t dtype, float *state, void *o, void *stream);

/* kda_decode_step with options (flags above); flags = 0 is kda_decode_step. */
kda_status_t kda_decode_step_ex(const void *q, const void *k, const void *v, const float *log_alpha,
                                const float *beta, int32_t batch, int32_t num_heads, int32_t d_k,
                                int32_t d_v, kda_dtype_t dtype, float *state, void *o, void *stream,
                                uint32_t flags);

/*
 * Synchronises `stream`, reads the device-side error record of the last
 * kda_prefill that used `workspace`, clears it, and returns the first error
 * found (KDA_OK when none).  Explicit synchronisation point.
 */
kda_status_t kda_read_device_status(void *workspace, void *stream);

/*
 * kda_prefill_no_alloc -- kda_prefill without a caller-provided workspace.
 * The pages have no counterpart to this entry point; it is a library facility.
 *
 * Who it is for: callers that cannot allocate device memory when they call the
 * prefill, so cannot hand kda_prefill its workspace.  Examples are a serving
 * runtime that carves all GPU memory out of a pool sized at start-up and
 * forbids allocations afterwards, and a latency-critical path that must not
 * call cudaMalloc (which may synchronise the whole device).
 *
 * What it does: exactly what kda_prefill does, with the same arguments, checks,
 * kernels and results, except that the workspace is a fixed device array built
 * into libkda.  That array is KDA_NO_ALLOC_SCRATCH_BYTES bytes; every GPU that
 * loads the library holds it until the process exits.  The call allocates
 * nothing: no cudaMalloc, cudaFree or allocating library routine.
 *
 *  num_seqs      at most KDA_NO_ALLOC_MAX_SEQS; larger values return
 *                KDA_ERR_UNSUPPORTED and enqueue nothing (use kda_prefill).
 *  device_errors optional DEVICE pointer to one uint32; when not NULL it receives
 *                this call's device-side error bits (0 = none, otherwise an OR of
 *                KDA_DEVICE_ERR_*), copied on `stream` after the prefill; a call
 *                with num_seqs == 0 runs no kernel and writes 0 there.
 *
 * The first call on each device looks up the array's device address (with that
 * device current) and caches it; make that first call before any stream capture
 * begins.  The cached address is not valid across cudaDeviceReset (the library's
 * module, and with it the array, may come back at another address): do not call
 * this entry point on a device after resetting it in the same process.  All calls share the one array and each call reinitialises it (error
 * word and schedule) before use, so calls ordered on one stream are fine, but
 * calls whose work can overlap on the GPU (unordered streams) race on the array
 * and must be serialised by the caller.
 */
#define KDA_NO_ALLOC_MAX_SEQS 4096
#define KDA_NO_ALLOC_SCRATCH_BYTES (512 + 4 * KDA_NO_ALLOC_MAX_SEQS) /* 16,896 */
#define KDA_DEVICE_ERR_SEQLENS 1u /* cu_seqlens is not a prefix sum ending at total_tokens */
#define KDA_DEVICE_ERR_TIMEOUT 2u /* a bounded device-side wait expired                   */
#define KDA_DEVICE_ERR_DECAY 4u   /* a chunk's cumulative log-decay left the supported range */
#define KDA_DEVICE_ERR_RANGE 8u   /* a value held in fp16 left the fp16 range (two-kernel path) */
#define KDA_DEVICE_ERR_SLOT 16u   /* a state-pool slot index out of range (the _slots calls)   */
kda_status_t kda_prefill_no_alloc(const void *q, const void *k, const void *v,
                                  const float *log_alpha, const float *beta,
                                  const int32_t *cu_seqlens, int32_t num_seqs,
                                  int64_t total_tokens, int32_t num_heads, int32_t d_k,
                                  int32_t d_v, kda_dtype_t dtype, const float *init_state,
                                  void *o, float *final_state, uint32_t *device_errors,
                                  void *stream);

/*
 * Self-test of the device-side failure path (the pages have no counterpart; it
 * checks this library's own error handling).  Enqueues on `stream` one small
 * kernel whose threads wait, one sleeping and one polling, on a barrier that
 * nothing ever completes.  Each wait gives up after limit_ns nanoseconds of wall
 * time (0 < limit_ns <= 1e9, else KDA_ERR_INVALID_ARG) exactly as every wait in
 * the prefill kernels does, and the kernel records the give-up in the status
 * word at the start of `workspace` (256-byte aligned device memory, at least 4
 * bytes; the word is cleared first).  kda_read_device_status(workspace, stream)
 * then returns KDA_ERR_TIMEOUT.  Nothing faults or hangs; the context stays usable.
 */
kda_status_t kda_selftest_bounded_wait(void *workspace, uint64_t limit_ns, void *stream);

/*
 * kda_prefill from host buffers, for a caller whose inputs and outputs live in host memory:
 * the prompt is cut into up to four segments at chunk boundaries (64-token multiples from the
 * start of the sequence a cut falls in; prompts under 2,048 tokens are not cut; the last
 * segment is about 1/16 of the prompt, so little follows the last upload), and the
 * host->device copies of later segments, the prefill of earlier ones and the device->host
 * copies of their outputs overlap on two internal streams.  Because every chunk and every
 * serial state step is the one kda_prefill would run, o and the final states are bit for bit
 * those of kda_prefill_ex with the same flags on the same shape of problem per segment (with
 * KDA_FLAG_NO_SEQ_SPLIT, or a problem too large for the sequence split, on every shape).
 *  q, k, v, log_alpha, beta, o   host memory, the layouts of kda_prefill; page-locked
 *                                memory lets the copies overlap (pageable memory works, slower)
 *  cu_seqlens                    HOST int32 [num_seqs + 1] (checked on the host), or NULL for
 *                                one sequence
 *  init_state                    host [num_seqs, H, d, d] fp32, or NULL (zero)
 *  final_state                   host [num_seqs, H, d, d] fp32, required
 *  o                             may be NULL (final states only)
 *  device_buffer, device_bytes   256-byte aligned device memory of at least
 *                                kda_prefill_host_buffer_size(...) bytes; its first word
 *                                collects the device-side errors of the call: read it with
 *                                kda_read_device_status(device_buffer, stream)
 *  flags                         KDA_FLAG_QK_L2NORM and KDA_FLAG_NO_SEQ_SPLIT
 *                                (KDA_FLAG_SCALAR_GATE: KDA_ERR_UNSUPPORTED)
 * Asynchronous on `stream`: the host buffers must stay valid, and the outputs unread, until
 * the stream is synchronised.  Calls from several host threads are serialised while they
 * enqueue.  Errors as kda_prefill; a cu_seqlens that is not a prefix sum from 0 to
 * total_tokens is KDA_ERR_INVALID_ARG here (it is on the host).
 */
kda_status_t kda_prefill_host(const void *q, const void *k, const void *v, const float *log_alpha,
                              const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                              int64_t total_tokens, int32_t num_heads, int32_t d_k, int32_t d_v,
                              kda_dtype_t dtype, const float *init_state, void *o, float *final_state,
                              void *device_buffer, size_t device_bytes, void *stream, uint32_t flags);

/* Device bytes kda_prefill_host needs for this problem (cu_seqlens on the host, or NULL for
 * one sequence); 0 for invalid arguments. */
size_t kda_prefill_host_buffer_size(const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                                    int32_t num_heads, int32_t d_k, int32_t d_v, kda_dtype_t dtype);

/* The segment boundaries kda_prefill_host uses: writes bounds[0] = 0 < ... < bounds[n] =
 * total_tokens and returns n (0 for no tokens), or -1 for invalid arguments.  max_bounds
 * must be at least 5. */
int32_t kda_prefill_host_segments(const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                                  int64_t *bounds, int32_t max_bounds);

/*
 * Measurement only (no counterpart on the pages): the tensor-core product groups of one
 * two-kernel-path prefill kernel, issued back to back by the kernel's own issue routines
 * on a constant operand image resident in shared memory, with no epilogues, no waits
 * between groups and no global traffic.  It isolates how fast the tensor pipe runs the
 * prefill's GEMM phases, apart from the work between them.
 *  pass  0: the chunk kernel's groups of one (chunk, head) item (k-k and q-k, W, P2, the
 *           three-term P, N, Q''), 9,961,472 executed FLOP per repetition, two CTAs per SM;
 *        1: the state kernel's chain and output groups of one chunk and 64-column value
 *           slice (P V, N S, P2 V, Q' S), 4,718,592 FLOP per repetition, one CTA per SM,
 *           each group issued by a thread of its own warp;
 *        2: the streamed kernel's walk group of one chunk and 64 value columns (the same
 *           four products transposed, S^T read from TMEM, as one M = 64, N = 192 group),
 *           4,718,592 FLOP per repetition, one CTA per SM, one issuing thread
 *  reps      repetitions per CTA, 1 .. 2^20
 *  workspace 256-byte aligned device memory of at least 4 bytes (status word, cleared)
 *  tflops    receives the executed TFLOP/s over the whole GPU (CUDA events on `stream`)
 * Synchronises `stream`.  KDA_ERR_TIMEOUT if a bounded wait gave up.
 */
kda_status_t kda_diag_tensor_phases(int32_t pass, int32_t reps, void *workspace, void *stream, double *tflops);

/* Static, human-readable name of a status code (never NULL). */
const char *kda_status_string(kda_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* LIBKDA_KDA_H */
