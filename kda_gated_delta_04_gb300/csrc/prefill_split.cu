// prefill_split.cu -- the tensor-core prefill as two kernels (bf16 q/k/v,
// d_k = d_v = 128, fp32 state), sm_103a.
//
// Everything in a 64-token chunk that does not involve the running state (the
// decay prefix, the decayed operands, the k-k / q-k matrices, the UT solve and
// the WY factor W) is independent across chunks ("From 124M to 2.8T", chapter
// 3: parallel inside a chunk; "K3 attention, three-piece set": WY
// representation + UT transform).  So it runs in its own kernel, one CTA per
// (chunk, head), over every chunk at once, and leaves a record per chunk-head in
// the workspace.  The state kernel then only walks the serial part, one CTA per
// (sequence, head, 32-column value slice), bulk-loading each record a chunk
// ahead:
//
//   chunk kernel   (as in the fused kernel)  record = [-W ; Qg] bf16, Ki^T tf32,
//                  T' = (I + A)^-1 diag(beta) tf32, Aqk bf16, e^{g_last}
//   state kernel   D_u  = T' V (tf32) - W S (bf16)          = u       (M = 64)
//                  D_o  = Qg S (bf16) + Aqk u (bf16)         = o       (M = 64)
//                  D5   = Ki^T u (tf32);  S <- e^{g_last} (S + D5)     (M = 128)
//
// Records are the chunk kernel's shared-memory operand images, byte for byte,
// so the state kernel feeds them to the MMAs without re-packing.
#include "tc_common.cuh"

namespace kda {
namespace {

using namespace ptx;
using namespace tc;

// Record of one chunk-head (also the contiguous tail of the chunk kernel's
// shared memory and the head of each state-kernel stage).
constexpr uint32_t R_O1 = 0;       // [-W ; Qg] bf16 K-major, 2 panels x 128 rows
constexpr uint32_t R_O3 = 32768;   // Ki^T tf32 K-major, 2 panels x 128 rows
constexpr uint32_t R_TT = 65536;   // T' tf32 K-major, 2 panels x 64 rows
constexpr uint32_t R_AQ = 81920;   // Aqk bf16 K-major, 64 rows
constexpr uint32_t R_GM = 90112;   // e^{g_last}, 128 fp32
constexpr uint32_t kRecBytes = 90624;
static_assert(kRecBytes % 16 == 0, "records are moved by bulk copies");

// Chunk kernel: 256 threads and 89 KB of shared memory, so two CTAs share an SM
// and hide each other's latencies.  Only the operands its own MMAs read live in
// shared memory; Ki^T, Aqk, T' (tf32) and e^{g_last} go straight to the record.
constexpr int kChunkThreads = 256;
struct ChunkLayout {
    static constexpr uint32_t IN_Q = 0, IN_K = 16384;  // TMA boxes
    static constexpr uint32_t O2 = 32768;   // Ki bf16, 64 rows x 128
    static constexpr uint32_t O1 = 49152;   // [Kg ; Qg] -> [-W ; Qg] (the record's first image)
    static constexpr uint32_t O4 = 81920;   // T' bf16, 64 rows x 64 (prefix group totals before)
    // solve scratch over the input boxes and O2, both dead by then
    static constexpr uint32_t SOLVE_A = 0, SOLVE_T = kC * kLdS * 4, SOLVE_X = 2 * kC * kLdS * 4;
    static constexpr uint32_t USED = 90112;
};
static_assert(ChunkLayout::SOLVE_X + 32 * kLdX * 4 <= ChunkLayout::O1, "solve scratch overlaps O1");

struct StateLayout {
    static constexpr uint32_t STAGE = 91136;  // record + padding to 1024 bytes
    static constexpr uint32_t IN_V = 2 * STAGE;               // 2 x v slice [64][32] bf16
    static constexpr uint32_t O6 = IN_V + 2 * 4096;           // V^T tf32, 32 rows x K 64
    static constexpr uint32_t O7 = O6 + 8192;                 // S^T bf16, 32 rows x K 128
    static constexpr uint32_t O9 = O7 + 8192;                 // u^T bf16, 32 rows x K 64
    static constexpr uint32_t O10 = O9 + 4096;                // u^T tf32, 32 rows x K 64
    static constexpr uint32_t USED = O10 + 8192;
};
static_assert(StateLayout::STAGE % 1024 == 0 && StateLayout::STAGE >= kRecBytes, "stage size");
static_assert(StateLayout::O6 % 1024 == 0 && StateLayout::O7 % 1024 == 0 &&
              StateLayout::O9 % 1024 == 0 && StateLayout::O10 % 1024 == 0, "operand alignment");

constexpr uint32_t kChunkSmem = ChunkLayout::USED + 1024;
constexpr uint32_t kStateSmem = StateLayout::USED + 1024;

// ============================================================== chunk kernel
__global__ void __launch_bounds__(kChunkThreads, 2)
prefill_chunk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const float *__restrict__ log_alpha, const float *__restrict__ beta,
                     const int32_t *__restrict__ cu, int64_t total, int H, int num_seqs,
                     const int32_t *__restrict__ cc, unsigned char *__restrict__ records,
                     uint32_t *status)
{
    using L = ChunkLayout;
    constexpr int NT = kChunkThreads;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bar_tma, bar_mma;
    __shared__ uint32_t tmem_holder;
    __shared__ __align__(16) float s_beta[kC];

    const int g = blockIdx.x, h = blockIdx.y;
    if (g >= cc[num_seqs]) return;  // past the last chunk (the grid is an upper bound)
    int lo = 0, hi = num_seqs;      // sequence n with cc[n] <= g < cc[n + 1]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cc[mid] <= g) lo = mid; else hi = mid;
    }
    const int n = lo;
    int64_t t0, t1;
    seq_range(cu, n, total, t0, t1);
    const int64_t c0 = t0 + (int64_t)(g - cc[n]) * kC;
    const int len = (t1 - c0) < kC ? (int)(t1 - c0) : kC;
    unsigned char *rec = records + ((size_t)g * H + h) * kRecBytes;

    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&bar_tma, 16384 + 16384);
        tma_load_3d(sm + L::IN_Q, &tm_q, &bar_tma, 0, h, (int)c0);
        tma_load_3d(sm + L::IN_K, &tm_k, &bar_tma, 0, h, (int)c0);
    }
    if (warp == 0) {
        tmem_alloc(&tmem_holder, 256);
        tmem_relinquish();
    }
    if (tid < kC) s_beta[tid] = tid < len ? beta[(size_t)(c0 + tid) * H + h] : 0.f;
    // a1: the in-chunk decay prefix reads log_alpha straight from global memory,
    // overlapping the q/k copies
    float *s_tot = reinterpret_cast<float *>(sm + L::O4);
    float2 gl[4096 / NT];
    float gmin, gmax;
    prefix_scan<NT>(log_alpha + ((size_t)c0 * H + h) * kD, H * kD, len, s_tot, gl, gmin, gmax);
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_holder, tD1 = tmem, tDW = tmem + 64;
    bool timed_out = false, tma_pending = true, mma_pending = false, decay_bad = false;
    do {
        bool ok = mbar_wait_ns(&bar_tma, 0, kWaitNs);
        if (__syncthreads_or(!ok)) { timed_out = true; break; }
        tma_pending = false;
        decay_bad = decayed_operands<L, NT>(sm, len, s_tot, rec + R_O3,
                                            reinterpret_cast<float *>(rec + R_GM), gl, gmin, gmax);
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after_sync();
            issue_g1<L>(sb, tD1);
            mma_commit(&bar_mma);
        }
        mma_pending = true;
        ok = mbar_wait_ns(&bar_mma, 0, kWaitNs);
        if (__syncthreads_or(!ok)) { timed_out = true; break; }
        mma_pending = false;
        tc_fence_after_sync();
        kk_epilogue<L, NT>(sm, tD1, s_beta, rec + R_AQ);
        tc_fence_before_sync();
        __syncthreads();
        solve_ut<L, NT>(sm, s_beta, rec + R_TT, 64);
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after_sync();
            issue_gw<L>(sb, tDW);
            mma_commit(&bar_mma);
        }
        mma_pending = true;
        ok = mbar_wait_ns(&bar_mma, 1, kWaitNs);
        if (__syncthreads_or(!ok)) { timed_out = true; break; }
        mma_pending = false;
        tc_fence_after_sync();
        w_epilogue<L, NT>(sm, tDW);
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();
        if (tid == 0) {  // [-W ; Qg] image of the record
            bulk_store(rec + R_O1, sm + L::O1, 32768);
            bulk_commit();
            bulk_wait_all();
        }
    } while (false);
    if (timed_out) {
        if (tid == 0) atomicOr(status, DEV_ERR_TIMEOUT);
        if (tma_pending) (void)mbar_wait_ns(&bar_tma, 0, kWaitNs);
        if (mma_pending) (void)mbar_wait_ns(&bar_mma, 0, kWaitNs);
    }
    if (decay_bad) atomicOr(status, DEV_ERR_DECAY);
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

// ============================================================== state kernel
constexpr uint32_t IDESC_U = idesc_tf32(64, 32, false, false);   // T' V
constexpr uint32_t IDESC_WS = idesc_bf16(64, 32, false, false);  // -W S, Qg S, Aqk u
constexpr uint32_t IDESC_K = idesc_tf32(128, 32, false, false);  // Ki^T u
constexpr uint32_t TM_U = 0, TM_O = 32, TM_5 = 64, kStateTmem = 128;

__device__ __forceinline__ void issue_state_loads(unsigned char *sm, const unsigned char *rec,
                                                  const CUtensorMap *tv, uint64_t *bar, int st,
                                                  int h, int j0, int row)
{
    using L = StateLayout;
    mbar_arrive_expect_tx(bar, kRecBytes + 4096);
    bulk_load(sm + st * L::STAGE, rec, kRecBytes, bar);
    tma_load_3d(sm + L::IN_V + st * 4096, tv, bar, j0, h, row);
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_state_kernel(const __grid_constant__ CUtensorMap tm_v, const int32_t *__restrict__ cu,
                     int64_t total, int H, const int32_t *__restrict__ cc,
                     const unsigned char *__restrict__ records, const float *init_state,
                     __nv_bfloat16 *__restrict__ o, float *final_state, uint32_t *status,
                     const int32_t *__restrict__ order)
{
    using L = StateLayout;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bar_ld[2], bar_mma;
    __shared__ uint32_t tmem_holder;

    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, part = warp >> 2;
    const int j0 = blockIdx.x * kDV, h = blockIdx.y, n = order[blockIdx.z];
    int64_t t0, t1;
    seq_range(cu, n, total, t0, t1);
    const int nchunks = (int)((t1 - t0 + kC - 1) / kC);
    const unsigned char *rec0 = records + ((size_t)cc[n] * H + h) * kRecBytes;
    const size_t rec_stride = (size_t)H * kRecBytes;

    if (tid == 0) {
        mbar_init(&bar_ld[0], 1);
        mbar_init(&bar_ld[1], 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
        prefetch_tmap(&tm_v);
        for (int c = 0; c < 2 && c < nchunks; ++c)
            issue_state_loads(sm, rec0 + c * rec_stride, &tm_v, &bar_ld[c], c, h, j0, (int)(t0 + c * kC));
    }
    if (warp == 0) {
        tmem_alloc(&tmem_holder, kStateTmem);
        tmem_relinquish();
    }
    // state row i, columns j0 + 8*part .. +7 in registers; S^T (bf16) operand in O7
    const int i_row = quarter * 32 + lane, jp = part * 8;
    float S[8];
    const size_t st_off = (((size_t)n * H + h) * kD + i_row) * kD + j0 + jp;
    if (init_state) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float4 x = *reinterpret_cast<const float4 *>(init_state + st_off + 4 * q);
            S[4 * q] = x.x; S[4 * q + 1] = x.y; S[4 * q + 2] = x.z; S[4 * q + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) S[j] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) store_bf16(sm + L::O7 + km16(jp + j, i_row, kDV), S[j]);
    fence_proxy_async_smem();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_holder;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int r64 = quarter * 16 + (lane & 15);  // row held by this lane in an M = 64 accumulator

    uint32_t ph_mma = 0;
    bool timed_out = false, mma_pending = false;
    int c = 0;
    for (; c < nchunks; ++c) {
        const int st = c & 1;
        const int64_t c0 = t0 + (int64_t)c * kC;
        const int len = (t1 - c0) < kC ? (int)(t1 - c0) : kC;
        unsigned char *stg = sm + st * L::STAGE;
        const uint32_t sg = sb + st * L::STAGE;

        bool ok = mbar_wait_ns(&bar_ld[st], (uint32_t)((c >> 1) & 1), kWaitNs);
        if (__syncthreads_or(!ok)) { timed_out = true; break; }
        {  // V^T (tf32, K-major [j][s]): one 4-row group of one column per thread
            const int j = tid % kDV, s4 = (tid / kDV) * 4;
            float x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                x[u] = (s4 + u) < len ? bf16_at(sm + L::IN_V + st * 4096 + ((s4 + u) * kDV + j) * 2) : 0.f;
            *reinterpret_cast<float4 *>(sm + L::O6 + km32(j, s4, kDV)) = make_float4(x[0], x[1], x[2], x[3]);
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ------------------------------------------------------ u = T'V - WS, Qg S
        if (tid == 0) {
            tc_fence_after_sync();
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t p = s >> 2, w = (s & 3) * 32;
                mma_tf32(tmem + TM_U, kdesc(sg + R_TT + p * 8192 + w), kdesc(sb + L::O6 + p * 4096 + w),
                         IDESC_U, s > 0);
            }
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t p = s >> 2, w = (s & 3) * 32;
                mma_bf16(tmem + TM_U, kdesc(sg + R_O1 + p * 16384 + w), kdesc(sb + L::O7 + p * 4096 + w),
                         IDESC_WS, 1);
                mma_bf16(tmem + TM_O, kdesc(sg + R_O1 + p * 16384 + 8192 + w),
                         kdesc(sb + L::O7 + p * 4096 + w), IDESC_WS, s > 0);
            }
            mma_commit(&bar_mma);
        }
        mma_pending = true;
        ok = mbar_wait_ns(&bar_mma, ph_mma, kWaitNs);
        if (__syncthreads_or(!ok)) { timed_out = true; break; }
        mma_pending = false;
        ph_mma ^= 1;
        tc_fence_after_sync();
        {  // u (M = 64 layout: row 16q + l in lane l < 16) -> u^T operands, row pairs
            float v[8];
            tmem_ld8(tmem + TM_U + lane_off + jp, v);
            tmem_ld_wait();
            const int odd = lane & 1, re = r64 & ~1;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float mine = odd ? v[4 + u] : v[u];
                const float give = odd ? v[u] : v[4 + u];
                const float other = __shfl_xor_sync(0xffffffffu, give, 1);
                const float lo = odd ? other : mine, hi = odd ? mine : other;  // rows re, re+1
                const int j = jp + 4 * odd + u;
                if (lane < 16) {
                    *reinterpret_cast<uint32_t *>(sm + L::O9 + km16(j, re, kDV)) = pack_bf16x2(lo, hi);
                    *reinterpret_cast<float2 *>(sm + L::O10 + km32(j, re, kDV)) =
                        make_float2(to_tf32(lo), to_tf32(hi));
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();

        // ------------------------------------------------------ o += Aqk u, D5 = Ki^T u
        if (tid == 0) {
            tc_fence_after_sync();
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma_bf16(tmem + TM_O, kdesc(sg + R_AQ + s * 32), kdesc(sb + L::O9 + s * 32), IDESC_WS, 1);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t p = s >> 2, w = (s & 3) * 32;
                mma_tf32(tmem + TM_5, kdesc(sg + R_O3 + p * 16384 + w), kdesc(sb + L::O10 + p * 4096 + w),
                         IDESC_K, s > 0);
            }
            mma_commit(&bar_mma);
        }
        mma_pending = true;
        ok = mbar_wait_ns(&bar_mma, ph_mma, kWaitNs);
        if (__syncthreads_or(!ok)) { timed_out = true; break; }
        mma_pending = false;
        ph_mma ^= 1;
        tc_fence_after_sync();
        {  // o rows (M = 64 layout)
            float v[8];
            tmem_ld8(tmem + TM_O + lane_off + jp, v);
            tmem_ld_wait();
            if (lane < 16 && r64 < len)
                *reinterpret_cast<uint4 *>(o + ((size_t)(c0 + r64) * H + h) * kD + j0 + jp) = pack_bf16x8(v);
        }
        {  // state rows: S <- gamma_c (S + Ki^T u); S^T (bf16) for the next chunk, row pairs
            float v[8];
            tmem_ld8(tmem + TM_5 + lane_off + jp, v);
            tmem_ld_wait();
            const float gc = reinterpret_cast<const float *>(stg + R_GM)[i_row];
#pragma unroll
            for (int j = 0; j < 8; ++j) S[j] = gc * (S[j] + v[j]);
            const int odd = lane & 1, ie = i_row & ~1;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float mine = odd ? S[4 + u] : S[u];
                const float give = odd ? S[u] : S[4 + u];
                const float other = __shfl_xor_sync(0xffffffffu, give, 1);
                const float lo = odd ? other : mine, hi = odd ? mine : other;
                *reinterpret_cast<uint32_t *>(sm + L::O7 + km16(jp + 4 * odd + u, ie, kDV)) = pack_bf16x2(lo, hi);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();
        if (tid == 0 && c + 2 < nchunks)  // this stage is free: load chunk c + 2 into it
            issue_state_loads(sm, rec0 + (size_t)(c + 2) * rec_stride, &tm_v, &bar_ld[st], st, h, j0,
                              (int)(c0 + 2 * kC));
    }
    if (timed_out) {
        if (tid == 0) atomicOr(status, DEV_ERR_TIMEOUT);
        // drain our own loads and MMAs (bounded) before releasing shared and tensor memory
        if (mma_pending) (void)mbar_wait_ns(&bar_mma, ph_mma, kWaitNs);
        for (int k = c; k < c + 2 && k < nchunks; ++k)
            (void)mbar_wait_ns(&bar_ld[k & 1], (uint32_t)((k >> 1) & 1), kWaitNs);
    } else {
        float *dst = final_state + st_off;
#pragma unroll
        for (int q = 0; q < 2; ++q)
            *reinterpret_cast<float4 *>(dst + 4 * q) = make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kStateTmem);
}

}  // namespace

size_t prefill_split_records_bytes(int64_t total_tokens, int num_seqs, int num_heads)
{
    return (size_t)(total_tokens / kC + num_seqs) * (size_t)num_heads * kRecBytes;
}

cudaError_t launch_prefill_split(const PrefillProblem &p, const int32_t *cc, void *records)
{
    static int dev_chunk = -1, dev_state = -1;
    cudaError_t err = allow_smem(prefill_chunk_kernel, (int)kChunkSmem, &dev_chunk);
    if (err != cudaSuccess) return err;
    err = allow_smem(prefill_state_kernel, (int)kStateSmem, &dev_state);
    if (err != cudaSuccess) return err;
    CUtensorMap tq, tk, tv;
    if (!make_map(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.q, p.total_tokens, p.num_heads, 2, kD) ||
        !make_map(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.k, p.total_tokens, p.num_heads, 2, kD) ||
        !make_map(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.v, p.total_tokens, p.num_heads, 2, kDV))
        return cudaErrorInvalidValue;
    const int64_t chunk_bound = p.total_tokens / kC + p.num_seqs;
    dim3 grid_a((unsigned)chunk_bound, p.num_heads);
    prefill_chunk_kernel<<<grid_a, kChunkThreads, kChunkSmem, p.stream>>>(
        tq, tk, p.log_alpha, p.beta, p.cu_seqlens, p.total_tokens, p.num_heads, p.num_seqs, cc,
        static_cast<unsigned char *>(records), p.status);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    dim3 grid_b(kD / kDV, p.num_heads, p.num_seqs);
    prefill_state_kernel<<<grid_b, kThreads, kStateSmem, p.stream>>>(
        tv, p.cu_seqlens, p.total_tokens, p.num_heads, cc,
        static_cast<const unsigned char *>(records), p.init_state,
        static_cast<__nv_bfloat16 *>(p.o), p.final_state, p.status, p.order);
    return cudaGetLastError();
}

}  // namespace kda
