// prefill_tc.cu -- chunkwise KDA prefill on the 5th-generation tensor cores
// (bf16 q/k/v, d_k = d_v = 128, fp32 state), sm_103a.
//
// One CTA owns one (sequence, head, 32-column value slice) and walks the
// sequence's 64-token chunks in order (parallel inside a chunk, serial across
// chunks: "From 124M to 2.8T", chapter 3; WY representation + UT transform:
// "K3 attention, three-piece set", KDA engineering details).  Per chunk, with
// g the in-chunk cumulative log-decay, Kg = k e^g, Ki = k e^-g, Qg = q e^g / sqrt(d):
//
//   TMA      q, k, log_alpha [64 x 128] and v [64 x 32] -> shared memory
//   prep     g, Kg, Qg, Ki (bf16 and tf32 copies), V^T (tf32)             (a1, a2)
//   G1 bf16  D1 = [Kg ; Qg] Ki^T   -> A = strict-lower(beta . D1[0:64]),
//                                     Aqk = lower(D1[64:128])              (a3)
//   solve    T' = (I + A)^-1 diag(beta), recursive doubling over 16 x 16 blocks (a4)
//   GW bf16  W^T = Kg^T T'^T                                               (a5)
//   GU tf32  D3  = [T' ; 0] V          (U~, the value part of the WY form)  (a5)
//   G3 bf16  D3 += [-W ; Qg] S         rows 0-63: u, rows 64-127: Qg S      (a6)
//   G4 bf16  D3 += [. ; Aqk] u         rows 64-127: o                       (a6)
//   G5 tf32  D5  = Ki^T u
//   state    S  <- e^{g_last} (S + D5)  (Kd = e^{g_last} Ki, so this is
//            Diag(e^{g_last}) S + Kd^T u)                                   (a7)
//
// Precision: the products that produce u and the state (T' V, Ki^T u) take
// tf32 operands; the k-k / q-k matrices, W S and Aqk u take bf16 operands;
// all accumulate in fp32 in tensor memory and the state stays fp32 in registers.
//
// Every operand lives in shared memory in the K-major 128-byte-swizzled layout
// the MMA descriptors expect; accumulators live in tensor memory (256 columns).
// Every mbarrier wait is bounded by wall-clock time; on expiry the CTA records
// KDA_DEVICE timeout in the workspace word, drains its own copies and MMAs
// (bounded again), frees its tensor memory and returns.
#include "tc_common.cuh"

namespace kda {
namespace {

using namespace ptx;
using namespace tc;

// Dynamic shared memory map (byte offsets from a 1024-byte aligned base).
struct FusedLayout {
    static constexpr uint32_t IN_Q = 0;       // q   [64][128] bf16 (TMA box, row-major)
    static constexpr uint32_t IN_K = 16384;   // k   [64][128] bf16
    static constexpr uint32_t IN_LA = 32768;  // log_alpha [64][128] fp32
    static constexpr uint32_t IN_V = 65536;   // v slice [64][32] bf16
    static constexpr uint32_t O1 = 69632;     // [Kg ; Qg] then [-W ; Qg]: bf16, 128 rows x K 128
    static constexpr uint32_t O2 = 102400;    // Ki: bf16, 64 rows x K 128
    static constexpr uint32_t O3 = 118784;    // Ki^T: tf32, 128 rows (i) x K 64 (r)
    static constexpr uint32_t O4 = 151552;    // T': bf16, 64 rows x K 64
    static constexpr uint32_t AQ = 159744;    // Aqk: bf16, 64 rows x K 64 (rows 64-127 of [T' ; Aqk])
    static constexpr uint32_t TT = 167936;    // [T' ; 0]: tf32, 128 rows x K 64
    static constexpr int TT_ROWS = 128;
    static constexpr uint32_t O6 = 200704;    // V^T: tf32, 32 rows (j) x K 64 (s)
    static constexpr uint32_t O7 = 208896;    // S^T: bf16, 32 rows (j) x K 128 (i)
    static constexpr uint32_t O9 = 217088;    // u^T: bf16, 32 rows (j) x K 64 (r)
    static constexpr uint32_t O10 = 221184;   // u^T: tf32, 32 rows (j) x K 64 (r)
    // solve scratch inside the input area (idle between the operand prep and the next TMA)
    static constexpr uint32_t SOLVE_A = 0, SOLVE_T = kC * kLdS * 4, SOLVE_X = 2 * kC * kLdS * 4;
    static constexpr uint32_t USED = 229376;
};
using L = FusedLayout;
constexpr uint32_t kSmemDyn = L::USED + 1024;  // slack to align the base to 1024 bytes
constexpr uint32_t kLaBoxBytes = kC * kD * 4;  // log_alpha [64 x 128] fp32
constexpr uint32_t kTxBytes = 16384 + 16384 + kLaBoxBytes + 4096;
static_assert(L::AQ == L::O4 + 8192, "[T' ; Aqk] must be one 128-row operand");
static_assert(L::SOLVE_X + 32 * kLdX * 4 <= L::IN_V, "solve scratch must fit in the input area");

// Tensor-memory columns (one allocation of 256).
constexpr uint32_t TM_D1 = 0, TM_DW = 64, TM_D3 = 192, TM_D5 = 224, kTmemCols = 256;

constexpr uint32_t IDESC_GU = idesc_tf32(128, 32, false, false);
constexpr uint32_t IDESC_G3 = idesc_bf16(128, 32, false, false);
constexpr uint32_t IDESC_G5 = idesc_tf32(128, 32, false, false);

__device__ __forceinline__ void issue_chunk_loads(unsigned char *sm, const CUtensorMap *tq,
                                                  const CUtensorMap *tk, const CUtensorMap *tla,
                                                  const CUtensorMap *tv, uint64_t *bar, int h,
                                                  int j0, int row, bool scalar_gate)
{
    // a scalar gate is read from global memory by the prefix scan: no log_alpha box
    mbar_arrive_expect_tx(bar, scalar_gate ? kTxBytes - kLaBoxBytes : kTxBytes);
    tma_load_3d(sm + L::IN_Q, tq, bar, 0, h, row);
    tma_load_3d(sm + L::IN_K, tk, bar, 0, h, row);
    if (!scalar_gate) tma_load_3d(sm + L::IN_LA, tla, bar, 0, h, row);
    tma_load_3d(sm + L::IN_V, tv, bar, j0, h, row);
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_la, const __grid_constant__ CUtensorMap tm_v,
                  const float *__restrict__ beta, const int32_t *__restrict__ cu, int64_t total,
                  int H, const float *init_state, __nv_bfloat16 *__restrict__ o,
                  float *final_state, uint32_t *status, const int32_t *__restrict__ order,
                  const float *__restrict__ la_scalar, StateSlots slots, bool qk_norm)
{
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bar_tma, bar_mma;
    __shared__ uint32_t tmem_holder;
    __shared__ __align__(16) float s_beta[kC];
    __shared__ __align__(8) float s_gam[kD];
    __shared__ float s_rn[2 * kC];  // reciprocal k, q row norms (qk_norm)

    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, part = warp >> 2;  // TMEM lane quarter; column part (0..3)
    const int j0 = blockIdx.x * kDV, h = blockIdx.y, n = order[blockIdx.z];
    int64_t t0, t1;
    seq_range(cu, n, total, t0, t1);
    const int nchunks = (int)((t1 - t0 + kC - 1) / kC);

    if (tid == 0) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_la);
        prefetch_tmap(&tm_v);
    }
    if (warp == 0) {
        tmem_alloc(&tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    for (int e = tid; e < 2 * 2048; e += kThreads)  // rows 64..127 of [T' ; 0] stay zero
        *reinterpret_cast<uint32_t *>(sm + L::TT + (e >> 11) * 16384 + 8192 + (e & 2047) * 4) = 0u;

    // State row i, columns j0 + 8*part .. +7, fp32 in registers.  The thread owns
    // TMEM lane i of every 128-lane accumulator.
    const int i_row = quarter * 32 + lane;
    const int jp = part * 8;
    float S[8];
    int64_t si, sf;
    if (!state_entries(slots, n, init_state != nullptr, si, sf) && tid == 0) atomicOr(status, DEV_ERR_SLOT);
    const size_t st_off = ((size_t)h * kD + i_row) * kD + j0 + jp, st_entry = (size_t)H * kD * kD;
    if (si >= 0) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float4 x = *reinterpret_cast<const float4 *>(init_state + si * st_entry + st_off + 4 * q);
            S[4 * q] = x.x; S[4 * q + 1] = x.y; S[4 * q + 2] = x.z; S[4 * q + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) S[j] = 0.f;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) store_bf16(sm + L::O7 + km16(jp + j, i_row, kDV), S[j]);
    // beta of the next chunk is loaded one chunk ahead (hides the global-load latency)
    float beta_next = (tid < kC && tid < t1 - t0) ? beta[(size_t)(t0 + tid) * H + h] : 0.f;

    fence_proxy_async_smem();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_holder;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;

    uint32_t ph_tma = 0, ph_mma = 0;
    bool tma_pending = nchunks > 0, mma_pending = false, timed_out = false, decay_bad = false;
    if (tid == 0 && nchunks > 0)
        issue_chunk_loads(sm, &tm_q, &tm_k, &tm_la, &tm_v, &bar_tma, h, j0, (int)t0, la_scalar);
    // group totals of the prefix scan; the tf32 u operand area is idle during the prep
    float *s_tot = reinterpret_cast<float *>(sm + L::O10);

    for (int c = 0; c < nchunks; ++c) {
        const int64_t c0 = t0 + (int64_t)c * kC;
        const int len = (t1 - c0) < kC ? (int)(t1 - c0) : kC;

        // ---------------------------------------------------------- inputs landed
        bool ok = mbar_wait_ns(&bar_tma, ph_tma, kWaitNs);
        if (__syncthreads_or(!ok)) { timed_out = true; break; }
        ph_tma ^= 1;
        tma_pending = false;
        if (qk_norm) qk_row_inv_norms<kThreads>(sm + L::IN_K, sm + L::IN_Q, s_rn);  // read after the barrier below

        // ---------------------------------------------------------- a1, a2
        float2 gl[8];
        float gmin, gmax;
        if (la_scalar)  // log_alpha [T, H]: one decay per token-head
            prefix_scan<kThreads>(la_scalar + (size_t)c0 * H + h, H, len, s_tot, gl, gmin, gmax, true);
        else
            prefix_scan<kThreads>(reinterpret_cast<const float *>(sm + L::IN_LA), kD, len, s_tot, gl,
                                  gmin, gmax);
        if (tid < kC) {
            s_beta[tid] = beta_next;
            const int64_t cn = c0 + kC;  // next chunk
            beta_next = (tid < t1 - cn) ? beta[(size_t)(cn + tid) * H + h] : 0.f;
        }
        {  // V^T (tf32, K-major [j][s]): one 4-row group of one column per thread
            const int j = tid % kDV, s4 = (tid / kDV) * 4;
            float x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                x[u] = (s4 + u) < len ? bf16_at(sm + L::IN_V + ((s4 + u) * kDV + j) * 2) : 0.f;
            *reinterpret_cast<float4 *>(sm + L::O6 + km32(j, s4, kDV)) = make_float4(x[0], x[1], x[2], x[3]);
        }
        __syncthreads();
        if (decayed_operands<L, kThreads, true, true>(sm, len, s_tot, sm + L::O3, s_gam, gl, gmin, gmax,
                                                      nullptr, qk_norm ? s_rn : nullptr))
            decay_bad = true;
        fence_proxy_async_smem();
        __syncthreads();

        // ---------------------------------------------------------- a3: G1
        if (tid == 0) {
            tc_fence_after_sync();
            issue_g1<L>(sb, tmem + TM_D1);
            mma_commit(&bar_mma);
        }
        ok = mbar_wait_ns(&bar_mma, ph_mma, kWaitNs);
        if (__syncthreads_or(!ok)) { timed_out = true; mma_pending = true; break; }
        ph_mma ^= 1;
        tc_fence_after_sync();
        kk_epilogue<L, kThreads>(sm, tmem + TM_D1, s_beta, sm + L::AQ);
        tc_fence_before_sync();
        __syncthreads();

        // ---------------------------------------------------------- a4: T = (I + A)^-1
        solve_ut<L, kThreads>(sm, s_beta, sm + L::TT, L::TT_ROWS);
        fence_proxy_async_smem();
        __syncthreads();

        // ---------------------------------------------------------- a5: GW, GU; next inputs
        if (tid == 0) {
            if (c + 1 < nchunks)
                issue_chunk_loads(sm, &tm_q, &tm_k, &tm_la, &tm_v, &bar_tma, h, j0,
                                  (int)(c0 + kC), la_scalar);
            tc_fence_after_sync();
            issue_gw<L>(sb, tmem + TM_DW);
#pragma unroll
            for (int s = 0; s < 8; ++s) {  // U~ = [T' ; 0] V  (tf32)
                const uint32_t p = s >> 2, w = (s & 3) * 32;
                mma_tf32(tmem + TM_D3, kdesc(sb + L::TT + p * 16384 + w), kdesc(sb + L::O6 + p * 4096 + w),
                         IDESC_GU, s > 0);
            }
            mma_commit(&bar_mma);
        }
        tma_pending = c + 1 < nchunks;
        ok = mbar_wait_ns(&bar_mma, ph_mma, kWaitNs);
        if (__syncthreads_or(!ok)) { timed_out = true; mma_pending = true; break; }
        ph_mma ^= 1;
        tc_fence_after_sync();
        w_epilogue<L, kThreads>(sm, tmem + TM_DW);
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();

        // ---------------------------------------------------------- a6: G3 -> u, Qg S
        if (tid == 0) {
            tc_fence_after_sync();
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t p = s >> 2, w = (s & 3) * 32;
                mma_bf16(tmem + TM_D3, kdesc(sb + L::O1 + p * 16384 + w), kdesc(sb + L::O7 + p * 4096 + w),
                         IDESC_G3, 1);
            }
            mma_commit(&bar_mma);
        }
        ok = mbar_wait_ns(&bar_mma, ph_mma, kWaitNs);
        if (__syncthreads_or(!ok)) { timed_out = true; mma_pending = true; break; }
        ph_mma ^= 1;
        tc_fence_after_sync();

        if (quarter < 2) {  // u rows 0..63 -> bf16 and tf32 operands (u^T, K-major)
            // Adjacent lanes (rows r, r^1) swap halves so each writes a row pair
            // (2 x bf16, 2 x tf32) for 4 of the thread's 8 columns.
            const int r = quarter * 32 + lane, odd = lane & 1, re = r & ~1;
            float v[8];
            tmem_ld8(tmem + TM_D3 + lane_off + jp, v);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float mine = odd ? v[4 + u] : v[u];
                const float give = odd ? v[u] : v[4 + u];
                const float other = __shfl_xor_sync(0xffffffffu, give, 1);
                const float lo = odd ? other : mine, hi = odd ? mine : other;  // rows re, re+1
                const int j = jp + 4 * odd + u;
                *reinterpret_cast<uint32_t *>(sm + L::O9 + km16(j, re, kDV)) = pack_bf16x2(lo, hi);
                *reinterpret_cast<float2 *>(sm + L::O10 + km32(j, re, kDV)) = make_float2(to_tf32(lo), to_tf32(hi));
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();

        // ---------------------------------------------------------- a6/a7: G4 -> o, G5
        if (tid == 0) {
            tc_fence_after_sync();
#pragma unroll
            for (int s = 0; s < 4; ++s)  // rows 64-127 of [T' ; Aqk] are Aqk
                mma_bf16(tmem + TM_D3, kdesc(sb + L::O4 + s * 32), kdesc(sb + L::O9 + s * 32), IDESC_G3, 1);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t p = s >> 2, w = (s & 3) * 32;
                mma_tf32(tmem + TM_D5, kdesc(sb + L::O3 + p * 16384 + w), kdesc(sb + L::O10 + p * 4096 + w),
                         IDESC_G5, s > 0);
            }
            mma_commit(&bar_mma);
        }
        ok = mbar_wait_ns(&bar_mma, ph_mma, kWaitNs);
        if (__syncthreads_or(!ok)) { timed_out = true; mma_pending = true; break; }
        ph_mma ^= 1;
        tc_fence_after_sync();

        if (quarter >= 2) {  // o rows 0..63 from lanes 64..127
            const int r = (quarter - 2) * 32 + lane;
            float v[8];
            tmem_ld8(tmem + TM_D3 + lane_off + jp, v);
            tmem_ld_wait();
            if (r < len && o)
                *reinterpret_cast<uint4 *>(o + ((size_t)(c0 + r) * H + h) * kD + j0 + jp) = pack_bf16x8(v);
        }
        {  // state rows: S <- gamma_c (S + Ki^T u); S^T (bf16) for the next chunk, row pairs
            float v[8];
            tmem_ld8(tmem + TM_D5 + lane_off + jp, v);
            tmem_ld_wait();
            const float gc = s_gam[i_row];
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
    }

    if (timed_out) {
        if (tid == 0) atomicOr(status, DEV_ERR_TIMEOUT);
        // drain our own copies and MMAs (bounded) before releasing shared and tensor memory
        if (tma_pending) (void)mbar_wait_ns(&bar_tma, ph_tma, kWaitNs);
        if (mma_pending) (void)mbar_wait_ns(&bar_mma, ph_mma, kWaitNs);
    } else if (sf >= 0) {
        float *dst = final_state + sf * st_entry + st_off;
#pragma unroll
        for (int q = 0; q < 2; ++q)
            *reinterpret_cast<float4 *>(dst + 4 * q) = make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
    }
    if (decay_bad) atomicOr(status, DEV_ERR_DECAY);
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool prefill_tc_supported(const PrefillProblem &p)
{
    return p.dtype == KDA_DTYPE_BF16 && p.d == kD && p.total_tokens > 0 &&
           p.total_tokens <= 0x7fffffffll;
}

cudaError_t launch_prefill_tc(const PrefillProblem &p)
{
    static int configured_device = -1;
    cudaError_t err = allow_smem(prefill_tc_kernel, (int)kSmemDyn, &configured_device);
    if (err != cudaSuccess) return err;
    CUtensorMap tq, tk, tla, tv;
    if (!make_map(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.q, p.total_tokens, p.num_heads, 2, kD) ||
        !make_map(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.k, p.total_tokens, p.num_heads, 2, kD) ||
        !make_map(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.v, p.total_tokens, p.num_heads, 2, kDV))
        return cudaErrorInvalidValue;
    // a scalar gate ([T, H]) is read by the prefix scan, never by TMA: its map slot repeats q's
    if (p.scalar_gate)
        tla = tq;
    else if (!make_map(&tla, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.log_alpha, p.total_tokens,
                       p.num_heads, 4, kD))
        return cudaErrorInvalidValue;
    dim3 grid(kD / kDV, p.num_heads, p.num_seqs);
    prefill_tc_kernel<<<grid, kThreads, kSmemDyn, p.stream>>>(
        tq, tk, tla, tv, p.beta, p.cu_seqlens, p.total_tokens, p.num_heads, p.init_state,
        static_cast<__nv_bfloat16 *>(p.o), p.final_state, p.status, p.order,
        p.scalar_gate ? p.log_alpha : nullptr, p.slots, p.qk_l2norm);
    return cudaGetLastError();
}

}  // namespace kda
