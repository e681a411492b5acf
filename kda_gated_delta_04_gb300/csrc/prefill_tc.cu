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
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr int kD = 128, kDV = 32, kC = 64, kTcThreads = 512;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait before giving up

// Dynamic shared memory map (byte offsets from a 1024-byte aligned base).
constexpr uint32_t IN_Q = 0;        // q   [64][128] bf16 (TMA box, row-major)
constexpr uint32_t IN_K = 16384;    // k   [64][128] bf16
constexpr uint32_t IN_LA = 32768;   // log_alpha [64][128] fp32
constexpr uint32_t IN_V = 65536;    // v slice [64][32] bf16
constexpr uint32_t O1 = 69632;      // [Kg ; Qg] then [-W ; Qg]: bf16, 128 rows x K 128
constexpr uint32_t O2 = 102400;     // Ki: bf16, 64 rows x K 128
constexpr uint32_t O3 = 118784;     // Ki^T: tf32, 128 rows (i) x K 64 (r)
constexpr uint32_t O4 = 151552;     // T': bf16, 64 rows x K 64
constexpr uint32_t O8 = 159744;     // Aqk: bf16, 64 rows x K 64 (rows 64-127 of [T' ; Aqk])
constexpr uint32_t O5 = 167936;     // [T' ; 0]: tf32, 128 rows x K 64
constexpr uint32_t O6 = 200704;     // V^T: tf32, 32 rows (j) x K 64 (s)
constexpr uint32_t O7 = 208896;     // S^T: bf16, 32 rows (j) x K 128 (i)
constexpr uint32_t O9 = 217088;     // u^T: bf16, 32 rows (j) x K 64 (r)
constexpr uint32_t O10 = 221184;    // u^T: tf32, 32 rows (j) x K 64 (r)
constexpr uint32_t kSmemUsed = 229376;
constexpr uint32_t kSmemDyn = kSmemUsed + 1024;  // slack to align the base to 1024 bytes
// Solve scratch inside the input area (idle between the operand prep and the next TMA).
constexpr int kLdS = kC + 4;   // row stride (floats) of A and T
constexpr int kLdX = 32 + 4;   // row stride of the block products X (up to 32 x 32)
constexpr uint32_t SOLVE_A = 0, SOLVE_T = kC * kLdS * 4, SOLVE_X = 2 * kC * kLdS * 4;
constexpr uint32_t kTxBytes = 16384 + 16384 + 32768 + 4096;
static_assert(O8 == O4 + 8192, "[T' ; Aqk] must be one 128-row operand");
static_assert(SOLVE_X + 32 * kLdX * 4 <= IN_V, "solve scratch must fit in the input area");

// Tensor-memory columns (one allocation of 256).
constexpr uint32_t TM_D1 = 0, TM_DW = 64, TM_D3 = 192, TM_D5 = 224, kTmemCols = 256;

constexpr uint32_t IDESC_G1 = idesc_bf16(128, 64, false, false);
constexpr uint32_t IDESC_GW = idesc_bf16(64, 128, false, true);  // W = T' Kg (Kg MN-major)
constexpr uint32_t IDESC_GU = idesc_tf32(128, 32, false, false);
constexpr uint32_t IDESC_G3 = idesc_bf16(128, 32, false, false);
constexpr uint32_t IDESC_G5 = idesc_tf32(128, 32, false, false);

// Byte offset of element (row, col) of a K-major, 128-byte-swizzled operand
// with `rows` rows per 64-element (bf16) or 32-element (tf32) column panel.
__device__ __forceinline__ uint32_t km16(int row, int col, int rows)
{
    return (uint32_t)((col >> 6) * rows * 128 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) +
                      ((col & 7) << 1));
}
__device__ __forceinline__ uint32_t km32(int row, int col, int rows)
{
    return (uint32_t)((col >> 5) * rows * 128 + row * 128 + ((((col & 31) >> 2) ^ (row & 7)) << 4) +
                      ((col & 3) << 2));
}

__device__ __forceinline__ uint64_t kdesc(uint32_t addr) { return sdesc(addr, 16, 1024, kSw128B); }

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float bf16_at(const unsigned char *p)
{
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(p));
}

__device__ __forceinline__ void store_bf16(unsigned char *p, float x)
{
    *reinterpret_cast<__nv_bfloat16 *>(p) = __float2bfloat16_rn(x);
}

__device__ __forceinline__ void issue_chunk_loads(unsigned char *sm, const CUtensorMap *tq,
                                                  const CUtensorMap *tk, const CUtensorMap *tla,
                                                  const CUtensorMap *tv, uint64_t *bar, int h,
                                                  int j0, int row)
{
    mbar_arrive_expect_tx(bar, kTxBytes);
    tma_load_3d(sm + IN_Q, tq, bar, 0, h, row);
    tma_load_3d(sm + IN_K, tk, bar, 0, h, row);
    tma_load_3d(sm + IN_LA, tla, bar, 0, h, row);
    tma_load_3d(sm + IN_V, tv, bar, j0, h, row);
}

__device__ __forceinline__ void unpack_bf16x8(uint4 raw, float (&x)[8])
{
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w[q]));
        x[2 * q] = f.x;
        x[2 * q + 1] = f.y;
    }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&x)[8])
{
    return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                      pack_bf16x2(x[6], x[7]));
}

__global__ void __launch_bounds__(kTcThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_la, const __grid_constant__ CUtensorMap tm_v,
                  const float *__restrict__ beta, const int32_t *__restrict__ cu, int64_t total,
                  int H, const float *init_state, __nv_bfloat16 *__restrict__ o,
                  float *final_state, uint32_t *status, const int32_t *__restrict__ order)
{
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bar_tma, bar_mma;
    __shared__ uint32_t tmem_holder;
    __shared__ __align__(16) float s_beta[kC];
    __shared__ __align__(8) float s_gam[kD];

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
    // rows 64..127 of [T' ; 0] (both 32-column panels) stay zero for the whole kernel
    for (int e = tid; e < 2 * 2048; e += kTcThreads)  // 2 panels x 64 rows x 32 words
        *reinterpret_cast<uint32_t *>(sm + O5 + (e >> 11) * 16384 + 8192 + (e & 2047) * 4) = 0u;

    // State row i, columns j0 + 8*part .. +7, fp32 in registers.  The thread owns
    // TMEM lane i of every 128-lane accumulator.
    const int i_row = quarter * 32 + lane;
    const int jp = part * 8;
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
    for (int j = 0; j < 8; ++j) store_bf16(sm + O7 + km16(jp + j, i_row, kDV), S[j]);
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
        issue_chunk_loads(sm, &tm_q, &tm_k, &tm_la, &tm_v, &bar_tma, h, j0, (int)t0);

    float *sA = reinterpret_cast<float *>(sm + SOLVE_A);
    float *sT = reinterpret_cast<float *>(sm + SOLVE_T);
    float *sX = reinterpret_cast<float *>(sm + SOLVE_X);
    const float *la_in = reinterpret_cast<const float *>(sm + IN_LA);
    // quarter totals of the prefix scan; the tf32 u operand area is idle during the prep
    float *s_tot = reinterpret_cast<float *>(sm + O10);

    for (int c = 0; c < nchunks; ++c) {
        const int64_t c0 = t0 + (int64_t)c * kC;
        const int len = (t1 - c0) < kC ? (int)(t1 - c0) : kC;

        // ---------------------------------------------------------- inputs landed
        bool ok = mbar_wait_ns(&bar_tma, ph_tma, kWaitNs);
        if (__syncthreads_or(!ok)) { timed_out = true; break; }
        ph_tma ^= 1;
        tma_pending = false;

        // ---------------------------------------------------------- a1: prefix over rows
        // Thread = (channel pair cp: channels 2cp, 2cp+1; row group rg: rows
        // 8rg .. 8rg+7).  Each scans its 8 rows in registers; group totals are
        // combined through shared memory.
        const int cp = tid & 63, rg = tid >> 6;
        float2 gl[8];
        float gmin = 0.f, gmax = 0.f;
        {
            float2 g = make_float2(0.f, 0.f);
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                const int r = rg * 8 + rr;
                const float2 la = r < len ? *reinterpret_cast<const float2 *>(la_in + r * kD + 2 * cp)
                                          : make_float2(0.f, 0.f);
                g.x += la.x;
                g.y += la.y;
                gl[rr] = g;
                gmin = fminf(gmin, fminf(g.x, g.y));
                gmax = fmaxf(gmax, fmaxf(g.x, g.y));
            }
            *reinterpret_cast<float2 *>(&s_tot[rg * kD + 2 * cp]) = g;
        }
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
                x[u] = (s4 + u) < len ? bf16_at(sm + IN_V + ((s4 + u) * kDV + j) * 2) : 0.f;
            *reinterpret_cast<float4 *>(sm + O6 + km32(j, s4, kDV)) = make_float4(x[0], x[1], x[2], x[3]);
        }
        __syncthreads();
        // ---------------------------------------------------------- a2: decayed operands
        {
            float2 off = make_float2(0.f, 0.f);
            for (int q = 0; q < rg; ++q) {
                const float2 t = *reinterpret_cast<const float2 *>(&s_tot[q * kD + 2 * cp]);
                off.x += t.x;
                off.y += t.y;
            }
            if (rg == 7)
                *reinterpret_cast<float2 *>(&s_gam[2 * cp]) =
                    make_float2(__expf(off.x + gl[7].x), __expf(off.y + gl[7].y));
            if (fminf(off.x, off.y) + gmin < KDA_MIN_CHUNK_LOG_DECAY ||
                fmaxf(off.x, off.y) + gmax > -KDA_MIN_CHUNK_LOG_DECAY)
                decay_bad = true;
            const float scale = rsqrtf((float)kD);
            // K-major swizzled byte offset of channel 2cp in a row, less the row part
            const uint32_t pbase1 = (uint32_t)((cp >> 5) * 16384 + ((cp & 3) << 2));
            const uint32_t pbase2 = (uint32_t)((cp >> 5) * 8192 + ((cp & 3) << 2));
            const uint32_t pchunk = (uint32_t)((cp & 31) >> 2);
#pragma unroll
            for (int r4 = 0; r4 < 8; r4 += 4) {
                float ka[4], kb[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int rr = r4 + u, r = rg * 8 + rr;
                    const bool valid = r < len;
                    const float gx = off.x + gl[rr].x, gy = off.y + gl[rr].y;
                    const float ex = __expf(gx), ey = __expf(gy);
                    const float ix = __expf(-gx), iy = __expf(-gy);
                    const uint32_t qraw = valid ? *reinterpret_cast<const uint32_t *>(sm + IN_Q + (r * kD + 2 * cp) * 2) : 0u;
                    const uint32_t kraw = valid ? *reinterpret_cast<const uint32_t *>(sm + IN_K + (r * kD + 2 * cp) * 2) : 0u;
                    const float2 qv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qraw));
                    const float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kraw));
                    const uint32_t sw = (pchunk ^ (uint32_t)(rr & 7)) << 4;  // (r & 7) == (rr & 7)
                    *reinterpret_cast<uint32_t *>(sm + O1 + pbase1 + r * 128 + sw) = pack_bf16x2(kv.x * ex, kv.y * ey);
                    *reinterpret_cast<uint32_t *>(sm + O1 + pbase1 + (64 + r) * 128 + sw) =
                        pack_bf16x2(qv.x * (scale * ex), qv.y * (scale * ey));
                    const float kix = kv.x * ix, kiy = kv.y * iy;
                    *reinterpret_cast<uint32_t *>(sm + O2 + pbase2 + r * 128 + sw) = pack_bf16x2(kix, kiy);
                    ka[u] = to_tf32(kix);
                    kb[u] = to_tf32(kiy);
                }
                // lanes 4-7 of every 8 store their odd channel first, so each store covers
                // 8 distinct swizzle positions (no bank conflict)
                const int rb = rg * 8 + r4, sel = (lane >> 2) & 1;
                const float4 va = make_float4(ka[0], ka[1], ka[2], ka[3]);
                const float4 vb = make_float4(kb[0], kb[1], kb[2], kb[3]);
                *reinterpret_cast<float4 *>(sm + O3 + km32(2 * cp + sel, rb, 128)) = sel ? vb : va;
                *reinterpret_cast<float4 *>(sm + O3 + km32(2 * cp + 1 - sel, rb, 128)) = sel ? va : vb;
            }
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ---------------------------------------------------------- a3: G1
        if (tid == 0) {
            tc_fence_after_sync();
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t p = s >> 2, w = (s & 3) * 32;
                mma_bf16(tmem + TM_D1, kdesc(sb + O1 + p * 16384 + w), kdesc(sb + O2 + p * 8192 + w),
                         IDESC_G1, s > 0);
            }
            mma_commit(&bar_mma);
        }
        ok = mbar_wait_ns(&bar_mma, ph_mma, kWaitNs);
        if (__syncthreads_or(!ok)) { timed_out = true; mma_pending = true; break; }
        ph_mma ^= 1;
        tc_fence_after_sync();

        if (quarter < 2) {  // lanes 0..63: rows of Kg Ki^T -> A (fp32, strict lower, beta rows)
            const int r = quarter * 32 + lane;
            const float br = s_beta[r];
            float v[16];
            tmem_ld16(tmem + TM_D1 + lane_off + part * 16, v);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 16; u += 4) {
                const int col = part * 16 + u;
                *reinterpret_cast<float4 *>(sA + r * kLdS + col) =
                    make_float4(col < r ? br * v[u] : 0.f, col + 1 < r ? br * v[u + 1] : 0.f,
                                col + 2 < r ? br * v[u + 2] : 0.f, col + 3 < r ? br * v[u + 3] : 0.f);
            }
        } else {  // lanes 64..127: rows of Qg Ki^T -> Aqk (bf16, lower incl. diagonal)
            const int r = (quarter - 2) * 32 + lane;
            float v[16];
            tmem_ld16(tmem + TM_D1 + lane_off + part * 16, v);
            tmem_ld_wait();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float x[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) x[u] = (part * 16 + hh * 8 + u) <= r ? v[hh * 8 + u] : 0.f;
                *reinterpret_cast<uint4 *>(sm + O8 + km16(r, part * 16 + hh * 8, 64)) = pack_bf16x8(x);
            }
        }
        tc_fence_before_sync();
        __syncthreads();

        // ---------------------------------------------------------- a4: T = (I + A)^-1
        // Recursive doubling on the unit lower-triangular system: invert the four
        // 16 x 16 diagonal blocks, then the two 16 x 16 blocks below them
        // (T_10 = -T_11 A_10 T_00, T_32 = -T_33 A_32 T_22), then the 32 x 32
        // block T_[2:4][0:2] = -T_[2:4][2:4] A_[2:4][0:2] T_[0:2][0:2].
        if (tid < 64) {  // diagonal blocks, one column per thread
            const int b = (tid >> 4) * 16, cc = tid & 15;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc = 0.f;
#pragma unroll
                for (int m = 0; m < r; ++m) acc += sA[(b + r) * kLdS + b + m] * x[m];
                x[r] = r < cc ? 0.f : (r == cc ? 1.f : -acc);
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) sT[(b + r) * kLdS + b + cc] = x[r];
        }
        __syncthreads();
        {  // X = A_{R,R-1} T_{R-1,R-1} for (R0, C0) = (16, 0), (48, 32)
            const int b = tid >> 8, rr = (tid >> 4) & 15, cc = tid & 15;
            const int R0 = 16 + 32 * b, C0 = 32 * b;
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const float a = sA[(R0 + rr) * kLdS + C0 + m], t = sT[(C0 + m) * kLdS + C0 + cc];
                acc += m >= cc ? a * t : 0.f;
            }
            sX[(b * 16 + rr) * kLdX + cc] = acc;
        }
        __syncthreads();
        {  // T_{R,R-1} = -T_RR X
            const int b = tid >> 8, rr = (tid >> 4) & 15, cc = tid & 15;
            const int R0 = 16 + 32 * b, C0 = 32 * b;
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const float t = sT[(R0 + rr) * kLdS + R0 + m], x = sX[(b * 16 + m) * kLdX + cc];
                acc += m <= rr ? t * x : 0.f;
            }
            sT[(R0 + rr) * kLdS + C0 + cc] = -acc;
        }
        __syncthreads();
        if (tid < 256) {  // X2 = A[32:64][0:32] T[0:32][0:32]: row r, columns c..c+3 per thread
            const int r = tid >> 3, c = (tid & 7) * 4, k0 = c & 16;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k4 = 0; k4 < 32; k4 += 4) {
                if (k4 < k0) continue;
                const float4 a = *reinterpret_cast<const float4 *>(sA + (32 + r) * kLdS + k4);
                const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 t = *reinterpret_cast<const float4 *>(sT + (k4 + u) * kLdS + c);
                    acc.x += av[u] * t.x; acc.y += av[u] * t.y; acc.z += av[u] * t.z; acc.w += av[u] * t.w;
                }
            }
            *reinterpret_cast<float4 *>(sX + r * kLdX + c) = acc;
        }
        __syncthreads();
        if (tid < 256) {  // T[32:64][0:32] = -T[32:64][32:64] X2
            const int r = tid >> 3, c = (tid & 7) * 4;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int m4 = 0; m4 < 32; m4 += 4) {
                const float4 t = *reinterpret_cast<const float4 *>(sT + (32 + r) * kLdS + 32 + m4);
                const float tv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float tm = m4 + u <= r ? tv[u] : 0.f;  // T22 is lower triangular
                    const float4 x = *reinterpret_cast<const float4 *>(sX + (m4 + u) * kLdX + c);
                    acc.x += tm * x.x; acc.y += tm * x.y; acc.z += tm * x.z; acc.w += tm * x.w;
                }
            }
            *reinterpret_cast<float4 *>(sT + (32 + r) * kLdS + c) = make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        }
        __syncthreads();
        // T' = T diag(beta): bf16 (for W) and tf32 (for U~)
        {
            const int r = tid >> 3, s8 = (tid & 7) * 8;
            const float4 ta = *reinterpret_cast<const float4 *>(sT + r * kLdS + s8);
            const float4 tb = *reinterpret_cast<const float4 *>(sT + r * kLdS + s8 + 4);
            const float4 ba = *reinterpret_cast<const float4 *>(s_beta + s8);
            const float4 bb = *reinterpret_cast<const float4 *>(s_beta + s8 + 4);
            const float tv[8] = {ta.x, ta.y, ta.z, ta.w, tb.x, tb.y, tb.z, tb.w};
            const float bv[8] = {ba.x, ba.y, ba.z, ba.w, bb.x, bb.y, bb.z, bb.w};
            float t[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) t[u] = s8 + u <= r ? tv[u] * bv[u] : 0.f;
            *reinterpret_cast<uint4 *>(sm + O4 + km16(r, s8, 64)) = pack_bf16x8(t);
            *reinterpret_cast<float4 *>(sm + O5 + km32(r, s8, 128)) =
                make_float4(to_tf32(t[0]), to_tf32(t[1]), to_tf32(t[2]), to_tf32(t[3]));
            *reinterpret_cast<float4 *>(sm + O5 + km32(r, s8 + 4, 128)) =
                make_float4(to_tf32(t[4]), to_tf32(t[5]), to_tf32(t[6]), to_tf32(t[7]));
        }
        fence_proxy_async_smem();
        __syncthreads();

        // ---------------------------------------------------------- a5: GW, GU; next inputs
        if (tid == 0) {
            if (c + 1 < nchunks)
                issue_chunk_loads(sm, &tm_q, &tm_k, &tm_la, &tm_v, &bar_tma, h, j0,
                                  (int)(c0 + kC));
            tc_fence_after_sync();
#pragma unroll
            for (int s = 0; s < 4; ++s)  // W = T' Kg (M = 64); Kg read MN-major from O1 rows 0-63
                mma_bf16(tmem + TM_DW, kdesc(sb + O4 + s * 32),
                         sdesc(sb + O1 + s * 2048, 16384, 1024, kSw128B), IDESC_GW, s > 0);
#pragma unroll
            for (int s = 0; s < 8; ++s) {  // U~ = [T' ; 0] V  (tf32)
                const uint32_t p = s >> 2, w = (s & 3) * 32;
                mma_tf32(tmem + TM_D3, kdesc(sb + O5 + p * 16384 + w), kdesc(sb + O6 + p * 4096 + w),
                         IDESC_GU, s > 0);
            }
            mma_commit(&bar_mma);
        }
        tma_pending = c + 1 < nchunks;
        ok = mbar_wait_ns(&bar_mma, ph_mma, kWaitNs);
        if (__syncthreads_or(!ok)) { timed_out = true; mma_pending = true; break; }
        ph_mma ^= 1;
        tc_fence_after_sync();

        {  // -W into rows 0-63 of O1 (Kg no longer needed).  The M = 64 accumulator
           // keeps row 16q + l in lane l < 16 of lane quarter q; this warp takes 32
           // of the 128 columns.
            const int r = quarter * 16 + (lane & 15);
#pragma unroll
            for (int cb = 0; cb < 32; cb += 16) {
                float v[16];
                tmem_ld16(tmem + TM_DW + lane_off + part * 32 + cb, v);
                tmem_ld_wait();
                if (lane < 16) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        float x[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) x[u] = -v[hh * 8 + u];
                        *reinterpret_cast<uint4 *>(sm + O1 + km16(r, part * 32 + cb + hh * 8, 128)) =
                            pack_bf16x8(x);
                    }
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();

        // ---------------------------------------------------------- a6: G3 -> u, Qg S
        if (tid == 0) {
            tc_fence_after_sync();
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t p = s >> 2, w = (s & 3) * 32;
                mma_bf16(tmem + TM_D3, kdesc(sb + O1 + p * 16384 + w), kdesc(sb + O7 + p * 4096 + w),
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
                *reinterpret_cast<uint32_t *>(sm + O9 + km16(j, re, kDV)) = pack_bf16x2(lo, hi);
                *reinterpret_cast<float2 *>(sm + O10 + km32(j, re, kDV)) = make_float2(to_tf32(lo), to_tf32(hi));
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
                mma_bf16(tmem + TM_D3, kdesc(sb + O4 + s * 32), kdesc(sb + O9 + s * 32), IDESC_G3, 1);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                const uint32_t p = s >> 2, w = (s & 3) * 32;
                mma_tf32(tmem + TM_D5, kdesc(sb + O3 + p * 16384 + w), kdesc(sb + O10 + p * 4096 + w),
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
            if (r < len)
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
                *reinterpret_cast<uint32_t *>(sm + O7 + km16(jp + 4 * odd + u, ie, kDV)) = pack_bf16x2(lo, hi);
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
    } else {
        float *dst = final_state + st_off;
#pragma unroll
        for (int q = 0; q < 2; ++q)
            *reinterpret_cast<float4 *>(dst + 4 * q) = make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
    }
    if (decay_bad) atomicOr(status, DEV_ERR_DECAY);
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// [T, H, 128] token-major tensor; box = 64 tokens x 1 head x box_x channels.
bool make_map(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, int64_t T, int H,
              uint32_t esz, uint32_t box_x)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)kD * esz, (cuuint64_t)H * kD * esz};
    const cuuint32_t box[3] = {box_x, 1, (cuuint32_t)kC};
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (configured_device != dev) {
        err = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)kSmemDyn);
        if (err != cudaSuccess) return err;
        configured_device = dev;
    }
    CUtensorMap tq, tk, tla, tv;
    if (!make_map(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.q, p.total_tokens, p.num_heads, 2, kD) ||
        !make_map(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.k, p.total_tokens, p.num_heads, 2, kD) ||
        !make_map(&tla, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.log_alpha, p.total_tokens, p.num_heads, 4,
                  kD) ||
        !make_map(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.v, p.total_tokens, p.num_heads, 2, kDV))
        return cudaErrorInvalidValue;
    dim3 grid(kD / kDV, p.num_heads, p.num_seqs);
    prefill_tc_kernel<<<grid, kTcThreads, kSmemDyn, p.stream>>>(
        tq, tk, tla, tv, p.beta, p.cu_seqlens, p.total_tokens, p.num_heads, p.init_state,
        static_cast<__nv_bfloat16 *>(p.o), p.final_state, p.status, p.order);
    return cudaGetLastError();
}

}  // namespace kda
