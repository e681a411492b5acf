// tc_common.cuh -- pieces shared by the tensor-core prefill kernels (the fused
// single-kernel prefill and the chunk / state kernel pair): shared-memory
// operand layouts, packing helpers, the chunk-local phases (in-chunk decay
// prefix, decayed operands, k-k / q-k matrices, UT solve, W epilogue) and the
// tensor-map set-up.  Every device function here is called by all threads of
// the CTA (NT = 256 or 512).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include <mutex>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace kda {
namespace tc {

using namespace ptx;

constexpr int kD = 128, kDV = 32, kC = 64, kThreads = 512;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s per wait before giving up
constexpr int kLdS = kC + 4;                 // row stride (floats) of A and T in the solve
constexpr int kLdX = 32 + 4;                 // row stride of the block products X (<= 32 x 32)
constexpr float kLog2e = 1.4426950408889634f;  // log2(e): e^x = 2^(x log2 e)

// 2^x by the hardware's approximate base-2 exponential (relative error about 2^-22;
// subnormal results flush to zero).  The in-chunk decay prefix is kept in log2 units,
// so each decay factor is this one instruction.
__device__ __forceinline__ float exp2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

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

// The bf16 high parts of a and b (round to nearest even), packed as pack_bf16x2 does, and
// the fp32 remainders a - hi(a), b - hi(b): one conversion for the pair, the remainders from
// the packed bits.
__device__ __forceinline__ uint32_t split_bf16x2(float a, float b, float &ra, float &rb)
{
    const uint32_t h = pack_bf16x2(a, b);
    ra = a - __uint_as_float(h << 16);
    rb = b - __uint_as_float(h & 0xffff0000u);
    return h;
}

// Eight fp16 values (round to nearest even); `ok` is cleared when one of them
// is outside the fp16 range or not finite.
__device__ __forceinline__ uint4 pack_f16x8(const float (&x)[8], bool &ok)
{
    uint32_t w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        ok &= fabsf(x[2 * u]) <= 65504.f && fabsf(x[2 * u + 1]) <= 65504.f;
        __half2 h = __floats2half2_rn(x[2 * u], x[2 * u + 1]);
        w[u] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Eight fp16 values (round to nearest even), no range check.
__device__ __forceinline__ uint4 pack_f16x8_plain(const float (&x)[8])
{
    uint32_t w[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        __half2 h = __floats2half2_rn(x[2 * u], x[2 * u + 1]);
        w[u] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ float bf16_at(const unsigned char *p)
{
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(p));
}

__device__ __forceinline__ void store_bf16(unsigned char *p, float x)
{
    *reinterpret_cast<__nv_bfloat16 *>(p) = __float2bfloat16_rn(x);
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&x)[8])
{
    return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                      pack_bf16x2(x[6], x[7]));
}

// A layout L provides byte offsets (from a 1024-aligned base) of:
//   IN_Q, IN_K [64][128] bf16 (the chunk's TMA boxes),
//   O1  [Kg ; Qg] (later [-W ; Qg]) bf16 K-major, 128 rows x 128,
//   O2  Ki bf16 K-major, 64 rows x 128,
//   O4  T' bf16 K-major, 64 rows x 64,
//   SOLVE_A, SOLVE_T, SOLVE_X  fp32 scratch over buffers that are dead by the solve.
// Operands that no MMA of the calling kernel reads (Ki^T tf32, Aqk, T' tf32,
// e^{g_last}) go to caller-given generic pointers: shared memory in the fused
// kernel, the chunk's record in global memory in the chunk kernel.  The byte
// images are the same either way.  NT (256 or 512) is the CTA size.

// ---------------------------------------------------------------- a1: prefix
// Thread = (channel pair cp: channels 2cp, 2cp+1; row group rg of R = 4096/NT
// rows).  Scans its rows of log_alpha (row stride `la_stride` floats, shared or
// global memory) in registers and leaves the group totals in s_tot.  With `scalar`
// each row holds one value, the decay of every key channel (scalar gate).  The
// prefix is kept in log2 units, g = log2(e) * sum(log alpha) (each add is one FMA),
// so that every decay factor e^(sum log alpha) = 2^g is a single exp2_approx.
template <int NT>
__device__ __forceinline__ void prefix_scan(const float *la, int la_stride, int len, float *s_tot,
                                            float2 (&gl)[4096 / NT], float &gmin, float &gmax, bool scalar = false)
{
    constexpr int R = 4096 / NT;
    const int tid = threadIdx.x, cp = tid & 63, rg = tid >> 6;
    float2 g = make_float2(0.f, 0.f);
    gmin = 0.f;
    gmax = 0.f;
    float2 x[R];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {  // all loads first (they may come from global memory)
        const int r = rg * R + rr;
        if (scalar) {
            const float a = r < len ? la[(size_t)r * la_stride] : 0.f;
            x[rr] = make_float2(a, a);
        } else {
            x[rr] = r < len ? *reinterpret_cast<const float2 *>(la + (size_t)r * la_stride + 2 * cp)
                            : make_float2(0.f, 0.f);
        }
    }
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        g.x = fmaf(x[rr].x, kLog2e, g.x);
        g.y = fmaf(x[rr].y, kLog2e, g.y);
        gl[rr] = g;
        gmin = fminf(gmin, fminf(g.x, g.y));
        gmax = fmaxf(gmax, fmaxf(g.x, g.y));
    }
    *reinterpret_cast<float2 *>(&s_tot[rg * kD + 2 * cp]) = g;
}

// ---------------------------------------------------------------- q/k L2 normalisation
// Reciprocal row norms of the chunk's raw q and k boxes (bf16 [64][128], row-major):
// rn[r] = 1 / max(|k_r|_2, eps) and rn[64 + r] the same for q_r.  The operand builders
// scale the raw values by them in fp32, so the normalised q, k are never rounded on
// their own.  One warp per row; each lane sums four channels.
template <int NT>
__device__ __forceinline__ void qk_row_inv_norms(const unsigned char *k_box, const unsigned char *q_box,
                                                 float *rn)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int row = warp; row < 2 * kC; row += NT / 32) {
        const unsigned char *box = row < kC ? k_box : q_box;
        const uint2 raw = *reinterpret_cast<const uint2 *>(box + ((row & (kC - 1)) * kD + 4 * lane) * 2);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&raw.y));
        float ss = a.x * a.x + a.y * a.y + b.x * b.x + b.y * b.y;
#pragma unroll
        for (int m = 16; m; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
        if (lane == 0) rn[row] = 1.f / fmaxf(sqrtf(ss), kQkNormEps);
    }
}

// ---------------------------------------------------------------- a2: operands
// After a barrier following prefix_scan (g in log2 units, e^g below meaning
// 2^g): Kg = k e^g and Qg = scale q e^g into
// O1, Ki = k e^-g into O2 (bf16) and, when KI_T, into o3 (tf32, transposed,
// K-major 128 rows x 64), e^{g_last} into gam[128].  When off_tot is given it
// receives this thread's group offset and the chunk total of g for its channel
// pair.  With NORM and rn (qk_row_inv_norms, after a barrier) q and k rows are normalised
// first; without NORM rn is ignored and the code is the plain operand build.
// Returns true when the in-chunk cumulative decay left the supported range.
template <class L, int NT, bool KI_T = true, bool NORM = false>
__device__ __forceinline__ bool decayed_operands(unsigned char *sm, int len, const float *s_tot,
                                                 unsigned char *o3, float *gam,
                                                 const float2 (&gl)[4096 / NT], float gmin, float gmax,
                                                 float2 *off_tot = nullptr, const float *rn = nullptr)
{
    constexpr int R = 4096 / NT, G = NT / 64;
    const int tid = threadIdx.x, lane = tid & 31, cp = tid & 63, rg = tid >> 6;
    float2 off = make_float2(0.f, 0.f), tot = make_float2(0.f, 0.f);
#pragma unroll
    for (int q = 0; q < G; ++q) {
        const float2 t = *reinterpret_cast<const float2 *>(&s_tot[q * kD + 2 * cp]);
        if (q < rg) {
            off.x += t.x;
            off.y += t.y;
        }
        tot.x += t.x;
        tot.y += t.y;
    }
    if (off_tot) {
        off_tot[0] = off;
        off_tot[1] = tot;
    }
    if (rg == G - 1)
        *reinterpret_cast<float2 *>(&gam[2 * cp]) =
            make_float2(exp2_approx(off.x + gl[R - 1].x), exp2_approx(off.y + gl[R - 1].y));
    // the supported range of the cumulative log-decay, in the prefix's log2 units
    const bool bad = fminf(off.x, off.y) + gmin < KDA_MIN_CHUNK_LOG_DECAY * kLog2e ||
                     fmaxf(off.x, off.y) + gmax > -KDA_MIN_CHUNK_LOG_DECAY * kLog2e;
    const float scale = rsqrtf((float)kD);
    // K-major swizzled byte offset of channel 2cp in a row, less the row part
    const uint32_t pbase1 = (uint32_t)((cp >> 5) * 16384 + ((cp & 3) << 2));
    const uint32_t pbase2 = (uint32_t)((cp >> 5) * 8192 + ((cp & 3) << 2));
    const uint32_t pchunk = (uint32_t)((cp & 31) >> 2);
#pragma unroll
    for (int r4 = 0; r4 < R; r4 += 4) {
        float ka[4], kb[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int rr = r4 + u, r = rg * R + rr;
            const bool valid = r < len;
            const float gx = off.x + gl[rr].x, gy = off.y + gl[rr].y;  // log2 units
            const float ex = exp2_approx(gx), ey = exp2_approx(gy);
            const float ix = exp2_approx(-gx), iy = exp2_approx(-gy);
            const uint32_t qraw = valid ? *reinterpret_cast<const uint32_t *>(sm + L::IN_Q + (r * kD + 2 * cp) * 2) : 0u;
            const uint32_t kraw = valid ? *reinterpret_cast<const uint32_t *>(sm + L::IN_K + (r * kD + 2 * cp) * 2) : 0u;
            float2 qv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qraw));
            float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kraw));
            if (NORM && rn) {
                const float kn = rn[r], qn = rn[kC + r];
                kv.x *= kn; kv.y *= kn;
                qv.x *= qn; qv.y *= qn;
            }
            const uint32_t sw = (pchunk ^ (uint32_t)(rr & 7)) << 4;  // (r & 7) == (rr & 7)
            *reinterpret_cast<uint32_t *>(sm + L::O1 + pbase1 + r * 128 + sw) = pack_bf16x2(kv.x * ex, kv.y * ey);
            *reinterpret_cast<uint32_t *>(sm + L::O1 + pbase1 + (64 + r) * 128 + sw) =
                pack_bf16x2(qv.x * (scale * ex), qv.y * (scale * ey));
            const float kix = kv.x * ix, kiy = kv.y * iy;
            *reinterpret_cast<uint32_t *>(sm + L::O2 + pbase2 + r * 128 + sw) = pack_bf16x2(kix, kiy);
            ka[u] = to_tf32(kix);
            kb[u] = to_tf32(kiy);
        }
        if (!KI_T) continue;
        // lanes 4-7 of every 8 store their odd channel first, so each store covers
        // 8 distinct swizzle positions (no bank conflict in shared memory)
        const int rb = rg * R + r4, sel = (lane >> 2) & 1;
        const float4 va = make_float4(ka[0], ka[1], ka[2], ka[3]);
        const float4 vb = make_float4(kb[0], kb[1], kb[2], kb[3]);
        *reinterpret_cast<float4 *>(o3 + km32(2 * cp + sel, rb, 128)) = sel ? vb : va;
        *reinterpret_cast<float4 *>(o3 + km32(2 * cp + 1 - sel, rb, 128)) = sel ? va : vb;
    }
    return bad;
}

// ---------------------------------------------------------------- a3: G1 + epilogue
// D1 = [Kg ; Qg] Ki^T (M = 128, N = 64, K = 128); one thread issues.
template <class L>
__device__ __forceinline__ void issue_g1(uint32_t sb, uint32_t d1)
{
    constexpr uint32_t idesc = idesc_bf16(128, 64, false, false);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const uint32_t p = s >> 2, w = (s & 3) * 32;
        mma_bf16(d1, kdesc(sb + L::O1 + p * 16384 + w), kdesc(sb + L::O2 + p * 8192 + w), idesc, s > 0);
    }
}

// Lanes 0-63 of D1 -> A = strict-lower(beta_r . Kg Ki^T) (fp32, solve scratch);
// lanes 64-127 -> Aqk = lower(Qg Ki^T) (bf16 operand image at aq).
template <class L, int NT>
__device__ __forceinline__ void kk_epilogue(unsigned char *sm, uint32_t d1, const float *s_beta,
                                            unsigned char *aq)
{
    constexpr int CW = 64 / (NT / 128);  // columns per thread
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quarter = warp & 3, part = warp >> 2;
#pragma unroll
    for (int cb = 0; cb < CW; cb += 16) {
        const int c0 = part * CW + cb;
        float v[16];
        tmem_ld16(d1 + ((uint32_t)(quarter * 32) << 16) + c0, v);
        tmem_ld_wait();
        if (quarter < 2) {
            const int r = quarter * 32 + lane;
            const float br = s_beta[r];
            float *sA = reinterpret_cast<float *>(sm + L::SOLVE_A);
#pragma unroll
            for (int u = 0; u < 16; u += 4) {
                const int col = c0 + u;
                *reinterpret_cast<float4 *>(sA + r * kLdS + col) =
                    make_float4(col < r ? br * v[u] : 0.f, col + 1 < r ? br * v[u + 1] : 0.f,
                                col + 2 < r ? br * v[u + 2] : 0.f, col + 3 < r ? br * v[u + 3] : 0.f);
            }
        } else {
            const int r = (quarter - 2) * 32 + lane;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float x[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) x[u] = (c0 + hh * 8 + u) <= r ? v[hh * 8 + u] : 0.f;
                *reinterpret_cast<uint4 *>(aq + km16(r, c0 + hh * 8, 64)) = pack_bf16x8(x);
            }
        }
    }
}

// ---------------------------------------------------------------- a4: UT solve
// T = (I + A)^-1 by recursive doubling on the unit lower-triangular system:
// the four 16 x 16 diagonal blocks, then T_10 = -T_11 A_10 T_00 and
// T_32 = -T_33 A_32 T_22, then T_[2:4][0:2] = -T_[2:4][2:4] A_[2:4][0:2] T_[0:2][0:2].
// solve_ut_core leaves T (lower triangle, unit diagonal) in SOLVE_T.  With
// INPLACE (SOLVE_T == SOLVE_A) each block of T overwrites the block of A it
// replaces once no later step reads that block of A; the strictly upper blocks
// of T are never read.  solve_ut then writes T' = T diag(beta) as bf16 (O4) and
// tf32 (image at tt with tt_rows rows per 32-column panel).  Both contain barriers.
template <class L, int NT, bool INPLACE>
__device__ __forceinline__ void solve_ut_core(unsigned char *sm)
{
    static_assert(!INPLACE || L::SOLVE_A == L::SOLVE_T, "in-place solve needs SOLVE_A == SOLVE_T");
    const int tid = threadIdx.x;
    const float *sA = reinterpret_cast<const float *>(sm + L::SOLVE_A);
    float *sT = reinterpret_cast<float *>(sm + L::SOLVE_T);
    float *sX = reinterpret_cast<float *>(sm + L::SOLVE_X);
    float x[16];
    const int b = (tid >> 4) * 16, cc = tid & 15;
    if (tid < 64) {  // diagonal blocks, one column per thread
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < r; ++m) acc += sA[(b + r) * kLdS + b + m] * x[m];
            x[r] = r < cc ? 0.f : (r == cc ? 1.f : -acc);
        }
    }
    if (INPLACE) __syncthreads();  // every column has read its diagonal block of A
    if (tid < 64) {
#pragma unroll
        for (int r = 0; r < 16; ++r) sT[(b + r) * kLdS + b + cc] = x[r];
    }
    __syncthreads();
#pragma unroll
    for (int e = tid; e < 512; e += NT) {  // X = A_{R,R-1} T_{R-1,R-1} for (R0, C0) = (16, 0), (48, 32)
        const int b = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
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
#pragma unroll
    for (int e = tid; e < 512; e += NT) {  // T_{R,R-1} = -T_RR X
        const int b = e >> 8, rr = (e >> 4) & 15, cc = e & 15;
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
}

// Sum of a float4 over the two lanes of an adjacent pair (lane ^ 1); every lane of the
// warp takes part.
__device__ __forceinline__ float4 add_pair_lanes(float4 a)
{
    a.x += __shfl_xor_sync(0xffffffffu, a.x, 1);
    a.y += __shfl_xor_sync(0xffffffffu, a.y, 1);
    a.z += __shfl_xor_sync(0xffffffffu, a.z, 1);
    a.w += __shfl_xor_sync(0xffffffffu, a.w, 1);
    return a;
}

// T' = T diag(beta) for one quad of four columns of row r, as bf16 high and low parts
// into the [t][s] images at L::O4 and L::TL (8 bytes each).
template <class L>
__device__ __forceinline__ void store_tprime_quad(unsigned char *sm, int r, int c, float4 t, const float *s_beta)
{
    const float4 bq = *reinterpret_cast<const float4 *>(s_beta + c);
    const float tv[4] = {t.x * bq.x, t.y * bq.y, t.z * bq.z, t.w * bq.w};
    float lo[4];
    const uint32_t h01 = split_bf16x2(tv[0], tv[1], lo[0], lo[1]), h23 = split_bf16x2(tv[2], tv[3], lo[2], lo[3]);
    *reinterpret_cast<uint2 *>(sm + L::O4 + km16(r, c, 64)) = make_uint2(h01, h23);
    *reinterpret_cast<uint2 *>(sm + L::TL + km16(r, c, 64)) = make_uint2(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]));
}

// solve_ut_doubling: the same T, in place (SOLVE_T == SOLVE_A): the four 16 x 16
// diagonal blocks by column-parallel forward substitution (one warp per block, one
// lane per column), then recursive doubling: for block size b = 16, 32 and every
// pair of b x b diagonal blocks, X = A_10 T_00 and T_10 = -T_11 X (X in SOLVE_X).
// Each output quad is one thread's float4; the strictly upper parts of A, which
// the k-k epilogue zeroed, stand in for the zero upper parts of T, so no product
// needs a mask.  The last level writes T' = T diag(beta) straight into its bf16
// high and low images (L::O4, L::TL): the diagonal 32 x 32 quadrants while X is
// formed, the lower-left one as it is formed, zeros above; T itself is not
// completed in fp32.  Called by the NT compute threads only; they synchronise at
// named barrier 1, and the caller fences and synchronises before the images are read.
template <class L, int NT>
__device__ __forceinline__ void solve_ut_doubling(unsigned char *sm, const float *s_beta)
{
    static_assert(L::SOLVE_A == L::SOLVE_T, "the doubling solve works in place");
    static_assert(NT == 256, "the last level maps one output quad to each thread");
    // the NT compute threads (warps 0 .. NT/32 - 1) meet at named barrier 1; a CTA's
    // other warps do not take part in the solve
    auto sync = [] { asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory"); };
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float *sT = reinterpret_cast<float *>(sm + L::SOLVE_T);  // holds A until overwritten
    float *sX = reinterpret_cast<float *>(sm + L::SOLVE_X);
    // 1. Warp w < 4 inverts the diagonal 16 x 16 block at 16w on its own: lane c < 16 forms
    //    column c by forward substitution, updating every later row's sum as soon as x[m]
    //    is known (the sixteen steps each add one FMA to the dependency chain).  The block of
    //    A is read in full before any lane overwrites it with its column of T.
    if (warp < 4 && lane < 16) {
        const int b0 = warp * 16, cc = lane;
        float acc[16], x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) acc[r] = 0.f;
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            x[m] = m < cc ? 0.f : (m == cc ? 1.f : -acc[m]);
#pragma unroll
            for (int r = m + 1; r < 16; ++r) acc[r] = fmaf(sT[(b0 + r) * kLdS + b0 + m], x[m], acc[r]);
        }
        __syncwarp(0xffffu);  // every column has read the block of A
#pragma unroll
        for (int r = 0; r < 16; ++r) sT[(b0 + r) * kLdS + b0 + cc] = x[r];
    }
    sync();
    // 2. The 16 level across the CTA: two pairs of 16 x 16 blocks, 128 output quads, two
    //    adjacent lanes per quad (each takes every other group of four m; a shuffle adds
    //    the halves).
    {
        constexpr int b = 16, quads = 4, items = 32 * quads;
        // X = A_10 T_00: a warp shares one column quad cq over the 32 rows of X, so the
        // loop can start at m = cq (T_00[m][cq..cq+3] = 0 for m < cq); A is read four m at
        // a time (rows 272 bytes apart: conflict-free float4 loads)
        for (int it = tid; it < items * 2; it += NT) {
            const int e = it / 2, half = it % 2;
            const int xr = e & 31, cq = (e >> 5) * 4, p = xr / b, rr = xr % b;
            const int R0 = 2 * b * p + b, C0 = 2 * b * p;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int m4 = cq + 4 * half; m4 < b; m4 += 8) {
                const float4 a = *reinterpret_cast<const float4 *>(sT + (R0 + rr) * kLdS + C0 + m4);
                const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 t = *reinterpret_cast<const float4 *>(sT + (C0 + m4 + u) * kLdS + C0 + cq);
                    acc.x += av[u] * t.x; acc.y += av[u] * t.y; acc.z += av[u] * t.z; acc.w += av[u] * t.w;
                }
            }
            acc = add_pair_lanes(acc);
            if (half == 0) *reinterpret_cast<float4 *>(sX + xr * kLdX + cq) = acc;
        }
        sync();
        // T_10 = -T_11 X over A_10: row rr needs m <= rr only (T_11 is lower triangular);
        // a warp covers few consecutive rows, so its trip counts stay close
        for (int it = tid; it < items * 2; it += NT) {
            const int e = it / 2, half = it % 2;
            const int xr = e / quads, cq = (e % quads) * 4, p = xr / b, rr = xr % b;
            const int R0 = 2 * b * p + b, C0 = 2 * b * p;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int m4 = 4 * half; m4 <= rr; m4 += 8) {
                const float4 t = *reinterpret_cast<const float4 *>(sT + (R0 + rr) * kLdS + R0 + m4);
                const float tv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 x = *reinterpret_cast<const float4 *>(sX + (p * b + m4 + u) * kLdX + cq);
                    acc.x += tv[u] * x.x; acc.y += tv[u] * x.y; acc.z += tv[u] * x.z; acc.w += tv[u] * x.w;
                }
            }
            acc = add_pair_lanes(acc);
            if (half == 0)
                *reinterpret_cast<float4 *>(sT + (R0 + rr) * kLdS + C0 + cq) =
                    make_float4(-acc.x, -acc.y, -acc.z, -acc.w);
        }
        sync();
    }
    // 3. The 32 level: one pair of 32 x 32 blocks, one output quad per thread.  T_00 and
    //    T_11 are final now: each thread also sends one quad of each to the T' images and
    //    zeros one quad of the upper-right quadrant.
    {
        const int xr = tid & 31, cq = (tid >> 5) * 4;  // X = A_10 T_00 (rows 32.., columns 0..31)
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int m4 = cq; m4 < 32; m4 += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(sT + (32 + xr) * kLdS + m4);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 t = *reinterpret_cast<const float4 *>(sT + (m4 + u) * kLdS + cq);
                acc.x += av[u] * t.x; acc.y += av[u] * t.y; acc.z += av[u] * t.z; acc.w += av[u] * t.w;
            }
        }
        *reinterpret_cast<float4 *>(sX + xr * kLdX + cq) = acc;
        const int r = tid >> 3, c = (tid & 7) * 4;  // this thread's quad of each 32 x 32 quadrant
        store_tprime_quad<L>(sm, r, c, *reinterpret_cast<const float4 *>(sT + r * kLdS + c), s_beta);
        store_tprime_quad<L>(sm, 32 + r, 32 + c, *reinterpret_cast<const float4 *>(sT + (32 + r) * kLdS + 32 + c),
                             s_beta);
        *reinterpret_cast<uint2 *>(sm + L::O4 + km16(r, 32 + c, 64)) = make_uint2(0u, 0u);
        *reinterpret_cast<uint2 *>(sm + L::TL + km16(r, 32 + c, 64)) = make_uint2(0u, 0u);
    }
    sync();
    {
        // T_10 = -T_11 X straight into the T' images (row 32 + rr, columns cq..cq+3)
        const int rr = tid >> 3, cq = (tid & 7) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int m4 = 0; m4 <= rr; m4 += 4) {
            const float4 t = *reinterpret_cast<const float4 *>(sT + (32 + rr) * kLdS + 32 + m4);
            const float tv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 x = *reinterpret_cast<const float4 *>(sX + (m4 + u) * kLdX + cq);
                acc.x += tv[u] * x.x; acc.y += tv[u] * x.y; acc.z += tv[u] * x.z; acc.w += tv[u] * x.w;
            }
        }
        store_tprime_quad<L>(sm, 32 + rr, cq, make_float4(-acc.x, -acc.y, -acc.z, -acc.w), s_beta);
    }
}

template <class L, int NT>
__device__ __forceinline__ void solve_ut(unsigned char *sm, const float *s_beta, unsigned char *tt,
                                         int tt_rows)
{
    solve_ut_core<L, NT, false>(sm);
    const int tid = threadIdx.x;
    const float *sT = reinterpret_cast<const float *>(sm + L::SOLVE_T);
#pragma unroll
    for (int e = tid; e < 512; e += NT) {  // T' = T diag(beta): bf16 (for W) and tf32 (for U~)
        const int r = e >> 3, s8 = (e & 7) * 8;
        const float4 ta = *reinterpret_cast<const float4 *>(sT + r * kLdS + s8);
        const float4 tb = *reinterpret_cast<const float4 *>(sT + r * kLdS + s8 + 4);
        const float4 ba = *reinterpret_cast<const float4 *>(s_beta + s8);
        const float4 bb = *reinterpret_cast<const float4 *>(s_beta + s8 + 4);
        const float tv[8] = {ta.x, ta.y, ta.z, ta.w, tb.x, tb.y, tb.z, tb.w};
        const float bv[8] = {ba.x, ba.y, ba.z, ba.w, bb.x, bb.y, bb.z, bb.w};
        float t[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) t[u] = s8 + u <= r ? tv[u] * bv[u] : 0.f;
        *reinterpret_cast<uint4 *>(sm + L::O4 + km16(r, s8, 64)) = pack_bf16x8(t);
        *reinterpret_cast<float4 *>(tt + km32(r, s8, tt_rows)) =
            make_float4(to_tf32(t[0]), to_tf32(t[1]), to_tf32(t[2]), to_tf32(t[3]));
        *reinterpret_cast<float4 *>(tt + km32(r, s8 + 4, tt_rows)) =
            make_float4(to_tf32(t[4]), to_tf32(t[5]), to_tf32(t[6]), to_tf32(t[7]));
    }
}

// ---------------------------------------------------------------- a5: W
// W = T' Kg (M = 64, N = 128, K = 64); Kg is read MN-major from O1 rows 0-63.
template <class L>
__device__ __forceinline__ void issue_gw(uint32_t sb, uint32_t dw)
{
    constexpr uint32_t idesc = idesc_bf16(64, 128, false, true);
#pragma unroll
    for (int s = 0; s < 4; ++s)
        mma_bf16(dw, kdesc(sb + L::O4 + s * 32), sdesc(sb + L::O1 + s * 2048, 16384, 1024, kSw128B),
                 idesc, s > 0);
}

// -W into rows 0-63 of O1 (Kg no longer needed).  The M = 64 accumulator keeps row
// 16q + l in lane l < 16 of lane quarter q; a warp takes 128/(NT/128) columns, its two
// half-warps one half each (16-lane loads, so every thread of the warp works).
template <class L, int NT>
__device__ __forceinline__ void w_epilogue(unsigned char *sm, uint32_t dw)
{
    constexpr int CW = 128 / (NT / 128), HW = CW / 2;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quarter = warp & 3, part = warp >> 2;
    const int r = quarter * 16 + (lane & 15), c0 = part * CW + (lane >> 4) * HW;
#pragma unroll
    for (int cb = 0; cb < HW; cb += 16) {
        float v[16];
        tmem_ld16x2_x16<HW>(dw + ((uint32_t)(quarter * 32) << 16) + part * CW + cb, v);
        tmem_ld_wait();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) x[u] = -v[hh * 8 + u];
            *reinterpret_cast<uint4 *>(sm + L::O1 + km16(r, c0 + cb + hh * 8, 128)) = pack_bf16x8(x);
        }
    }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn()
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
inline bool make_map(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, int64_t T, int H,
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

// Sets the dynamic shared memory limit of `kern` once per device.
template <class K>
inline cudaError_t allow_smem(K kern, int bytes, int *configured_device)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (*configured_device != dev) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (err != cudaSuccess) return err;
        *configured_device = dev;
    }
    return cudaSuccess;
}

}  // namespace tc
}  // namespace kda
