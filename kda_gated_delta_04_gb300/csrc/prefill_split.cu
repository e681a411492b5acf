// prefill_split.cu -- the tensor-core prefill as two kernels (bf16 q/k/v,
// d_k = d_v = 128, fp32 state), sm_103a.
//
// Everything in a 64-token chunk that does not involve the running state is
// independent across chunks ("From 124M to 2.8T", chapter 3: parallel inside a
// chunk; "K3 attention, three-piece set": WY representation + UT transform).
// The chunk kernel, one CTA per (chunk, head) over every chunk at once, folds
// all of it into four matrices per chunk-head, so that the serial walk over the
// chunks is a single matrix product per chunk.  With g the in-chunk prefix of
// log alpha, gamma = e^{g_last}, Kg = k e^g, Qg = scale q e^g, Kd = k e^{g_last - g},
// Aqk = lower(Qg Ki^T), T' = (I + A)^-1 diag(beta) and W = T' Kg:
//
//   S_{c+1} = gamma . S_c + P V + N S_c      P  = Kd^T T'          (128 x 64)
//                                            N  = -Kd^T W           (128 x 128)
//   o_c     = Q' S_c + P2 V                  Q' = Qg - Aqk W        (64 x 128)
//                                            P2 = Aqk T'            (64 x 64)
//
// (u = T'V - W S is substituted into S <- gamma.(S + Ki^T u) and o = Qg S + Aqk u.)
// The record of a chunk-head holds N, Q' (bf16), P, P2 (fp16: the 10-bit
// mantissa P needs, at half the bytes of tf32) and gamma as the state kernel's
// MMA operand images, byte for byte.  P is formed from bf16 high/low splits of
// Kd and T' (hi.hi + hi.lo + lo.hi), which is more accurate than one tf32 product.
// The state kernel walks the chunks of one (sequence, head, 32-column value
// slice): per chunk one MMA group P V + N S on the critical path and the output
// group P2 V + Q' S beside it, issued by a second thread.
#include <climits>

#include "tc_common.cuh"

namespace kda {
namespace {

using namespace ptx;
using namespace tc;

// Record of one chunk-head.  N and Q' interleave by K panel, [N panel 0 | Q' panel 0 |
// N panel 1 | Q' panel 1], so that each K panel of the two is one 192-row operand image and
// the pair travels as one copy.
constexpr uint32_t R_NQ_PANEL = 24576;  // bytes from one K panel of N and Q' to the next
constexpr uint32_t R_N = 0;        // N  bf16 K-major, 128 rows per panel (rows i, K = j)
constexpr uint32_t R_Q = 16384;    // Q' bf16 K-major, 64 rows per panel  (rows t, K = j)
constexpr uint32_t R_P = 49152;    // P  fp16 K-major, 128 rows            (rows i, K = s)
constexpr uint32_t R_P2 = 65536;   // P2 fp16 K-major, 64 rows             (rows t, K = s)
constexpr uint32_t R_GM = 73728;   // gamma, 128 fp32
constexpr uint32_t kRecBytes = 74240;
static_assert(kRecBytes % 16 == 0, "records are moved by bulk copies");

// Chunk kernel: eight compute warps and one issuing warp (288 threads) and 105 KB
// of shared memory, so two CTAs share an SM and hide each other's latencies.  The
// issuing warp owns the barriers, the TMEM allocation, every MMA group and every
// bulk store, so the compute warps go on to their next phase as soon as a group is
// handed off.  CTAs take the chunks last to first, so the records the serial pass
// reads first are the ones written last (most likely still in L2).
constexpr int kChunkCompute = 256;                  // compute threads (warps 0-7)
constexpr int kChunkThreads = kChunkCompute + 32;   // + the issuing warp
constexpr int kChunkIssuer = kChunkCompute;         // its lane 0 issues
struct ChunkLayout {
    static constexpr uint32_t IN_K = 0, IN_Q = 16384;  // TMA boxes; k lives until the Kd build
    static constexpr uint32_t O2 = 32768;   // Ki bf16, 64 rows x 128 (B of the k-k product)
    static constexpr uint32_t O1 = 49152;   // [Kg ; Qg] -> [-W ; Qg] bf16, 128 rows x 128
    static constexpr uint32_t AQ = 81920;   // Aqk bf16 K-major 64 x 64 (prefix group totals before)
    static constexpr uint32_t O4 = 90112;   // T' high part bf16 [t][s]
    static constexpr uint32_t TL = 98304;   // T' low part bf16 [t][s]
    // in-place solve over the q box and Ki (both dead by then); Kd^T over the same bytes after it
    static constexpr uint32_t SOLVE_A = 16384, SOLVE_T = 16384, SOLVE_X = 16384 + kC * kLdS * 4;
    static constexpr uint32_t KDH = 16384, KDL = 32768;  // Kd^T high / low bf16 K-major, 128 rows x 64
    // record images staged for bulk stores, each over bytes dead by then:
    static constexpr uint32_t ST_P = 0;        // P over the k box (after the Kd build)
    static constexpr uint32_t ST_P2 = 90112;   // P2 over T' high (after the P products)
    // N's two K panels over Kd^T low and over Aqk and T' high (after N, Q''), then Q' over the
    // first once its store has read it: clear of the next item's boxes (k, q, log_alpha),
    // which are copied in meanwhile
    static constexpr uint32_t ST_A = 32768, ST_B = 81920;
    static constexpr uint32_t USED = 106496;
};
static_assert(ChunkLayout::ST_A >= ChunkLayout::IN_Q + 16384 && ChunkLayout::ST_A + 16384 <= ChunkLayout::O1 &&
                  ChunkLayout::ST_B >= ChunkLayout::O1 + 32768 && ChunkLayout::ST_B + 16384 <= ChunkLayout::USED,
              "record staging overlaps the boxes");
static_assert(ChunkLayout::SOLVE_X + 32 * kLdX * 4 <= ChunkLayout::O1, "solve scratch overlaps O1");

// State kernel (608 threads: sixteen state warps, two issuing warps, a copy warp) over a
// value slice of SV = 32 or 64 columns: two record stages, a ring of v slices, the V^T
// operand of two chunks and the S operand of two chunks.  The 32-column form has the
// shorter chain per chunk; the 64-column form halves the CTA count (and doubles the width
// of every tensor-core product group), which wins once the slices no longer fit in one
// wave of SMs.
template <int SV>
struct StateShape {
    static_assert(SV == 32 || SV == 64, "value slices of 32 or 64 columns");
    static constexpr uint32_t kVBytes = kC * SV * 2;    // one v slice [64 tokens][SV] bf16, and V^T fp16
    static constexpr uint32_t kSBytes = kD * SV * 2;    // the S operand, bf16
    static constexpr int kVRing = SV == 32 ? 4 : 3;     // v slices in flight
    static constexpr int kSCols = SV / 4;               // state columns per state-warp thread
    static constexpr uint32_t STAGE = 75776;            // record + padding to 1024 bytes
    static constexpr uint32_t VBOX = 2 * STAGE;         // kVRing x v slice
    static constexpr uint32_t VIMG = VBOX + kVRing * kVBytes;  // 2 x V^T fp16, SV rows x K 64
    static constexpr uint32_t O7 = VIMG + 2 * kVBytes;  // 2 x S bf16, MN-major, K 128 x SV columns
    static constexpr uint32_t USED = O7 + 2 * kSBytes;
    static constexpr uint32_t SMEM = USED + 1024;
    // TMEM columns: state increment (M = 128), outputs of two chunks (M = 64)
    static constexpr uint32_t TM_5 = 0, TM_O = SV, TMEM = SV == 32 ? 128 : 256;
    // The S operand (K = state row i, N = value column j): MN-major.  64 columns: rows of
    // 128 bytes, 128-byte swizzle (8-row atoms of 1024 bytes); 32 columns: rows of 64 bytes,
    // 64-byte swizzle (8-row atoms of 512 bytes).  SK: bytes per K step of 16 rows.
    static constexpr uint32_t SK = SV * 32;
    __device__ static uint32_t mn(int i, int j)
    {
        if (SV == 64) return km16(i, j, kD);
        return (uint32_t)(i * 64 + ((((j >> 3) ^ (i >> 1)) & 3) << 4) + ((j & 7) << 1));
    }
    __device__ static uint64_t sdesc_s(uint32_t addr)
    {
        return SV == 64 ? sdesc(addr, kSBytes, 1024, kSw128B) : sdesc(addr, 512, 512, kSw64B);
    }
    static constexpr uint32_t IDESC_PV = idesc_f16(128, SV, false, false);   // P V
    static constexpr uint32_t IDESC_NS = idesc_bf16(128, SV, false, true);   // N S (S MN-major)
    static constexpr uint32_t IDESC_P2V = idesc_f16(64, SV, false, false);   // P2 V
    static constexpr uint32_t IDESC_QS = idesc_bf16(64, SV, false, true);    // Q' S (S MN-major)
    static_assert(STAGE % 1024 == 0 && STAGE >= kRecBytes, "stage size");
    static_assert(VIMG % 1024 == 0 && O7 % 1024 == 0, "operand alignment");
    static_assert(SMEM <= 232448, "state kernel shared memory over the per-CTA limit");
    static_assert(TM_O + 2 * SV <= TMEM, "state kernel TMEM map");
};

constexpr uint32_t kChunkSmem = ChunkLayout::USED + 1024;

// ============================================================== chunk kernel
// TMEM columns: k-k / q-k product 0..63; then W 0..127, P2 128..191, P 192..255;
// then N 0..127, Q'' = Aqk(-W) 128..255.
constexpr uint32_t TC_W = 0, TC_P2 = 128, TC_P = 192, TC_N = 0, TC_Q = 128, kChunkTmem = 256;

// MN-major bf16 operand of 64-row K panels (rows = K index, 128-byte swizzled rows)
__device__ __forceinline__ uint64_t mndesc(uint32_t addr, uint32_t panel_stride)
{
    return sdesc(addr, panel_stride, 1024, kSw128B);
}

// Kd^T = (k e^{g_last - g})^T as bf16 high and low parts, K-major [i][s] at KDH
// and KDL.  Thread = (channel pair cp, row group rg) as in decayed_operands.
template <class L, int NT, bool NORM>
__device__ __forceinline__ void build_kd(unsigned char *sm, int len, const float2 (&gl)[4096 / NT],
                                         float2 off, float2 tot, const float *rn)
{
    constexpr int R = 4096 / NT;
    static_assert(R % 8 == 0, "row groups cover whole 8-column chunks");
    const int tid = threadIdx.x, lane = tid & 31, cp = tid & 63, rg = tid >> 6;
    const int sel = lane & 1;  // odd lanes store their odd channel first (no bank conflicts)
#pragma unroll
    for (int r8 = 0; r8 < R; r8 += 8) {
        uint32_t hxy[8];  // the high parts of channels (2cp, 2cp + 1) of row r8 + u
        float lx[8], ly[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int rr = r8 + u, r = rg * R + rr;
            const bool valid = r < len;
            const uint32_t kraw = valid ? *reinterpret_cast<const uint32_t *>(sm + L::IN_K + (r * kD + 2 * cp) * 2) : 0u;
            float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&kraw));
            if (NORM) {  // normalised k (KDA_FLAG_QK_L2NORM)
                kv.x *= rn[r];
                kv.y *= rn[r];
            }
            const float dx = kv.x * exp2_approx(tot.x - (off.x + gl[rr].x));  // log2 units
            const float dy = kv.y * exp2_approx(tot.y - (off.y + gl[rr].y));
            hxy[u] = split_bf16x2(dx, dy, lx[u], ly[u]);
        }
        const int s0 = rg * R + r8;
        // the high parts regrouped by channel (rows u, u + 1 per word, as pack_bf16x8 packs)
        const uint4 hxv = make_uint4(__byte_perm(hxy[0], hxy[1], 0x5410), __byte_perm(hxy[2], hxy[3], 0x5410),
                                     __byte_perm(hxy[4], hxy[5], 0x5410), __byte_perm(hxy[6], hxy[7], 0x5410));
        const uint4 hyv = make_uint4(__byte_perm(hxy[0], hxy[1], 0x7632), __byte_perm(hxy[2], hxy[3], 0x7632),
                                     __byte_perm(hxy[4], hxy[5], 0x7632), __byte_perm(hxy[6], hxy[7], 0x7632));
        const uint4 lxv = pack_bf16x8(lx), lyv = pack_bf16x8(ly);
        *reinterpret_cast<uint4 *>(sm + L::KDH + km16(2 * cp + sel, s0, 128)) = sel ? hyv : hxv;
        *reinterpret_cast<uint4 *>(sm + L::KDH + km16(2 * cp + 1 - sel, s0, 128)) = sel ? hxv : hyv;
        *reinterpret_cast<uint4 *>(sm + L::KDL + km16(2 * cp + sel, s0, 128)) = sel ? lyv : lxv;
        *reinterpret_cast<uint4 *>(sm + L::KDL + km16(2 * cp + 1 - sel, s0, 128)) = sel ? lxv : lyv;
    }
}

// Product group 2a: W = T' Kg (M = 64, N = 128) and, when outputs are wanted, P2 = Aqk T' (M = 64, N = 64).
template <class L>
__device__ __forceinline__ void issue_w_p2(uint32_t sb, uint32_t tmem, bool with_o)
{
    issue_gw<L>(sb, tmem + TC_W);
    if (!with_o) return;
    constexpr uint32_t idesc = idesc_bf16(64, 64, false, true);
#pragma unroll
    for (int s = 0; s < 4; ++s)
        mma_bf16(tmem + TC_P2, kdesc(sb + L::AQ + s * 32), mndesc(sb + L::O4 + s * 2048, 8192), idesc, s > 0);
}

// Product group 2b: P = Kd^T T' (M = 128, N = 64) from the three leading terms of the
// high/low split, hi.hi + hi.lo + lo.hi.
template <class L>
__device__ __forceinline__ void issue_p(uint32_t sb, uint32_t tmem)
{
    constexpr uint32_t idesc = idesc_bf16(128, 64, false, true);
    const uint32_t a[3] = {L::KDH, L::KDH, L::KDL}, b[3] = {L::O4, L::TL, L::O4};
#pragma unroll
    for (int t = 0; t < 3; ++t)
#pragma unroll
        for (int s = 0; s < 4; ++s)
            mma_bf16(tmem + TC_P, kdesc(sb + a[t] + s * 32), mndesc(sb + b[t] + s * 2048, 8192), idesc,
                     (t | s) != 0);
}

// Product group 3: N = Kd^T (-W) (M = 128, N = 128) and, when outputs are wanted, Q' = Qg + Aqk (-W)
// (M = 64, N = 128), accumulated onto Qg, which the compute warps store into its columns.
template <class L>
__device__ __forceinline__ void issue_n_q(uint32_t sb, uint32_t tmem, bool with_o)
{
    constexpr uint32_t id_n = idesc_bf16(128, 128, false, true), id_q = idesc_bf16(64, 128, false, true);
#pragma unroll
    for (int s = 0; s < 4; ++s)
        mma_bf16(tmem + TC_N, kdesc(sb + L::KDH + s * 32), mndesc(sb + L::O1 + s * 2048, 16384), id_n, s > 0);
    if (!with_o) return;
#pragma unroll
    for (int s = 0; s < 4; ++s)
        mma_bf16(tmem + TC_Q, kdesc(sb + L::AQ + s * 32), mndesc(sb + L::O1 + s * 2048, 16384), id_q, 1);
}

// Epilogues into shared-memory images of the record's parts, which one thread
// then bulk-copies to the record.  Warp w reads TMEM lane quarter w % 4 and the
// (w / 4)-th of NT / 128 equal column ranges.
template <int NT>
__device__ __forceinline__ void epi_p2(uint32_t tmem, unsigned char *dst, bool &ok)
{
    constexpr int CW = 64 / (NT / 128), HW = CW / 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, quarter = warp & 3, part = warp >> 2;
    const int r = quarter * 16 + (lane & 15), c0 = part * CW + (lane >> 4) * HW;  // M = 64: 16-lane loads
#pragma unroll
    for (int cb = 0; cb < HW; cb += 16) {
        float v[16];
        tmem_ld16x2_x16<HW>(tmem + TC_P2 + ((uint32_t)(quarter * 32) << 16) + part * CW + cb, v);
        tmem_ld_wait();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) x[u] = v[hh * 8 + u];
            *reinterpret_cast<uint4 *>(dst + km16(r, c0 + cb + hh * 8, 64)) = pack_f16x8(x, ok);
        }
    }
}

template <int NT>
__device__ __forceinline__ void epi_p(uint32_t tmem, unsigned char *dst, bool &ok)
{
    constexpr int CW = 64 / (NT / 128);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, quarter = warp & 3, part = warp >> 2;
    const int i = quarter * 32 + lane;
#pragma unroll
    for (int cb = 0; cb < CW; cb += 16) {
        float v[16];
        tmem_ld16(tmem + TC_P + ((uint32_t)(quarter * 32) << 16) + part * CW + cb, v);
        tmem_ld_wait();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) x[u] = v[hh * 8 + u];
            *reinterpret_cast<uint4 *>(dst + km16(i, part * CW + cb + hh * 8, 128)) = pack_f16x8(x, ok);
        }
    }
}

// N: the compute warps of part p (warps 4p .. 4p + 3) write K panel p (columns 64p ..) to
// dst[p], 128 rows of 128 bytes.
template <int NT>
__device__ __forceinline__ void epi_n(uint32_t tmem, unsigned char *dst0, unsigned char *dst1)
{
    static_assert(NT == 256, "one K panel per part");
    constexpr int CW = 64;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, quarter = warp & 3, part = warp >> 2;
    const int i = quarter * 32 + lane;
    unsigned char *dst = part ? dst1 : dst0;
#pragma unroll
    for (int cb = 0; cb < CW; cb += 16) {
        float v[16];
        tmem_ld16(tmem + TC_N + ((uint32_t)(quarter * 32) << 16) + part * CW + cb, v);
        tmem_ld_wait();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) x[u] = v[hh * 8 + u];
            *reinterpret_cast<uint4 *>(dst + km16(i, cb + hh * 8, 128)) = pack_bf16x8(x);
        }
    }
}

// Qg (rows 64..127 of O1, bf16) into the Q'' accumulator columns, before the products that
// add Aqk (-W) onto it.  M = 64: 16-lane stores, the mapping of epi_q.
template <class L, int NT>
__device__ __forceinline__ void qg_to_tmem(const unsigned char *sm, uint32_t tmem)
{
    constexpr int CW = 128 / (NT / 128), HW = CW / 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, quarter = warp & 3, part = warp >> 2;
    const int r = quarter * 16 + (lane & 15), c0 = part * CW + (lane >> 4) * HW;
#pragma unroll
    for (int cb = 0; cb < HW; cb += 16) {
        float v[16];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const uint4 qraw = *reinterpret_cast<const uint4 *>(sm + L::O1 + km16(64 + r, c0 + cb + hh * 8, 128));
            const uint32_t qw[4] = {qraw.x, qraw.y, qraw.z, qraw.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float2 qf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&qw[u]));
                v[hh * 8 + 2 * u] = qf.x;
                v[hh * 8 + 2 * u + 1] = qf.y;
            }
        }
        tmem_st16x2_x16<HW>(tmem + TC_Q + ((uint32_t)(quarter * 32) << 16) + part * CW + cb, v);
    }
}

// Q' = Qg + Aqk (-W), whole in TMEM.  M = 64: 16-lane loads, as in w_epilogue.
template <int NT>
__device__ __forceinline__ void epi_q(uint32_t tmem, unsigned char *dst)
{
    constexpr int CW = 128 / (NT / 128), HW = CW / 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, quarter = warp & 3, part = warp >> 2;
    const int r = quarter * 16 + (lane & 15), c0 = part * CW + (lane >> 4) * HW;
#pragma unroll
    for (int cb = 0; cb < HW; cb += 16) {
        float v[16];
        tmem_ld16x2_x16<HW>(tmem + TC_Q + ((uint32_t)(quarter * 32) << 16) + part * CW + cb, v);
        tmem_ld_wait();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            float x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) x[u] = v[hh * 8 + u];
            *reinterpret_cast<uint4 *>(dst + km16(r, c0 + cb + hh * 8, 64)) = pack_bf16x8(x);
        }
    }
}

// Waits (acquire, GPU scope) until the counter at p reaches v; false once kWaitNs has
// passed without it.
__device__ __forceinline__ bool wait_count_at_least(const int *p, int v)
{
    if (ld_acquire_gpu(p) >= v) return true;
    const uint64_t ts = globaltimer_ns();
    for (;;) {
        __nanosleep(128);
        if (ld_acquire_gpu(p) >= v) return true;
        if (globaltimer_ns() - ts > kWaitNs) return false;
    }
}

// The chunk work: items it0, it0 + stride, ... of the seg_chunks x H (chunk, head) items
// over the packed chunks g_base .. g_base + seg_chunks - 1, heads fastest.  Run by the
// chunk kernel (chunks last to first) and by the worker CTAs of the streamed kernel
// (STREAM: chunks first to last, each record published by a release store of its flag,
// flags[g * H + h] = 1, once its bulk stores are complete).  Items past the last packed
// chunk (the chunk count is an upper bound) are skipped.  Records are indexed from g_base.
// With STREAM the items are not strided but claimed in order from the counter *claim, the
// next one while the current item is in work (after its first barrier), so the items taken
// are always the earliest not yet taken, whichever CTAs are resident, and finish about in
// the order they were claimed.
// NORM: q and k arrive raw and are L2-normalised here (KDA_FLAG_QK_L2NORM).
// RING (with STREAM): chunk g's record goes to slot g mod ring, once both walkers have
// counted chunk g - ring's record as copied in (cons[(g - ring) * H + h] == 2).
template <bool NORM, bool STREAM, bool RING = false>
__device__ __forceinline__ void chunk_items(const CUtensorMap &tm_q, const CUtensorMap &tm_k,
                                            const CUtensorMap &tm_la, const float *__restrict__ log_alpha,
                                            const float *__restrict__ beta, const int2 *__restrict__ desc, int H,
                                            int g_base, int seg_chunks, unsigned char *__restrict__ records,
                                            uint32_t *status, bool with_o, bool scalar_gate, int it0, int stride,
                                            int *flags, const int *cons, int *claim, int ring)
{
    using L = ChunkLayout;
    constexpr int NT = kChunkCompute;  // the compute threads' mappings are over 256 threads
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bar_tma, bar_mma, bar_p, bar_drain;
    __shared__ uint32_t tmem_holder;
    __shared__ __align__(16) float s_beta[kC];
    __shared__ float s_rn[2 * kC];  // reciprocal k, q row norms (NORM)
    __shared__ int s_claim;         // STREAM: the item claimed next

    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5;
    const bool compute = tid < kChunkCompute, issuer = tid == kChunkIssuer;
    constexpr int kIssueWarp = kChunkIssuer / 32;
    const int items = seg_chunks * H;
    auto next_item = [&](int it, int &h, int &g, int2 &dsc) -> int {
        for (; it < items; it += stride) {
            h = it % H;
            g = STREAM ? g_base + it / H : g_base + seg_chunks - 1 - it / H;
            dsc = desc[g];  // first token and row count of packed chunk g
            if (dsc.y > 0) break;
            if (STREAM) return items;  // claimed in order: no packed chunk follows this one
        }
        return it;
    };
    int h = 0, g = 0;
    int2 dsc = make_int2(0, 0);
    if (STREAM) {
        if (tid == 0) s_claim = atomicAdd(claim, 1);
        __syncthreads();
        it0 = s_claim;
    }
    int it = next_item(it0, h, g, dsc);
    // q and k boxes, and (per-channel gate) the log_alpha box into O1, which is free until
    // the decayed operands are written there
    const uint32_t tma_bytes = 16384 + 16384 + (scalar_gate ? 0u : 32768u);
    if (issuer) {
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        mbar_init(&bar_p, 1);
        mbar_init(&bar_drain, 1);
        fence_mbar_init();
        if (it < items) {
            mbar_arrive_expect_tx(&bar_tma, tma_bytes);
            if (!scalar_gate) tma_load_3d(sm + L::O1, &tm_la, &bar_tma, 0, h, dsc.x);
            tma_load_3d(sm + L::IN_Q, &tm_q, &bar_tma, 0, h, dsc.x);
            tma_load_3d(sm + L::IN_K, &tm_k, &bar_tma, 0, h, dsc.x);
        }
    }
    if (warp == kIssueWarp) {
        tmem_alloc(&tmem_holder, kChunkTmem);
        tmem_relinquish();
    }
    __syncthreads();  // barriers initialised, TMEM allocated
    tc_fence_after_sync();
    const uint32_t tmem = tmem_holder;
    float *s_tot = reinterpret_cast<float *>(sm + L::AQ);
    bool timed_out = false, decay_bad = false, range_ok = true, stores_pending = false;
    int pub = -1;    // STREAM: the flag of the record whose last stores are in flight (issuer)
    uint32_t n = 0;  // items done by this CTA: the barriers' phase parities follow it
    for (; it < items; ++n) {
        // the previous item's N and Q' stores must have read their staging, which the prefix
        // (s_tot over Aqk) and the decayed operands (Ki over Kd^T low) write next
        if (n > 0) {
            if (issuer) bulk_wait_read();
            __syncthreads();
        }
        if (STREAM && issuer && pub >= 0) {  // the previous record, complete in global memory once
            bulk_wait_all();                   // its stores are: publish it (the compute warps go on)
            fence_proxy_async_global();
            st_release_gpu(flags + pub, 1);
            pub = -1;
        }
        const int64_t c0 = dsc.x;
        const int len = dsc.y;
        // RING: the ring slot of chunk g (otherwise every chunk has its own)
        unsigned char *rec = records + ((size_t)(RING ? g % ring : g - g_base) * H + h) * kRecBytes;
        // the next item, so that its descriptor load overlaps this item's work
        int hn = 0, gn = 0;
        int2 dn = make_int2(0, 0);
        int itn = STREAM ? items : next_item(it + stride, hn, gn, dn);
        const uint32_t pm = (3u * n) & 1u;  // bar_mma completes three times per item
        if (tid < kC) s_beta[tid] = tid < len ? beta[(size_t)(c0 + tid) * H + h] : 0.f;
        float2 gl[4096 / NT];
        float gmin = 0.f, gmax = 0.f;
        // scalar gate (log_alpha [T, H], one decay per token-head): the prefix reads its 64
        // values straight from global memory while the boxes fly
        if (compute && scalar_gate)
            prefix_scan<NT>(log_alpha + (size_t)c0 * H + h, H, len, s_tot, gl, gmin, gmax, true);
        // RING: both walkers of the slot's previous record (chunk g - ring) have copied it in
        // before anything of this one (its gamma first) is written there; checked while the
        // boxes are on their way
        bool ok = !(RING && tid == 0 && g >= ring) || wait_count_at_least(cons + (size_t)(g - ring) * H + h, 2);
        ok = ok && (!compute || mbar_wait_ns(&bar_tma, n & 1u, kWaitNs));
        if (compute && !scalar_gate && ok)  // the per-channel prefix from the log_alpha box
            prefix_scan<NT>(reinterpret_cast<const float *>(sm + L::O1), kD, len, s_tot, gl, gmin, gmax);
        // every thread is past its reads of the log_alpha box and s_tot is complete
        if (__syncthreads_or(!ok)) { timed_out = true; break; }
        if (STREAM && tid == 0) s_claim = atomicAdd(claim, 1);  // the next item
        if (NORM) {
            if (compute) qk_row_inv_norms<NT>(sm + L::IN_K, sm + L::IN_Q, s_rn);
            __syncthreads();
        }
        float2 ot[2];
        if (compute)
            decay_bad |= decayed_operands<L, NT, false, NORM>(sm, len, s_tot, nullptr,
                                                        reinterpret_cast<float *>(rec + R_GM), gl, gmin, gmax, ot,
                                                        s_rn);
        fence_proxy_async_smem();
        __syncthreads();
        if (STREAM) itn = next_item(s_claim, hn, gn, dn);  // its descriptor, for its boxes at the end
        if (issuer) {
            tc_fence_after_sync();
            issue_g1<L>(sb, tmem);
            mma_commit(&bar_mma);
        }
        // From here the compute warps wait for their products themselves; whether any wait
        // gave up is agreed on at the next block-wide barrier, so the issuing warp never
        // holds them up while it issues.
        bool late = false;
        if (compute) {
            late = !mbar_wait_ns(&bar_mma, pm, kWaitNs);
            tc_fence_after_sync();
            if (!late) kk_epilogue<L, NT>(sm, tmem, s_beta, sm + L::AQ);
            tc_fence_before_sync();
            // A complete for the solve; the compute warps enter it all or none
            late = bar_sync_or(1, NT, late);
            if (!late) solve_ut_doubling<L, NT>(sm, s_beta);  // T' high / low images straight from the last level
        }
        fence_proxy_async_smem();
        if (__syncthreads_or(late)) { timed_out = true; break; }
        if (issuer) {
            tc_fence_after_sync();
            issue_w_p2<L>(sb, tmem, with_o);
            mma_commit(&bar_mma);
        }
        if (compute) build_kd<L, NT, NORM>(sm, len, gl, ot[0], ot[1], s_rn);  // over the solve scratch, overlapping W and P2
        fence_proxy_async_smem();
        __syncthreads();
        if (issuer) {
            tc_fence_after_sync();
            issue_p<L>(sb, tmem);
            mma_commit(&bar_p);
        }
        if (compute) {  // the issuing warp is still issuing P meanwhile
            late = !mbar_wait_ns(&bar_mma, pm ^ 1u, kWaitNs);
            tc_fence_after_sync();
            if (!late) w_epilogue<L, NT>(sm, tmem + TC_W);  // -W over Kg in O1
            late = late || !mbar_wait_ns(&bar_p, n & 1u, kWaitNs);
            tc_fence_after_sync();
            if (!late) {
                epi_p<NT>(tmem, sm + L::ST_P, range_ok);    // the k box is dead
                if (with_o) epi_p2<NT>(tmem, sm + L::ST_P2, range_ok);  // T' (high) is dead: every product reading it is done
            }
            if (with_o) {  // Qg into the Q'' columns, once every compute warp has read P and P2 from them
                tc_fence_before_sync();
                late = bar_sync_or(1, NT, late);
                tc_fence_after_sync();
                if (!late) {
                    qg_to_tmem<L, NT>(sm, tmem);
                    tmem_st_wait();
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before_sync();
        if (__syncthreads_or(late)) { timed_out = true; break; }
        if (issuer) {
            // the P and P2 images go out first, so their reads overlap the N, Q'' issue
            bulk_store(rec + R_P, sm + L::ST_P, 16384);
            if (with_o) bulk_store(rec + R_P2, sm + L::ST_P2, 8192);
            bulk_commit();
            stores_pending = true;
            tc_fence_after_sync();
            issue_n_q<L>(sb, tmem, with_o);
            mma_commit(&bar_mma);
        }
        ok = mbar_wait_ns(&bar_mma, pm, kWaitNs);
        if (issuer) bulk_wait_read();  // the P and P2 images: the next boxes and the N staging go over them
        if (__syncthreads_or(!ok)) { timed_out = true; break; }
        tc_fence_after_sync();
        if (issuer && itn < items) {
            // the next item's boxes: every byte they land on is dead now, and N and Q' are
            // staged clear of them, so the copies run while this item's records go out
            mbar_arrive_expect_tx(&bar_tma, tma_bytes);
            if (!scalar_gate) tma_load_3d(sm + L::O1, &tm_la, &bar_tma, 0, hn, dn.x);
            tma_load_3d(sm + L::IN_Q, &tm_q, &bar_tma, 0, hn, dn.x);
            tma_load_3d(sm + L::IN_K, &tm_k, &bar_tma, 0, hn, dn.x);
        }
        if (compute) epi_n<NT>(tmem, sm + L::ST_A, sm + L::ST_B);
        fence_proxy_async_smem();
        if (with_o) {  // then Q' over N's first panel, once its store has read it
            __syncthreads();
            if (issuer) {
                bulk_store(rec + R_N, sm + L::ST_A, 16384u);
                bulk_store(rec + R_N + R_NQ_PANEL, sm + L::ST_B, 16384u);
                bulk_commit();
                bulk_wait_read();
            }
            __syncthreads();
            if (compute) epi_q<NT>(tmem, sm + L::ST_A);
            fence_proxy_async_smem();
        }
        tc_fence_before_sync();  // this item's TMEM reads precede the next item's products
        __syncthreads();
        if (issuer) {
            if (with_o) {  // Q' staged as its two K panels back to back
                bulk_store(rec + R_Q, sm + L::ST_A, 8192u);
                bulk_store(rec + R_Q + R_NQ_PANEL, sm + L::ST_A + 8192, 8192u);
            } else {
                bulk_store(rec + R_N, sm + L::ST_A, 16384u);
                bulk_store(rec + R_N + R_NQ_PANEL, sm + L::ST_B, 16384u);
            }
            bulk_commit();
            if (STREAM) pub = g * H + h;  // published once its stores are complete (next item's start)
        }
        it = itn;
        h = hn;
        g = gn;
        dsc = dn;
    }
    if (STREAM && issuer && pub >= 0) {  // the last record: its stores were all issued
        bulk_wait_all();
        fence_proxy_async_global();
        st_release_gpu(flags + pub, 1);
    }
    if (timed_out) {
        if (issuer) {
            atomicOr(status, DEV_ERR_TIMEOUT);
            mma_commit(&bar_drain);  // completes once every MMA issued so far has
        }
        (void)mbar_wait_ns(&bar_drain, 0, kWaitNs);
        // the item that gave up may still have its boxes in flight
        (void)mbar_wait_ns(&bar_tma, n & 1u, kWaitNs);
    }
    // the record stores must have read their shared-memory sources before the CTA exits
    // and its shared memory is reused; their global writes complete before the kernel does
    if (issuer && stores_pending) bulk_wait_read();
    if (decay_bad) atomicOr(status, DEV_ERR_DECAY);
    if (!range_ok) atomicOr(status, DEV_ERR_RANGE);
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kIssueWarp) tmem_dealloc(tmem, kChunkTmem);
}

template <bool NORM>
__global__ void __launch_bounds__(kChunkThreads, 2)
prefill_chunk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_la, const float *__restrict__ log_alpha,
                     const float *__restrict__ beta,
                     const int2 *__restrict__ desc, int H, int g_base, int seg_chunks,
                     unsigned char *__restrict__ records, uint32_t *status, bool with_o, bool scalar_gate)
{
    // launched with programmatic stream serialization behind the schedule kernel:
    // nothing that kernel writes (cc, the status word) is touched before pdl_wait.  The
    // state kernel may be scheduled once every CTA is past this point, so it can read the
    // schedule (complete by then) before it waits for this kernel's records.
    pdl_wait();
    pdl_launch_dependents();
    // persistent: this CTA takes items blockIdx.x, blockIdx.x + gridDim.x, ...
    chunk_items<NORM, false>(tm_q, tm_k, tm_la, log_alpha, beta, desc, H, g_base, seg_chunks, records, status,
                             with_o, scalar_gate, (int)blockIdx.x, (int)gridDim.x, nullptr, nullptr, nullptr, 0);
}

// ============================================================== state kernel
// Warps 0-15 hold the state; warp 16 issues the chain MMAs; warp 17 copies and
// converts; warp 18 issues the output MMAs.
constexpr int kStateWarps = 16, kChainWarp = 16, kCopyWarp = 17, kOutWarp = 18;
constexpr int kStateThreads = 19 * 32;
constexpr int kL2Ahead = 3;  // records brought into L2 this many chunks ahead

// A state-warp thread's kSCols columns of state row i, as bf16, into the S operand image.
template <class Sh>
__device__ __forceinline__ void store_s_operand(unsigned char *img, int i, int jp, const float (&S)[Sh::kSCols])
{
#pragma unroll
    for (int q = 0; q < Sh::kSCols / 8; ++q) {
        float x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = S[8 * q + u];
        *reinterpret_cast<uint4 *>(img + Sh::mn(i, jp + 8 * q)) = pack_bf16x8(x);
    }
}

// The chain group of one chunk: P V (fp16) + N S_c (bf16) into the M = 128 accumulator.
// dr, dv, ds: descriptors of the record, the V^T image and the S image in use.
template <class Sh>
__device__ __forceinline__ void issue_chain(uint32_t acc, uint64_t dr, uint64_t dv, uint64_t ds)
{
#pragma unroll
    for (int s = 0; s < 4; ++s)  // P V (fp16)
        mma_bf16(acc, dr + ((R_P + s * 32) >> 4), dv + ((s * 32) >> 4), Sh::IDESC_PV, s > 0);
#pragma unroll
    for (int s = 0; s < 8; ++s) {  // + N S_c (bf16)
        const uint32_t off = (s >> 2) * R_NQ_PANEL + (s & 3) * 32, offs = s * Sh::SK;
        mma_bf16(acc, dr + ((R_N + off) >> 4), ds + (offs >> 4), Sh::IDESC_NS, 1);
    }
}

// The output group of one chunk: P2 V (fp16) + Q' S_c (bf16) into an M = 64 accumulator.
template <class Sh>
__device__ __forceinline__ void issue_out(uint32_t acc, uint64_t dr, uint64_t dv, uint64_t ds)
{
#pragma unroll
    for (int s = 0; s < 4; ++s)  // P2 V (fp16)
        mma_bf16(acc, dr + ((R_P2 + s * 32) >> 4), dv + ((s * 32) >> 4), Sh::IDESC_P2V, s > 0);
#pragma unroll
    for (int s = 0; s < 8; ++s) {  // + Q' S_c (bf16)
        const uint32_t off = (s >> 2) * R_NQ_PANEL + (s & 3) * 32, offs = s * Sh::SK;
        mma_bf16(acc, dr + ((R_Q + off) >> 4), ds + (offs >> 4), Sh::IDESC_QS, 1);
    }
}

// The serial pass over the chunks of one (sequence, head, SV-column value slice),
// as four roles that meet only at mbarriers (no block-wide barrier per chunk):
//   bar_ready[c&1]  S_c and V_c (both written by the 16 state warps) are in shared memory
//   bar_rec[c&1]    record c has arrived
//   bar_s           the chain of the latest chunk is done
//   bar_o[c&1]      the output group of chunk c is done
// Chunk c:
//   warp 16 (one lane)   waits ready(c), record c; issues P V + N S_c; commits bar_s
//   warp 18 (one lane)   waits ready(c), record c; issues P2 V + Q' S_c; commits bar_o
//   warps 0-15           write the outputs of chunk c - 1 (waiting bar_o), convert the
//                        v slice of chunk c + 1 over V_{c-1} while the chain runs, wait
//                        bar_s, S_{c+1} = gamma . S_c + (P V + N S_c), arrive on ready(c + 1)
//   warp 17              once ready(c) and bar_o(c - 1) hold, copies record c + 1 over
//                        record c - 1, prefetches a later record into L2 and refills the
//                        v slot of chunk c (converted by then) with chunk c + kVRing
// Every producer runs at most one chunk ahead of the consumer of the buffer it
// refills, and each ready / output barrier alternates with the chunk parity, so no
// barrier is ever waited on more than one phase behind.  Each issuing lane has a
// warp of its own: MMA issue slows down badly when the rest of its warp is busy.
//
// CTAs with blockIdx.z >= z_ident run the transition pass of the sequence-split prefill:
// the state starts as the identity, every value row reads as zero (tm_v_zero maps one
// zero row, so every box past it is filled with zeros), and the final state goes to
// final_ident.  Their result is the linear map of the sequence's chunks.  A CTA whose
// sequence has no final state to store and no outputs to write returns at once.
template <int SV>
__global__ void __launch_bounds__(kStateThreads, 1)
prefill_state_kernel(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_v_zero,
                     const int32_t *__restrict__ cu, int64_t total, int H, const int32_t *__restrict__ cc,
                     const unsigned char *__restrict__ records, const float *init_state,
                     __nv_bfloat16 *__restrict__ o, float *final_state, uint32_t *status,
                     const int32_t *__restrict__ order, StateSlots slots, int z_ident, float *final_ident,
                     StateSegment seg)
{
    using Sh = StateShape<SV>;
    using L = Sh;
    constexpr int kVRing = Sh::kVRing, kSCols = Sh::kSCols;
    constexpr uint32_t kVBytes = Sh::kVBytes, kSBytes = Sh::kSBytes, TM_5 = Sh::TM_5, TM_O = Sh::TM_O;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bar_rec[2], bar_v[kVRing], bar_s, bar_o[2], bar_ready[2], bar_drain;
    __shared__ uint32_t tmem_holder;

    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool state_warp = warp < kStateWarps;
    const int quarter = warp & 3, part = (warp >> 2) & 3;
    // launched with programmatic stream serialization behind the chunk kernel, which signals
    // only once the schedule kernel is complete: the schedule (order, cc, descriptors), the
    // initial states and the value rows are read at once, the records only after pdl_wait
    // (the chunk kernel's completion), so this prologue overlaps that kernel's last CTAs
    const bool ident = (int)blockIdx.z >= z_ident;
    const int j0 = blockIdx.x * SV, h = blockIdx.y, n = order[ident ? blockIdx.z - z_ident : blockIdx.z];
    int64_t t0, t1;
    seq_range(cu, n, total, t0, t1);
    int nchunks = (int)((t1 - t0 + kC - 1) / kC);
    // the sequence's packed chunks inside this launch's segment [seg.g_lo, seg.g_hi)
    const int cn0 = cc[n], ca = cn0 > seg.g_lo ? cn0 : seg.g_lo;
    const int cb = cn0 + nchunks < seg.g_hi ? cn0 + nchunks : seg.g_hi;
    bool from_carry = false, to_carry = false;
    if (nchunks == 0) {
        if (seg.g_lo != 0) return;  // an empty sequence is settled by the first segment
    } else {
        if (cb <= ca) return;       // none of its chunks in this segment
        from_carry = cn0 < seg.g_lo;
        to_carry = cn0 + nchunks > seg.g_hi;
        const int64_t s0 = t0;
        t0 = s0 + (int64_t)(ca - cn0) * kC;
        if (to_carry) t1 = s0 + (int64_t)(cb - cn0) * kC;
        nchunks = cb - ca;
    }
    int64_t si, sf;
    if (!state_entries(slots, n, !ident && init_state != nullptr, si, sf) && tid == 0)
        atomicOr(status, DEV_ERR_SLOT);
    if (ident) o = nullptr;
    const bool store_end = to_carry || sf >= 0;
    if (!store_end && (o == nullptr || nchunks == 0)) return;  // nothing to store or write
    float *const fpool = ident ? final_ident : final_state;
    const CUtensorMap *const tmv = ident ? &tm_v_zero : &tm_v;
    const unsigned char *rec0 = records + ((size_t)(ca - seg.g_lo) * H + h) * kRecBytes;
    const size_t rec_stride = (size_t)H * kRecBytes;

    // copies: issued by lane 0 of the copy warp only, which alone keeps these counts
    int rec_issued = 0, v_issued = 0;
    auto load_record = [&](int k) {
        mbar_arrive_expect_tx(&bar_rec[k & 1], kRecBytes);
        bulk_load(sm + (k & 1) * L::STAGE, rec0 + (size_t)k * rec_stride, kRecBytes, &bar_rec[k & 1]);
        rec_issued = k + 1;
    };
    auto load_v = [&](int k) {
        mbar_arrive_expect_tx(&bar_v[k % kVRing], kVBytes);
        tma_load_3d(sm + L::VBOX + (k % kVRing) * kVBytes, tmv, &bar_v[k % kVRing], j0, h,
                    (int)(t0 + (int64_t)k * kC));
        v_issued = k + 1;
    };
    const bool copier = warp == kCopyWarp && lane == 0;
    if (tid == 0) {
        mbar_init(&bar_rec[0], 1);
        mbar_init(&bar_rec[1], 1);
        for (int k = 0; k < kVRing; ++k) mbar_init(&bar_v[k], 1);
        mbar_init(&bar_s, 1);
        mbar_init(&bar_o[0], 1);
        mbar_init(&bar_o[1], 1);
        mbar_init(&bar_ready[0], kStateWarps);
        mbar_init(&bar_ready[1], kStateWarps);
        mbar_init(&bar_drain, 2);  // both issuing lanes commit to it on a timeout
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_holder, Sh::TMEM);
        tmem_relinquish();
    }
    // state row i, columns j0 + jp .. jp + kSCols - 1 in registers; S (bf16) operands in O7
    const int i_row = quarter * 32 + lane, jp = part * kSCols;
    float S[kSCols];
    const size_t st_off = ((size_t)h * kD + i_row) * kD + j0 + jp, st_entry = (size_t)H * kD * kD;
    if (state_warp) {
        if (ident) {
#pragma unroll
            for (int j = 0; j < kSCols; ++j) S[j] = i_row == j0 + jp + j ? 1.f : 0.f;
        } else if (from_carry || si >= 0) {
            const float *src = from_carry ? seg.carry_in + st_off : init_state + si * st_entry + st_off;
#pragma unroll
            for (int q = 0; q < kSCols / 4; ++q) {
                const float4 x = *reinterpret_cast<const float4 *>(src + 4 * q);
                S[4 * q] = x.x; S[4 * q + 1] = x.y; S[4 * q + 2] = x.z; S[4 * q + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < kSCols; ++j) S[j] = 0.f;
        }
        store_s_operand<Sh>(sm + L::O7, i_row, jp, S);
    }
    fence_proxy_async_smem();
    __syncthreads();  // barriers initialised, S_0 written
    tc_fence_after_sync();
    const uint32_t tmem = tmem_holder;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int r64 = quarter * 16 + (lane & 15);  // row held by this lane in an M = 64 accumulator
    bool range_ok = true;
    // operand descriptors of buffer 0; buffer 1 is a fixed byte distance further
    const uint64_t d_rec0 = kdesc(sb), d_v0 = kdesc(sb + L::VIMG), d_s0 = Sh::sdesc_s(sb + L::O7);
    // ready(c) for c >= 1 (chunk 0's operands are known ready from the first barrier)
    auto wait_ready = [&](int c) -> bool {
        return c < 1 || mbar_wait_ns(&bar_ready[c & 1], (uint32_t)(((c - 1) >> 1) & 1), kWaitNs);
    };
    auto wait_record = [&](int c) -> bool {
        return mbar_wait_ns(&bar_rec[c & 1], (uint32_t)((c >> 1) & 1), kWaitNs);
    };

    // o rows of chunk cp (M = 64 accumulator TM_O + SV*(cp&1)), once its MMAs finished
    // (with no outputs wanted the barrier still marks the chunk's operands as released)
    auto write_o = [&](int cp) -> bool {
        if (!mbar_wait_ns(&bar_o[cp & 1], (uint32_t)((cp >> 1) & 1), kWaitNs)) return false;
        if (!o) return true;
        tc_fence_after_sync();
        // the warp's kSCols columns, half to each half-warp (16-lane load of the M = 64 rows)
        const int64_t cs = t0 + (int64_t)cp * kC;
        __nv_bfloat16 *dst = o + ((size_t)(cs + r64) * H + h) * kD + j0 + jp + (kSCols / 2) * (lane >> 4);
        if constexpr (SV == 64) {
            float v[8];
            tmem_ld16x2_x8<8>(tmem + TM_O + SV * (cp & 1) + lane_off + jp, v);
            tmem_ld_wait();
            if (cs + r64 < t1) *reinterpret_cast<uint4 *>(dst) = pack_bf16x8(v);
        } else {
            float v[4];
            tmem_ld16x2_x4<4>(tmem + TM_O + SV * (cp & 1) + lane_off + jp, v);
            tmem_ld_wait();
            if (cs + r64 < t1) *reinterpret_cast<uint2 *>(dst) = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
        }
        return true;
    };
    // state warps: the v slice of chunk k -> V^T fp16 K-major in VIMG[k & 1]; one
    // group of RV rows of one column per thread
    auto convert_v = [&](int k) -> bool {
        constexpr int RV = SV / 8;  // 512 state threads cover 64 rows x SV columns
        if (!mbar_wait_ns(&bar_v[k % kVRing], (uint32_t)((k / kVRing) & 1), kWaitNs)) return false;
        const int64_t ck = t0 + (int64_t)k * kC;
        const int lenk = (t1 - ck) < kC ? (int)(t1 - ck) : kC;
        const unsigned char *box = sm + L::VBOX + (k % kVRing) * kVBytes;
        const int j = tid % SV, s0 = (tid / SV) * RV;
        float x[RV];
#pragma unroll
        for (int u = 0; u < RV; ++u) {
            x[u] = (s0 + u) < lenk ? bf16_at(box + ((s0 + u) * SV + j) * 2) : 0.f;
            range_ok &= fabsf(x[u]) <= 65504.f;
        }
        unsigned char *img = sm + L::VIMG + (k & 1) * kVBytes + km16(j, s0, SV);
        if constexpr (RV == 8) {
            *reinterpret_cast<uint4 *>(img) = pack_f16x8_plain(x);
        } else {
            __half2 a = __floats2half2_rn(x[0], x[1]), b = __floats2half2_rn(x[2], x[3]);
            *reinterpret_cast<uint2 *>(img) = make_uint2(*reinterpret_cast<uint32_t *>(&a), *reinterpret_cast<uint32_t *>(&b));
        }
        return true;
    };

    bool ok = true;
    if (copier) {
        for (int k = 0; k < kVRing && k < nchunks; ++k) load_v(k);
        prefetch_tmap(tmv);
    }
    pdl_wait();  // the chunk kernel has completed: its records are visible
    if (copier) {
        for (int k = 0; k < 2 && k < nchunks; ++k) load_record(k);
        for (int k = 2; k < kL2Ahead && k < nchunks; ++k) bulk_prefetch_l2(rec0 + (size_t)k * rec_stride, kRecBytes);
    }
    if (state_warp && nchunks > 0) {
        ok = convert_v(0);
        fence_proxy_async_smem();
    }
    bool timed_out = __syncthreads_or(!ok);  // S_0 and V_0 are in place for every role
    int c = 0;
    if (!timed_out) {
        if (state_warp) {
            for (; ok && c < nchunks; ++c) {
                const int st = c & 1;
                if (c >= 1) ok = write_o(c - 1);  // also frees O7 and VIMG of chunk c - 1
                if (ok && c + 1 < nchunks) {     // V_{c+1} while the chain of chunk c runs
                    ok = convert_v(c + 1);
                    fence_proxy_async_smem();
                }
                // gamma comes from the record (its copy long complete): read before the chain's wait
                if (ok) ok = wait_record(c);
                const float gc = ok ? reinterpret_cast<const float *>(sm + st * L::STAGE + R_GM)[i_row] : 0.f;
                if (ok) ok = mbar_wait_ns(&bar_s, (uint32_t)(c & 1), kWaitNs);
                if (ok) {  // S <- gamma . S + (P V + N S); its bf16 operand image for the next chunk
                    tc_fence_after_sync();
                    float v[kSCols];
                    if constexpr (kSCols == 16)
                        tmem_ld16(tmem + TM_5 + lane_off + jp, v);
                    else
                        tmem_ld8(tmem + TM_5 + lane_off + jp, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < kSCols; ++j) S[j] = fmaf(gc, S[j], v[j]);
                    store_s_operand<Sh>(sm + L::O7 + (st ^ 1) * kSBytes, i_row, jp, S);
                    fence_proxy_async_smem();
                }
                tc_fence_before_sync();  // this warp's TMEM reads precede the arrival
                ok = __all_sync(0xffffffffu, ok);
                if (ok && lane == 0 && c + 1 < nchunks) mbar_arrive(&bar_ready[(c + 1) & 1]);  // S, V of c + 1
            }
            if (ok && nchunks > 0) ok = write_o(nchunks - 1);
        } else if (warp == kChainWarp || warp == kOutWarp) {
            const bool chain = warp == kChainWarp;
            for (; ok && c < nchunks; ++c) {
                const int st = c & 1;
                if (lane == 0) {
                    ok = wait_ready(c) && wait_record(c);
                    if (ok) {
                        tc_fence_after_sync();
                        // descriptors: base of each operand plus the constant byte offset >> 4
                        const uint64_t dr = d_rec0 + st * (L::STAGE >> 4), dv = d_v0 + st * (kVBytes >> 4),
                                       ds = d_s0 + st * (kSBytes >> 4);
                        if (chain) {
                            issue_chain<Sh>(tmem + TM_5, dr, dv, ds);
                            mma_commit(&bar_s);
                        } else {
                            if (o) issue_out<Sh>(tmem + TM_O + SV * st, dr, dv, ds);  // none when no outputs are wanted
                            mma_commit(&bar_o[st]);  // also marks chunk c's operands as released
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
            }
        } else if (warp == kCopyWarp) {  // record c + 1, one chunk ahead of the state warps
            for (; ok && c < nchunks; ++c) {
                if (c >= 1) {  // the record stage of chunk c - 1 is free; V_c is converted
                    ok = wait_ready(c) &&
                         mbar_wait_ns(&bar_o[(c - 1) & 1], (uint32_t)(((c - 1) >> 1) & 1), kWaitNs);
                    if (copier && ok && c + 1 < nchunks) load_record(c + 1);
                }
                if (copier && ok && c + kL2Ahead < nchunks)
                    bulk_prefetch_l2(rec0 + (size_t)(c + kL2Ahead) * rec_stride, kRecBytes);
                if (copier && ok && c + kVRing < nchunks) load_v(c + kVRing);  // V_c's slot
                ok = __shfl_sync(0xffffffffu, ok, 0);
            }
        }
    }
    timed_out = __syncthreads_or(timed_out || !ok);  // every role has finished or given up
    if (timed_out) {
        if (tid == 0) atomicOr(status, DEV_ERR_TIMEOUT);
        // completes once every MMA of both issuing lanes has
        if ((warp == kChainWarp || warp == kOutWarp) && lane == 0) mma_commit(&bar_drain);
        (void)mbar_wait_ns(&bar_drain, 0, kWaitNs);
        // our own copies still in flight (the copying thread knows how many)
        for (int k = rec_issued > 2 ? rec_issued - 2 : 0; k < rec_issued; ++k)
            (void)mbar_wait_ns(&bar_rec[k & 1], (uint32_t)((k >> 1) & 1), kWaitNs);
        for (int k = v_issued > kVRing ? v_issued - kVRing : 0; k < v_issued; ++k)
            (void)mbar_wait_ns(&bar_v[k % kVRing], (uint32_t)((k / kVRing) & 1), kWaitNs);
    } else if (state_warp && store_end) {
        float *dst = to_carry ? seg.carry_out + st_off : fpool + sf * st_entry + st_off;
#pragma unroll
        for (int q = 0; q < kSCols / 4; ++q)
            *reinterpret_cast<float4 *>(dst + 4 * q) = make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
    }
    if (!range_ok) atomicOr(status, DEV_ERR_RANGE);
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, Sh::TMEM);
}

// ============================================================== streamed prefill
// One launch of two CTAs per SM.  CTAs [0, n_walk) each walk the state of half a (sequence,
// head) unit through its chunks; the others run the chunk work (chunk_items, chunks first
// to last, items claimed in order from a counter) and publish every record with a release
// store of its flag.  A walker copies a record only after an acquire load has seen its
// flag, so the serial pass follows the chunk work closely, its records come back from L2,
// and the serial chain overlaps the chunk work instead of following it.
//
// With a workspace that holds every record, progress does not depend on which CTAs are
// resident: only walkers wait, and only for records; a worker never waits for another CTA,
// and the items are claimed in order by workers that are running, so the earliest
// unpublished record is always in work.  The walkers (at most kMaxWalkers) are fewer than
// the CTAs that one wave holds, so workers always run beside them.
//
// A bounded workspace holds the records of `ring` packed chunks: chunk g's record goes to
// slot g mod ring, and its worker writes there only once both walkers of chunk g - ring
// (the slot's previous record) have copied that one in, which each signals by adding one to
// the record's copy count.  Every such wait is for an earlier chunk than the waiter's, whose
// item was claimed earlier, so with the grid resident there is no cycle; the chunk work
// then leads the walk by at most `ring` chunks, and the records stay in L2 (T = 65536,
// H = 32, 16 chunks: 1.16 times the path's algorithmic DRAM bytes, against 2.46 with every
// record).  The ring is the RING instantiation; with every record held the kernel is
// instantiated without it and no worker waits.  The ring is not the faster form then:
// workers held to the walk's pace share the SMs with it to the end, where unheld they
// finish early and leave the walkers their SMs (2.16 ms with 16 chunks, against 1.97).
//
// Every wait is bounded (a flag or count that does not come up within the limit is
// recorded as KDA_ERR_TIMEOUT and the CTA unwinds).
//
// Two walkers share a head, each with 64 of its value columns (the columns of S evolve
// independently), and each forms the transposed products, so that its part fits in a CTA
// of the chunk work's size.  With S^T (value column j x key row i) as the A operand, the
// state update and the outputs share their A operands and run as one product group:
//   [S_{c+1}^T | o_c^T] = [gamma_c . S_c^T | 0] + V_c^T [P_c^T | P2_c^T] + S_c^T [N_c^T | Q'_c^T]
// (M = 64 rows j; N = 128 key rows i for the state and 64 tokens t for the outputs, 192 in
// all).  The record's P, P2, N and Q' images (rows over their first index, K-major over
// the second) are the B operands: P and P2, and each K panel of N and Q', sit back to back
// in the record as 192-row operands, so the walker copies them in two pieces as they stand
// (fewer copies shorten the wait for them: every extra copy per chunk cost about 30 ns of
// the walk).  TMEM holds the state itself: the
// accumulator's first 128 columns (fp32, lane j, column i), into which the state warps store
// gamma_c . S_c (and zeros into the output columns) before the products accumulate onto
// them; and S_c^T in bf16 as the A operand of the N, Q' products.  V_c^T (fp16, K-major) is
// in shared memory.
struct WalkLayout {
    // the record in use: [N panel 0 | Q' panel 0 | N panel 1 | Q' panel 1 | P | P2]
    static constexpr uint32_t NQ = 0, NQ_PANEL = 24576;  // 192 rows x 128 bytes per K panel
    static constexpr uint32_t PP = 2 * NQ_PANEL;         // P (128 rows) then P2 (64 rows)
    static constexpr uint32_t VT = PP + 24576;           // V^T fp16, 64 rows (j) x K 64 (t)
    static constexpr uint32_t VBOX = VT + kC * 64 * 2;   // raw v box [64 tokens][64] bf16
    static constexpr uint32_t GAM = VBOX + kC * 64 * 2;  // gamma of two chunks, 2 x 128 fp32
    static constexpr uint32_t USED = GAM + 2 * kD * 4;
};
static_assert(WalkLayout::NQ_PANEL % 1024 == 0 && WalkLayout::PP % 1024 == 0 && WalkLayout::VT % 1024 == 0 &&
                  WalkLayout::VBOX % 128 == 0,
              "walker layout alignment");
static_assert(R_P2 == R_P + 16384, "P2 follows P in the record");
static_assert(WalkLayout::NQ_PANEL == R_NQ_PANEL && R_Q == R_N + 16384 && R_P == R_N + 2 * R_NQ_PANEL,
              "the walker's N | Q' operand is the record's, copied whole");
constexpr uint32_t kStreamSmem =
    (WalkLayout::USED > ChunkLayout::USED ? WalkLayout::USED : ChunkLayout::USED) + 1024;
// walker TMEM columns: accumulator (state 0-127, outputs 128-191), bf16 S^T.  An M = 64
// operand or accumulator keeps its row r in lane 32 (r / 16) + r % 16 (lanes 0-15 of each
// lane quarter); the walker's warps reach them with the 16-lane load and store shapes.
constexpr uint32_t TW_D = 0, TW_O = 128, TW_A = 192, kWalkTmem = 256;
constexpr int kWalkStateWarps = 8;
constexpr int kWalkCols = 64;    // value columns per walker: two walkers per (sequence, head)
constexpr int kMaxWalkers = 64;  // walker CTAs of the streamed prefill at most (32 units)
// Fewest (sequence, head) units for which the streamed prefill is the faster form, by the
// chunks per unit.  The walk takes about 1.9 us per chunk whatever the unit count, and the
// two kernels' time grows with it (the chunk work, before the state pass at about 1 us per
// chunk); the walk's fixed start (the first records) matters less on longer sequences.
// Measured crossovers (one sequence): about 31 units at 64 chunks (T = 4096: 0.153 ms as two
// kernels against 0.158 streamed at 30 units, 0.160 against 0.157 at 32), about 27 at 256
// (T = 16384: 0.486 against 0.506 ms at 24 units, 0.533 against 0.515 at 28), fewer still at
// 1024 (T = 65536, 32 units: 2.24 against 2.0 ms).
inline int min_stream_units(int64_t chunks_per_unit)
{
    return chunks_per_unit <= 96 ? 31 : (chunks_per_unit <= 384 ? 27 : 24);
}
// First chunk whose record a walker prefetches into L2 two chunks ahead.  The walk trails the
// chunk work by a little more each chunk (about 12 %), so early records are read while still
// in L2 and the prefetch only costs a copy on the critical path (T = 4096: 1.7 % slower with
// it); later ones have left L2 by the time they are read (T = 65536: 4 % slower without it).
constexpr int kWalkPrefetchFrom = 128;

// The product group of one chunk: D += V^T [P^T | P2^T] (fp16) + S^T [N^T | Q'^T] (bf16, S^T
// from TMEM), M = 64, N = 192, or N = 128 (state only) without the outputs; in two parts,
// the V^T products first (their operands, P and P2, arrive first).
__device__ __forceinline__ void issue_walk_pv(uint32_t tmem, uint32_t sb, bool with_o)
{
    const uint32_t id_pv = with_o ? idesc_f16(64, 192, false, false) : idesc_f16(64, 128, false, false);
    const uint64_t dvt = kdesc(sb + WalkLayout::VT), dp = kdesc(sb + WalkLayout::PP);
#pragma unroll
    for (int s = 0; s < 4; ++s) mma_bf16(tmem + TW_D, dvt + 2 * s, dp + 2 * s, id_pv, 1);
}
__device__ __forceinline__ void issue_walk_ns(uint32_t tmem, uint32_t sb, bool with_o)
{
    const uint32_t id_ns = with_o ? idesc_bf16(64, 192, false, false) : idesc_bf16(64, 128, false, false);
    const uint64_t dn = kdesc(sb + WalkLayout::NQ);
#pragma unroll
    for (int s = 0; s < 8; ++s)
        mma_tmem_a(tmem + TW_D, tmem + TW_A + 8 * s, dn + (((s >> 2) * WalkLayout::NQ_PANEL + (s & 3) * 32) >> 4),
                   id_ns, 1);
}
__device__ __forceinline__ void issue_walk(uint32_t tmem, uint32_t sb, bool with_o)
{
    issue_walk_pv(tmem, sb, with_o);
    issue_walk_ns(tmem, sb, with_o);
}

// One walker CTA over one (sequence, head, value half).  Warps 0-7 move the state through
// TMEM, write the outputs and convert the v boxes: warp w holds rows r = 16 (w & 3) + l of
// the half (value column j = 64 half + r) in TMEM lane 32 (w & 3) + l, l = lane & 15, and
// key rows 64 (w >> 2) + 32 (lane >> 4) .. + 31.  Lane 0 of warp 8 copies the records and
// the v boxes and issues the product group; lane 0 of warp 0 waits for the records' flags
// and copies the gammas.  Per chunk c:
//   warp 8    waits ready(c) and record c (P and P2, then N and Q'); issues the group
//             (commit w_mma); loads the v box of c + 2 once that of c + 1 is read (w_vfree);
//             copies record c + 1 once w_mma(c) holds (its flag was seen before ready(c)).
//   warps 0-7 read the v box of c + 1 into registers (arrive w_vfree); lane 0 of warp 0
//             waits for record c + 2's flag and, its buffer being free after ready(c), copies
//             its gamma and prefetches the record into L2; all wait w_mma(c); store V^T of
//             c + 1; read S_{c+1} from D, store bf16(S_{c+1}) and gamma_{c+1} . S_{c+1} back;
//             read o_c into registers and zero the output columns; arrive on ready(c + 1);
//             then store o_c while the next group runs.
// Every barrier's producer stays within one phase of its consumers (each refill waits for
// the consumption of what it overwrites), so no wait is ever more than one phase behind.
template <bool RING>
__device__ __forceinline__ void walk_unit(int walker, const CUtensorMap &tm_v, const int32_t *__restrict__ cu,
                                          int64_t total, int H, const int32_t *__restrict__ cc,
                                          const unsigned char *__restrict__ records, const int *flags, int *cons,
                                          int ring, const float *init_state, __nv_bfloat16 *__restrict__ o,
                                          float *final_state, uint32_t *status, const StateSlots &slots)
{
    using L = WalkLayout;
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t w_ready, w_mma, w_rec, w_pp, w_v, w_vfree, w_g[2], w_drain;
    __shared__ uint32_t w_tmem;
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool state_warp = warp < kWalkStateWarps, ctl_warp = warp == kWalkStateWarps;
    const int half = walker & 1, unit = walker >> 1, n = unit / H, h = unit % H;
    int64_t t0, t1;
    seq_range(cu, n, total, t0, t1);
    const int nch = (int)((t1 - t0 + kC - 1) / kC);
    int64_t si, sf;
    if (!state_entries(slots, n, init_state != nullptr, si, sf) && tid == 0 && half == 0)
        atomicOr(status, DEV_ERR_SLOT);
    const int part = (warp >> 2) & 1, hs = lane >> 4;
    const int jrow = kWalkCols * half + 16 * (warp & 3) + (lane & 15);  // this thread's value column
    const int ib = 64 * part + 32 * hs;                                 // its key rows ib .. ib + 31
    const size_t st_entry = (size_t)H * kD * kD, st_head = (size_t)h * kD * kD;
    if (nch == 0) {  // no tokens: the final state is the initial one
        if (state_warp && sf >= 0)
            for (int i = ib; i < ib + 32; ++i)
                final_state[sf * st_entry + st_head + (size_t)i * kD + jrow] =
                    si >= 0 ? init_state[si * st_entry + st_head + (size_t)i * kD + jrow] : 0.f;
        return;
    }
    // record c: chunk cc[n] + c, its ready flag, its copy count and its slot (without RING:
    // every chunk has its own and no count is kept)
    const int g0 = cc[n];  // read once: the waits' memory clobbers would reload it at every use
    const int *flag0 = flags + (size_t)g0 * H + h;
    int *cons0 = cons + (size_t)g0 * H + h;
    const unsigned char *rec_h = records + (size_t)h * kRecBytes;
    const size_t rec_stride = (size_t)H * kRecBytes;
    auto rec_at = [&](int c) {
        const int g = g0 + c;
        return rec_h + (size_t)(RING ? g % ring : g) * rec_stride;
    };
    if (sf < 0 && o == nullptr) {  // nothing to store and no outputs: each slot is free once filled
        if (RING && tid == 0)
            for (int c = 0; c < nch; ++c) {
                if (!wait_count_at_least(flag0 + (size_t)c * H, 1)) {
                    atomicOr(status, DEV_ERR_TIMEOUT);
                    break;
                }
                red_release_add_gpu(cons0 + (size_t)c * H, 1);
            }
        return;
    }
    if (tid == 0) {
        mbar_init(&w_ready, kWalkStateWarps);
        mbar_init(&w_mma, 1);
        mbar_init(&w_rec, 1);
        mbar_init(&w_pp, 1);
        mbar_init(&w_v, 1);
        mbar_init(&w_vfree, kWalkStateWarps);
        mbar_init(&w_g[0], 1);
        mbar_init(&w_g[1], 1);
        mbar_init(&w_drain, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&w_tmem, kWalkTmem);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();  // barriers initialised, TMEM allocated
    tc_fence_after_sync();
    const uint32_t tmem = w_tmem;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;

    // copies: the records and v boxes issued by lane 0 of warp 8, the gammas by lane 0 of
    // warp 0; each keeps its own counts
    int rec_issued = 0, v_issued = 0, g_issued = 0;
    auto wait_flag = [&](int c) -> bool {  // record c is complete in global memory
        const int *f = flag0 + (size_t)c * H;
        if (ld_acquire_gpu(f) == 0) {
            const uint64_t ts = globaltimer_ns();
            for (;;) {
                __nanosleep(128);
                if (ld_acquire_gpu(f) != 0) break;
                if (globaltimer_ns() - ts > kWaitNs) return false;
            }
        }
        fence_proxy_async_global();  // the bulk copies below read what the flag published
        return true;
    };
    auto load_gamma = [&](int c) {
        mbar_arrive_expect_tx(&w_g[c & 1], kD * 4);
        bulk_load(sm + L::GAM + (c & 1) * kD * 4, rec_at(c) + R_GM, kD * 4, &w_g[c & 1]);
        g_issued = c + 1;
    };
    // N, P (and with outputs Q', P2) as the group's operands: P and P2 first (w_pp), then
    // N and Q' (w_rec)
    auto load_record = [&](int c) {
        const unsigned char *r = rec_at(c);
        mbar_arrive_expect_tx(&w_pp, o ? 24576u : 16384u);
        bulk_load(sm + L::PP, r + R_P, o ? 24576u : 16384u, &w_pp);  // P2 follows P in both
        mbar_arrive_expect_tx(&w_rec, o ? 49152u : 32768u);
        if (o) {  // N and Q' as laid out in the record: one copy
            bulk_load(sm + L::NQ, r + R_N, 49152u, &w_rec);
        } else {
            bulk_load(sm + L::NQ, r + R_N, 16384u, &w_rec);
            bulk_load(sm + L::NQ + L::NQ_PANEL, r + R_N + R_NQ_PANEL, 16384u, &w_rec);
        }
        rec_issued = c + 1;
    };
    auto load_v = [&](int c) {  // this half's 64 value columns of the chunk's 64 tokens
        mbar_arrive_expect_tx(&w_v, kC * kWalkCols * 2);
        tma_load_3d(sm + L::VBOX, &tm_v, &w_v, kWalkCols * half, h, (int)(t0 + (int64_t)c * kC));
        v_issued = c + 1;
    };
    bool range_ok = true;
    // State warps (whole warps; every wait result is made uniform over the warp, as the
    // TMEM loads and stores are warp-collective).  The v box is read into registers (vt) as
    // soon as it arrives, the warp then arrives on w_vfree, and the registers go to the V^T
    // image (fp16, K-major rows j, 128-byte swizzle) once the products reading it are done;
    // rows past the unit's last token read as zero.
    const int vj = tid & (kWalkCols - 1), vs0 = (tid >> 6) * 16;  // V^T row vj, tokens vs0 .. + 15
    auto read_v = [&](int c, uint4 (&vt)[2]) -> bool {
        if (!__all_sync(0xffffffffu, mbar_wait_ns(&w_v, (uint32_t)(c & 1), kWaitNs))) return false;
        const int64_t cs = t0 + (int64_t)c * kC;
        const int lenc = (t1 - cs) < kC ? (int)(t1 - cs) : kC;
        const unsigned char *box = sm + L::VBOX;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int s = vs0 + 8 * q + u;
                x[u] = s < lenc ? bf16_at(box + (s * kWalkCols + vj) * 2) : 0.f;
                range_ok &= fabsf(x[u]) <= 65504.f;
            }
            vt[q] = pack_f16x8_plain(x);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&w_vfree);  // this warp is done with the box
        return true;
    };
    auto store_v = [&](const uint4 (&vt)[2]) {
#pragma unroll
        for (int q = 0; q < 2; ++q)
            *reinterpret_cast<uint4 *>(sm + L::VT + km16(vj, vs0 + 8 * q, kWalkCols)) = vt[q];
    };
    // 16 key rows ib + 16 k .. + 15 of this thread's column: bf16(S) into the A operand,
    // gamma . S (fp32) into D (A column c holds key rows 2c, 2c + 1)
    auto put_state = [&](int k, float (&x)[16], const float *gam) {
        uint32_t pk[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) pk[u] = pack_bf16x2(x[2 * u], x[2 * u + 1]);
        tmem_st16x2_x8<16>(tmem + lane_off + TW_A + 32 * part + 8 * k, pk);
        const int i0 = ib + 16 * k;
#pragma unroll
        for (int u = 0; u < 16; u += 4) {
            const float4 g = *reinterpret_cast<const float4 *>(gam + i0 + u);
            x[u] *= g.x;
            x[u + 1] *= g.y;
            x[u + 2] *= g.z;
            x[u + 3] *= g.w;
        }
        tmem_st16x2_x16<32>(tmem + lane_off + TW_D + 64 * part + 16 * k, x);
    };
    auto load_state = [&](int k, float (&x)[16]) {  // the same 16 key rows of D
        tmem_ld16x2_x16<32>(tmem + lane_off + TW_D + 64 * part + 16 * k, x);
        tmem_ld_wait();
    };
    // zeros into this thread's 16 output columns (the group accumulates onto D)
    auto zero_out = [&]() {
        float z[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) z[u] = 0.f;
        tmem_st16x2_x16<16>(tmem + lane_off + TW_O + 32 * part, z);
    };

    bool ok = true;
    if (ctl_warp) {
        if (lane == 0) {
            load_v(0);
            ok = wait_flag(0);
            if (ok) load_record(0);
            if (ok && nch > 1) {  // the box of chunk 1, once chunk 0's is read
                ok = mbar_wait_ns(&w_vfree, 0, kWaitNs);
                if (ok) load_v(1);
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
    } else if (state_warp) {  // S_0: gamma_0 . S_0 into D, bf16(S_0) into the A operand
        if (warp == 0 && lane == 0) {  // lane 0 of warp 0 loads every gamma (its flag seen first)
            ok = wait_flag(0);
            if (ok) load_gamma(0);
            if (ok && nch > 1) {
                ok = wait_flag(1);
                if (ok) load_gamma(1);
            }
        }
        ok = __all_sync(0xffffffffu, ok) && __all_sync(0xffffffffu, mbar_wait_ns(&w_g[0], 0, kWaitNs));
        const float *gam = reinterpret_cast<const float *>(sm + L::GAM);
        if (ok) {
#pragma unroll 1
            for (int k = 0; k < 2; ++k) {
                float x[16];
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    x[u] = si >= 0 ? init_state[si * st_entry + st_head + (size_t)(ib + 16 * k + u) * kD + jrow] : 0.f;
                put_state(k, x, gam);
            }
            if (o) zero_out();
            uint4 vt[2];
            ok = read_v(0, vt);
            if (ok) store_v(vt);
        }
        tmem_st_wait();
        fence_proxy_async_smem();
        tc_fence_before_sync();
        ok = __all_sync(0xffffffffu, ok);
        if (ok && lane == 0) mbar_arrive(&w_ready);
    }
    if (ctl_warp) {
        for (int c = 0; ok && c < nch; ++c) {
            if (lane == 0) {  // polls (the only thread of its warp at work: the group's issuer)
                ok = mbar_wait_spin_ns(&w_ready, (uint32_t)(c & 1), kWaitNs) &&
                     mbar_wait_spin_ns(&w_pp, (uint32_t)(c & 1), kWaitNs);
                if (ok) {
                    tc_fence_after_sync();
                    issue_walk_pv(tmem, sb, o != nullptr);
                    ok = mbar_wait_spin_ns(&w_rec, (uint32_t)(c & 1), kWaitNs);
                    if (ok) issue_walk_ns(tmem, sb, o != nullptr);
                    mma_commit(&w_mma);
                    // record c is in shared memory (its gamma since ready(c)): every read of its
                    // slot has completed, so the slot may be refilled.  A relaxed add: a release
                    // here would wait for this thread's copies in flight, on the walk's chain.
                    if (RING && ok) red_relaxed_add_gpu(cons0 + (size_t)c * H, 1);
                }
                if (ok && c + 2 < nch) {  // the box of chunk c + 2, once that of c + 1 is read
                    ok = mbar_wait_ns(&w_vfree, (uint32_t)((c + 1) & 1), kWaitNs);
                    if (ok) load_v(c + 2);
                }
                if (ok && c + 1 < nch) {
                    ok = mbar_wait_spin_ns(&w_mma, (uint32_t)(c & 1), kWaitNs);  // record c is read
                    // record c + 1's flag was seen (by lane 0 of warp 0) before ready(c)
                    fence_proxy_async_global();
                    if (ok) load_record(c + 1);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
    } else if (state_warp) {
        const int par = lane & 1;  // lane pairs (j, j ^ 1) store two columns of one token
        const int tb = 32 * part + 16 * hs;  // this thread's output tokens tb .. tb + 15
        uint32_t opk[8];           // o_c, paired bf16 columns, 8 token pairs
        // o_c^T (row j, tokens tb ..) into registers, paired over lanes j, j ^ 1; then zeros
        // into the output columns for the next group
        auto read_o = [&]() {
            float v[16];
            tmem_ld16x2_x16<16>(tmem + lane_off + TW_O + 32 * part, v);
            tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                // even lane: (own, partner's) at token 2k; odd lane: (partner's, own) at 2k + 1
                const float mine = par ? v[2 * k + 1] : v[2 * k];
                const float other = __shfl_xor_sync(0xffffffffu, par ? v[2 * k] : v[2 * k + 1], 1);
                opk[k] = par ? pack_bf16x2(other, mine) : pack_bf16x2(mine, other);
            }
            zero_out();
        };
        for (int c = 0; ok && c < nch; ++c) {
            const int64_t cs = t0 + (int64_t)c * kC;
            uint4 vt[2];  // the next chunk's V^T, read while this chunk's products run
            if (c + 1 < nch) ok = read_v(c + 1, vt);
            if (ok && warp == 0 && lane == 0 && c + 2 < nch) {
                // while this chunk's products run: record c + 2's flag, then (its buffer is
                // free once every state warp is past chunk c - 1: ready(c)) its gamma
                ok = wait_flag(c + 2) && mbar_wait_ns(&w_ready, (uint32_t)(c & 1), kWaitNs);
                if (ok) {
                    load_gamma(c + 2);
                    if (c + 2 >= kWalkPrefetchFrom) bulk_prefetch_l2(rec_at(c + 2), kRecBytes);
                }
            }
            ok = __all_sync(0xffffffffu, ok) && __all_sync(0xffffffffu, mbar_wait_ns(&w_mma, (uint32_t)(c & 1), kWaitNs));
            tc_fence_after_sync();
            if (ok && c + 1 < nch) store_v(vt);  // V^T of chunk c is no longer read
            if (c + 1 < nch) {
                if (ok) ok = __all_sync(0xffffffffu, mbar_wait_ns(&w_g[(c + 1) & 1], (uint32_t)(((c + 1) >> 1) & 1), kWaitNs));
                if (ok) {
                    const float *gam = reinterpret_cast<const float *>(sm + L::GAM + ((c + 1) & 1) * kD * 4);
#pragma unroll 1
                    for (int k = 0; k < 2; ++k) {
                        float x[16];
                        load_state(k, x);
                        put_state(k, x, gam);
                    }
                }
                if (ok && o) read_o();
                tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before_sync();
                ok = __all_sync(0xffffffffu, ok);
                if (ok && lane == 0) mbar_arrive(&w_ready);
            } else if (ok) {
                if (o) read_o();
#pragma unroll 1
                for (int k = 0; k < 2 && sf >= 0; ++k) {  // the final state S_T is D
                    float x[16];
                    load_state(k, x);
#pragma unroll
                    for (int u = 0; u < 16; ++u)
                        final_state[sf * st_entry + st_head + (size_t)(ib + 16 * k + u) * kD + jrow] = x[u];
                }
            }
            if (ok && o) {  // the outputs of chunk c, while the next chunk's products run
                __nv_bfloat16 *orow = o + (size_t)h * kD + (jrow & ~1);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int64_t t = cs + tb + 2 * k + par;
                    if (t < t1) *reinterpret_cast<uint32_t *>(orow + (size_t)t * H * kD) = opk[k];
                }
            }
        }
    }
    const bool timed_out = __syncthreads_or(!ok);  // every role has finished or given up
    if (timed_out) {
        if (tid == 0) {
            atomicOr(status, DEV_ERR_TIMEOUT);
            // the gamma copies still in flight (lane 0 of warp 0 issues them all)
            for (int k = g_issued > 2 ? g_issued - 2 : 0; k < g_issued; ++k)
                (void)mbar_wait_ns(&w_g[k & 1], (uint32_t)((k >> 1) & 1), kWaitNs);
        }
        if (ctl_warp && lane == 0) {
            mma_commit(&w_drain);  // completes once every MMA issued so far has
            (void)mbar_wait_ns(&w_drain, 0, kWaitNs);
            // our own copies still in flight: the last phase of each barrier
            if (rec_issued > 0) {
                (void)mbar_wait_ns(&w_rec, (uint32_t)((rec_issued - 1) & 1), kWaitNs);
                (void)mbar_wait_ns(&w_pp, (uint32_t)((rec_issued - 1) & 1), kWaitNs);
            }
            if (v_issued > 0) (void)mbar_wait_ns(&w_v, (uint32_t)((v_issued - 1) & 1), kWaitNs);
        }
    }
    if (!range_ok) atomicOr(status, DEV_ERR_RANGE);
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kWalkTmem);
}

// The streamed prefill: walkers (blockIdx.x < n_walk, two per (sequence, head)) and chunk
// workers in one grid.
template <bool NORM, bool RING>
__global__ void __launch_bounds__(kChunkThreads, 2)
prefill_stream_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_la, const __grid_constant__ CUtensorMap tm_v,
                      const float *__restrict__ log_alpha, const float *__restrict__ beta,
                      const int2 *__restrict__ desc, int H, int chunks, unsigned char *records, int *flags,
                      uint32_t *status, bool scalar_gate, const int32_t *__restrict__ cu, int64_t total,
                      const int32_t *__restrict__ cc, const float *init_state, __nv_bfloat16 *o,
                      float *final_state, StateSlots slots, int n_walk, int ring)
{
    // launched with programmatic stream serialization behind the schedule kernel, which
    // zeroes the flags, the copy counts and the claim counter: nothing it writes is read
    // before this wait
    pdl_wait();
    pdl_launch_dependents();
    // the workspace's ready flags, then the records' copy counts, then the claim counter
    int *cons = flags + (size_t)chunks * H, *claim = cons + (size_t)chunks * H;
    if ((int)blockIdx.x < n_walk)
        walk_unit<RING>((int)blockIdx.x, tm_v, cu, total, H, cc, records, flags, cons, ring, init_state, o,
                        final_state, status, slots);
    else
        chunk_items<NORM, true, RING>(tm_q, tm_k, tm_la, log_alpha, beta, desc, H, 0, chunks, records, status,
                                o != nullptr, scalar_gate, 0, 1, flags, cons, claim, ring);
}

// ============================================================== product-group diagnostic
// Measurement only.  The tensor-core product groups of one prefill kernel, issued back to
// back `reps` times per CTA by the same routines the kernels use, on a constant operand
// image resident in shared memory: no epilogues, no waits between groups, no global
// traffic.  PASS 0: the chunk kernel's groups of one (chunk, head) item (k-k and q-k, W,
// P2, the three-term P, N, Q''), issued by one thread, two CTAs per SM as that kernel runs.
// PASS 1: the state kernel's chain and output groups of one chunk and 64-column slice,
// one CTA per SM, each group issued by a thread of its own warp as in that kernel.
// PASS 2: the streamed kernel's walk group of one chunk (64 value columns, S^T from TMEM,
// the state and output products as one M = 64, N = 192 group), one CTA per SM, one issuing
// thread.
constexpr uint64_t kDiagFlops[3] = {
    2ull * (128 * 64 * 128 + 64 * 128 * 64 + 64 * 64 * 64 + 3 * 128 * 64 * 64 + 128 * 128 * 64 + 64 * 128 * 64),
    2ull * (128 * 64 * 64 + 128 * 64 * 128 + 64 * 64 * 64 + 64 * 64 * 128),
    2ull * (64 * 192 * 64 + 64 * 192 * 128)};
using DiagState = StateShape<64>;  // pass 1 measures the 64-column groups

template <int PASS>
__global__ void __launch_bounds__(256, PASS == 0 ? 2 : 1) tensor_phase_kernel(int reps, uint32_t *status)
{
    extern __shared__ unsigned char smem_raw[];
    __shared__ __align__(8) uint64_t bar[2], bar_drain;
    __shared__ uint32_t tmem_holder;
    constexpr uint32_t used = PASS == 0 ? ChunkLayout::USED : (PASS == 1 ? DiagState::USED : WalkLayout::USED);
    constexpr uint32_t cols = PASS == 0 ? kChunkTmem : (PASS == 1 ? DiagState::TMEM : kWalkTmem);
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    const int tid = threadIdx.x;
    // 0x3c00: 2^-7 as bf16, 1.0 as fp16; finite products and sums in every group
    for (uint32_t e = tid; e < used / 16; e += blockDim.x)
        reinterpret_cast<uint4 *>(sm)[e] = make_uint4(0x3c003c00u, 0x3c003c00u, 0x3c003c00u, 0x3c003c00u);
    fence_proxy_async_smem();
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_init(&bar_drain, PASS == 1 ? 2 : 1);  // one commit per issuing thread
        fence_mbar_init();
    }
    if (tid < 32) {
        tmem_alloc(&tmem_holder, cols);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_holder;
    if (PASS == 2 && tid < 128) {  // the bf16 S^T operand in TMEM: the same constant
        float x[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) x[u] = __uint_as_float(0x3c003c00u);
        for (int c = 0; c < 64; c += 16) tmem_st16(tmem + ((uint32_t)(tid & ~31) << 16) + TW_A + c, x);
        tmem_st_wait();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // PASS 0 and 2: thread 0 issues everything; PASS 1: thread 0 the chain group, thread 128
    // the output group
    const int issuer = tid == 0 ? 0 : (PASS == 1 && tid == 128 ? 1 : -1);
    if (issuer >= 0) {
        bool ok = true;
        for (int r = 0; r < reps && ok; ++r) {
            if (PASS == 0) {
                issue_g1<ChunkLayout>(sb, tmem);
                issue_w_p2<ChunkLayout>(sb, tmem, true);
                issue_p<ChunkLayout>(sb, tmem);
                issue_n_q<ChunkLayout>(sb, tmem, true);
            } else if (PASS == 2) {
                issue_walk(tmem, sb, true);
            } else {
                const uint64_t dr = kdesc(sb), dv = kdesc(sb + DiagState::VIMG), ds = DiagState::sdesc_s(sb + DiagState::O7);
                if (issuer == 0)
                    issue_chain<DiagState>(tmem + DiagState::TM_5, dr, dv, ds);
                else
                    issue_out<DiagState>(tmem + DiagState::TM_O, dr, dv, ds);
            }
            mma_commit(&bar[issuer]);
            ok = mbar_wait_ns(&bar[issuer], (uint32_t)(r & 1), kWaitNs);
            tc_fence_after_sync();
        }
        if (!ok) atomicOr(status, DEV_ERR_TIMEOUT);
    }
    // a drain barrier that every issuer commits to: all MMAs complete before TMEM is freed
    if (issuer >= 0) mma_commit(&bar_drain);
    if (tid == 0) (void)mbar_wait_ns(&bar_drain, 0, kWaitNs);
    tc_fence_before_sync();
    __syncthreads();
    if (tid < 32) tmem_dealloc(tmem, cols);
}

template <int PASS>
cudaError_t run_tensor_phases(int reps, uint32_t *status, cudaStream_t stream, double *tflops)
{
    static int configured = -1, num_sms = 0;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const int smem = PASS == 0 ? (int)kChunkSmem : (PASS == 1 ? (int)DiagState::SMEM : (int)kStreamSmem);
    if (configured != dev) {
        if ((err = cudaFuncSetAttribute(tensor_phase_kernel<PASS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        smem)) != cudaSuccess ||
            (err = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return err;
        configured = dev;
    }
    const int grid = (PASS == 0 ? 2 : 1) * num_sms;
    cudaEvent_t a, b;
    if ((err = cudaEventCreate(&a)) != cudaSuccess) return err;
    if ((err = cudaEventCreate(&b)) != cudaSuccess) { cudaEventDestroy(a); return err; }
    err = cudaEventRecord(a, stream);
    if (err == cudaSuccess) {
        tensor_phase_kernel<PASS><<<grid, 256, smem, stream>>>(reps, status);
        err = cudaGetLastError();
    }
    if (err == cudaSuccess) err = cudaEventRecord(b, stream);
    if (err == cudaSuccess) err = cudaEventSynchronize(b);
    float ms = 0.f;
    if (err == cudaSuccess) err = cudaEventElapsedTime(&ms, a, b);
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    if (err == cudaSuccess) *tflops = (double)grid * reps * (double)kDiagFlops[PASS] / (ms * 1e9);
    return err;
}

}  // namespace

cudaError_t diag_tensor_phases(int pass, int reps, uint32_t *status, cudaStream_t stream, double *tflops)
{
    if (pass == 0) return run_tensor_phases<0>(reps, status, stream, tflops);
    if (pass == 1) return run_tensor_phases<1>(reps, status, stream, tflops);
    return run_tensor_phases<2>(reps, status, stream, tflops);
}

size_t prefill_split_record_bytes() { return kRecBytes; }

size_t prefill_split_records_bytes(int64_t total_tokens, int num_seqs, int num_heads)
{
    return (size_t)(total_tokens / kC + num_seqs) * (size_t)num_heads * kRecBytes;
}

namespace {

// The state pass with SV-column value slices (the chunk kernel has run before it).
template <int SV>
cudaError_t launch_state_pass(const PrefillProblem &p, const int32_t *cc, const unsigned char *rec,
                              cudaLaunchConfig_t cfg, StateSegment seg)
{
    using Sh = StateShape<SV>;
    static int dev_state = -1;
    cudaError_t err = allow_smem(prefill_state_kernel<SV>, (int)Sh::SMEM, &dev_state);
    if (err != cudaSuccess) return err;
    CUtensorMap tv;
    if (!make_map(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.v, p.total_tokens, p.num_heads, 2, SV))
        return cudaErrorInvalidValue;
    cfg.blockDim = dim3(kStateThreads);
    cfg.dynamicSmemBytes = Sh::SMEM;
    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(p.o);
    if (p.split.lseg == 0) {
        cfg.gridDim = dim3(kD / SV, p.num_heads, p.num_seqs);
        return cudaLaunchKernelEx(&cfg, prefill_state_kernel<SV>, tv, tv, p.cu_seqlens, p.total_tokens, p.num_heads,
                                  cc, rec, p.init_state, o, p.final_state, p.status,
                                  static_cast<const int32_t *>(p.order), p.slots, INT_MAX, (float *)nullptr, seg);
    }
    // sequence split: transition pass (R for grid z < nv_max, M above), start states, state pass
    const SeqSplit &s = p.split;
    CUtensorMap tz;  // one zero value row: every box of the transition pass reads zeros
    if (!make_map(&tz, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, s.vzero, 1, p.num_heads, 2, SV))
        return cudaErrorInvalidValue;
    StateSlots sa;
    sa.fin = s.fin_a;
    sa.num = (int64_t)s.nv_max + 1;
    cfg.gridDim = dim3(kD / SV, p.num_heads, 2 * s.nv_max);
    err = cudaLaunchKernelEx(&cfg, prefill_state_kernel<SV>, tv, tz, (const int32_t *)s.vcu, p.total_tokens,
                             p.num_heads, (const int32_t *)s.vcc, rec, (const float *)nullptr,
                             (__nv_bfloat16 *)nullptr, s.R, p.status, (const int32_t *)s.vorder, sa, s.nv_max, s.M,
                             StateSegment());
    if (err != cudaSuccess) return err;
    if ((err = launch_seqsplit_combine(p)) != cudaSuccess) return err;
    StateSlots sc;
    sc.init = s.init_c;
    sc.fin = s.fin_c;
    const int64_t user_entries = p.slots.fin ? p.slots.num : p.num_seqs;
    sc.num = user_entries > (int64_t)s.nv_max + 1 ? user_entries : (int64_t)s.nv_max + 1;
    cfg.gridDim = dim3(kD / SV, p.num_heads, s.nv_max);
    return cudaLaunchKernelEx(&cfg, prefill_state_kernel<SV>, tv, tv, (const int32_t *)s.vcu, p.total_tokens,
                              p.num_heads, (const int32_t *)s.vcc, rec, (const float *)s.start, o, p.final_state,
                              p.status, (const int32_t *)s.vorder, sc, INT_MAX, (float *)nullptr, StateSegment());
}

// SMs of the current device (cached per device).
int sm_count()
{
    static int count[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!count[dev] && cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        count[dev] = 0;
    return count[dev];
}

// The streamed prefill (walkers and chunk workers in one grid of two CTAs per SM), for
// problems with at most kMaxWalkers (sequence, head) units and every record in the
// workspace, or (RING) the records of p.ring_chunks chunks as a ring.  cudaErrorNotSupported when the grid would leave fewer worker CTAs than SMs
// (the caller then runs the two kernels).
template <bool NORM, bool RING>
cudaError_t launch_stream(const PrefillProblem &p, const CUtensorMap &tq, const CUtensorMap &tk,
                          const CUtensorMap &tla, const int32_t *cc, void *records, int units)
{
    static int dev_cfg = -1;
    cudaError_t err = allow_smem(prefill_stream_kernel<NORM, RING>, (int)kStreamSmem, &dev_cfg);
    if (err != cudaSuccess) return err;
    const int sms = sm_count();
    if (sms <= 0 || 2 * sms - (kD / kWalkCols) * units < sms) return cudaErrorNotSupported;
    CUtensorMap tv;  // v boxes of 64 tokens x 64 columns (one walker's value half)
    if (!make_map(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.v, p.total_tokens, p.num_heads, 2, kWalkCols))
        return cudaErrorInvalidValue;
    cudaLaunchAttribute pdl;
    pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = p.stream;
    cfg.attrs = &pdl;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(2 * sms);
    cfg.blockDim = dim3(kChunkThreads);
    cfg.dynamicSmemBytes = kStreamSmem;
    return cudaLaunchKernelEx(&cfg, prefill_stream_kernel<NORM, RING>, tq, tk, tla, tv, p.log_alpha, p.beta,
                              (const int2 *)p.desc, p.num_heads, p.chunk_bound, static_cast<unsigned char *>(records),
                              p.flags, p.status, p.scalar_gate, p.cu_seqlens, p.total_tokens, cc, p.init_state,
                              static_cast<__nv_bfloat16 *>(p.o), p.final_state, p.slots, (kD / kWalkCols) * units,
                              RING ? p.ring_chunks : 0);
}

}  // namespace

int64_t mean_chunks_per_sequence(int32_t num_seqs, int64_t total_tokens)
{
    if (num_seqs <= 0 || total_tokens <= 0) return 0;
    return ((total_tokens + num_seqs - 1) / num_seqs + kC - 1) / kC;
}

bool prefill_stream_fits(int64_t units, int64_t chunks_per_unit, bool force)
{
    const int sms = sm_count();  // the walkers leave at least one worker CTA per SM
    const int64_t walkers = (kD / kWalkCols) * units;
    if (units < 1 || walkers > kMaxWalkers || sms <= 0 || 2 * (int64_t)sms - walkers < sms) return false;
    return force || units >= min_stream_units(chunks_per_unit);
}

bool prefill_stream_eligible(const PrefillProblem &p)
{
    return p.flags && p.split.lseg == 0 && p.seg_chunks == 0 &&
           prefill_stream_fits((int64_t)p.num_seqs * p.num_heads, mean_chunks_per_sequence(p.num_seqs, p.total_tokens),
                               p.stream_force);
}

cudaError_t launch_prefill_split(const PrefillProblem &p, const int32_t *cc, void *records, cudaEvent_t mid)
{
    static int dev_chunk = -1, dev_chunk_norm = -1;
    auto chunk_kernel = p.qk_l2norm ? prefill_chunk_kernel<true> : prefill_chunk_kernel<false>;
    cudaError_t err = allow_smem(chunk_kernel, (int)kChunkSmem, p.qk_l2norm ? &dev_chunk_norm : &dev_chunk);
    if (err != cudaSuccess) return err;
    CUtensorMap tq, tk, tla;
    if (!make_map(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.q, p.total_tokens, p.num_heads, 2, kD) ||
        !make_map(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.k, p.total_tokens, p.num_heads, 2, kD))
        return cudaErrorInvalidValue;
    // a scalar gate ([T, H]) is read by the prefix scan, never by TMA: its map slot repeats q's
    if (p.scalar_gate)
        tla = tq;
    else if (!make_map(&tla, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.log_alpha, p.total_tokens, p.num_heads, 4, kD))
        return cudaErrorInvalidValue;
    const int64_t chunk_bound = p.total_tokens / kC + p.num_seqs;
    if (chunk_bound * p.num_heads > INT32_MAX || !p.desc || p.chunk_bound != chunk_bound)
        return cudaErrorInvalidValue;
    // both kernels may start while the kernel before them drains (programmatic
    // dependent launch); each waits for its inputs with griddepcontrol.wait
    if (p.split.lseg > 0 && (err = launch_seqsplit_plan(p)) != cudaSuccess) return err;
    cudaLaunchAttribute pdl;
    pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = p.stream;
    cfg.attrs = &pdl;
    cfg.numAttrs = 1;
    // 32-column state slices while every (sequence, head, slice) of the pass fits in one wave
    // of SMs (their chain per chunk is shorter); 64-column slices beyond that, and for the
    // sequence split, whose transition pass is sized for them
    // records for only ring_chunks chunks: the streamed kernel or nothing (the two kernels
    // would need every record)
    const bool ring_only = p.ring_chunks > 0 && p.ring_chunks < p.chunk_bound;
    if (prefill_stream_eligible(p)) {
        const int units = p.num_seqs * p.num_heads;
        if (ring_only)
            err = p.qk_l2norm ? launch_stream<true, true>(p, tq, tk, tla, cc, records, units)
                              : launch_stream<false, true>(p, tq, tk, tla, cc, records, units);
        else
            err = p.qk_l2norm ? launch_stream<true, false>(p, tq, tk, tla, cc, records, units)
                              : launch_stream<false, false>(p, tq, tk, tla, cc, records, units);
        if (err != cudaErrorNotSupported || ring_only) {
            if (err == cudaSuccess && mid) err = cudaEventRecord(mid, p.stream);
            return err;
        }
    } else if (ring_only) {
        return cudaErrorInvalidValue;
    }
    const unsigned char *rec = static_cast<const unsigned char *>(records);
    const int64_t slices32 = (int64_t)p.num_seqs * p.num_heads * (kD / 32);
    const bool narrow = p.split.lseg == 0 && slices32 <= sm_count();
    // the records cover seg packed chunks at a time: all of them, or (bounded workspace)
    // segments of p.seg_chunks chunks walked one after the other
    const bool segmented = p.seg_chunks > 0 && p.seg_chunks < chunk_bound;
    const int seg = segmented ? p.seg_chunks : (int)chunk_bound;
    const size_t carry_entry = (size_t)p.num_heads * kD * kD;
    for (int g_lo = 0, k = 0; g_lo < chunk_bound; g_lo += seg, ++k) {
        const int g_hi = g_lo + seg < chunk_bound ? g_lo + seg : (int)chunk_bound;
        // persistent: two CTAs per SM (or one per item when there are fewer)
        const int64_t items = (int64_t)(g_hi - g_lo) * p.num_heads, slots = 2 * (int64_t)sm_count();
        cfg.gridDim = dim3((unsigned)(items < slots || slots <= 0 ? items : slots));
        cfg.blockDim = dim3(kChunkThreads);
        cfg.dynamicSmemBytes = kChunkSmem;
        err = cudaLaunchKernelEx(&cfg, chunk_kernel, tq, tk, tla, p.log_alpha, p.beta, (const int2 *)p.desc,
                                 p.num_heads, g_lo, g_hi - g_lo, static_cast<unsigned char *>(records), p.status,
                                 p.o != nullptr, p.scalar_gate);
        if (err != cudaSuccess) return err;
        if (mid && k == 0 && (err = cudaEventRecord(mid, p.stream)) != cudaSuccess) return err;
        StateSegment sg;
        if (segmented) {
            sg.g_lo = g_lo;
            sg.g_hi = g_hi;
            sg.carry_in = k > 0 ? p.carry + ((k - 1) & 1) * carry_entry : nullptr;
            sg.carry_out = p.carry + (k & 1) * carry_entry;
        }
        err = narrow ? launch_state_pass<32>(p, cc, rec, cfg, sg) : launch_state_pass<64>(p, cc, rec, cfg, sg);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

}  // namespace kda
