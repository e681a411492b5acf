// prefill_simt.cu -- chunkwise KDA prefill on CUDA cores (fp32 arithmetic).
//
// The exact path: every product is an fp32 FFMA, so fp32 inputs reach the
// oracle to ~1e-6.  One CTA owns one (sequence, head, value-column slice); the
// recurrence is independent across value columns, so slices run in parallel
// and only the chunk-local key/query work is repeated per slice.
//
// Per chunk of C = 64 rows (rows past the end of the sequence are zero-filled,
// with log_alpha = 0 and beta = 0, which makes them inert):
//   a1  g_r     = sum_{s<=r} log_alpha_s           (per key channel)
//   a2  Qg = scale q e^g, Kg = k e^g, Ki = k e^-g, Kd = k e^(g_last - g)
//   a3  A   = strict-lower(diag(beta) Kg Ki^T),  Aqk = lower(Qg Ki^T)
//   a4-a6 (I + A) U = diag(beta)(V - Kg S)          forward substitution
//       o   = Qg S + Aqk U
//   a7  S  <- Diag(e^g_last) S + Kd^T U
// This is the chunkwise-parallel form the pages name without its algebra
// ("K3 attention, three-piece set", KDA engineering details: chunkwise with WY
// representation and UT transform; "From 124M to 2.8T", chapter 3: parallel
// inside a chunk, serial across chunks).  Here the triangular system is solved
// directly against the state-dependent right-hand side, which is the same
// algebra as the UT/WY factors with the multiplication by S moved inside.
#include <algorithm>

#include "common.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;

// ---------------------------------------------------------------- prep kernel
// Clears the workspace error word, checks cu_seqlens, writes the order in
// which sequences are processed (longest first, ties by index) and, when cc is
// given, each sequence's first chunk in a packed chunk numbering
// (cc[n] = sum over m < n of ceil(len_m / 64); cc[num_seqs] = all chunks) and, when desc
// is given, every packed chunk's first token and row count (0 rows past the last chunk),
// so that a chunk CTA finds its rows with one load.
constexpr int kPrepStaged = 4096;  // sequences whose boundaries and chunk offsets live in shared memory

__global__ void prefill_prep_kernel(const int32_t *__restrict__ cu, int num_seqs, int64_t total,
                                    uint32_t *status, int32_t *order, int32_t *cc, int2 *desc,
                                    int chunk_bound, int *flags, int64_t num_flags)
{
    // the chunk kernel may be scheduled now; it waits for this kernel's results itself
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (int64_t e = threadIdx.x; e < num_flags; e += blockDim.x) flags[e] = 0;  // no record published yet
    __shared__ int bad;
    // up to kPrepStaged sequences: cu (clamped as seq_range clamps it) and the chunk offsets
    // cc are kept here, so the sort and the descriptor search read no global memory
    __shared__ int32_t s_cu[kPrepStaged + 1];
    __shared__ int32_t s_cc[kPrepStaged + 1];
    const bool staged = cu && num_seqs <= kPrepStaged;
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    if (cu) {
        for (int n = threadIdx.x; n <= num_seqs; n += blockDim.x) {
            const int64_t c = cu[n];
            if (n == 0 && c != 0) bad = 1;
            if (n == num_seqs && c != total) bad = 1;
            if (n < num_seqs && cu[n + 1] < c) bad = 1;
            if (staged) s_cu[n] = c;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) *status = bad ? DEV_ERR_SEQLENS : 0u;
    // the range [t0, t1) of sequence n, clamped exactly as seq_range clamps it
    auto range = [&](int n, int64_t &t0, int64_t &t1) {
        if (!staged) { seq_range(cu, n, total, t0, t1); return; }
        int64_t a = s_cu[n], b = s_cu[n + 1];
        a = a < 0 ? 0 : (a > total ? total : a);
        b = b < a ? a : (b > total ? total : b);
        t0 = a;
        t1 = b;
    };
    const bool sort = cu && num_seqs <= kPrepStaged;
    for (int n = threadIdx.x; n < num_seqs; n += blockDim.x) {
        if (!sort) { order[n] = n; continue; }
        int64_t t0, t1;
        range(n, t0, t1);
        const int64_t len = t1 - t0;
        int rank = 0;
        for (int m = 0; m < num_seqs; ++m) {
            int64_t a0, a1;
            range(m, a0, a1);
            const int64_t lm = a1 - a0;
            rank += (lm > len) || (lm == len && m < n);
        }
        order[rank] = n;
    }
    if (!cc) return;
    __shared__ int warp_sums[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    int carry = 0;
    for (int base = 0; base < num_seqs; base += blockDim.x) {
        const int n = base + threadIdx.x;
        int cnt = 0;
        if (n < num_seqs) {
            int64_t t0, t1;
            range(n, t0, t1);
            cnt = (int)((t1 - t0 + kChunk - 1) / kChunk);
        }
        int incl = cnt;  // inclusive scan inside the warp
        for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += t;
        }
        if (lane == 31) warp_sums[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = lane < nwarps ? warp_sums[lane] : 0;
            for (int off = 1; off < 32; off <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off) w += t;
            }
            warp_sums[lane] = w;
        }
        __syncthreads();
        const int before = warp > 0 ? warp_sums[warp - 1] : 0;
        if (n < num_seqs) {
            cc[n] = carry + before + incl - cnt;
            if (staged || !cu) s_cc[n] = carry + before + incl - cnt;
        }
        carry += warp_sums[31];
        __syncthreads();
    }
    if (threadIdx.x == 0) cc[num_seqs] = carry;
    if (!desc) return;
    const bool cc_shared = staged || !cu;  // (without cu_seqlens there is one sequence)
    __syncthreads();  // cc complete (global writes of this block are visible to it after the barrier)
    for (int g = threadIdx.x; g < chunk_bound; g += blockDim.x) {
        int2 d = make_int2(0, 0);
        if (g < carry) {
            int lo = 0, hi = num_seqs;  // the sequence n with cc[n] <= g < cc[n + 1]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if ((cc_shared ? s_cc[mid] : cc[mid]) <= g) lo = mid; else hi = mid;
            }
            int64_t t0, t1;
            range(lo, t0, t1);
            const int64_t c0 = t0 + (int64_t)(g - (cc_shared ? s_cc[lo] : cc[lo])) * kChunk;
            d = make_int2((int)c0, (int)((t1 - c0) < kChunk ? (t1 - c0) : kChunk));
        }
        desc[g] = d;
    }
}

// ---------------------------------------------------------------- SIMT chunk kernel
template <int D, int DV>
struct SimtSmem {
    static constexpr int LD = D + 4;   // padded row stride (floats) of C x D tiles
    static constexpr int LA = kChunk + 1;
    float q[kChunk * LD];              // q, then Qg
    float k[kChunk * LD];              // k, then Kd
    float g[kChunk * LD];              // log_alpha, then g, then Kg
    float ki[kChunk * LD];             // Ki
    float v[kChunk * DV];              // v, then rhs, then U
    float S[D * DV];                   // state slice
    float A[kChunk * LA];
    float Aqk[kChunk * LA];
    float beta[kChunk];
    float glast[D];
};

template <int D, int DV, typename IO>
__global__ void __launch_bounds__(kThreads, 1)
prefill_simt_kernel(const IO *__restrict__ q, const IO *__restrict__ k, const IO *__restrict__ v,
                    const float *__restrict__ log_alpha, const float *__restrict__ beta,
                    const int32_t *__restrict__ cu, int64_t total, int H,
                    const float *init_state, IO *__restrict__ o, float *final_state,
                    uint32_t *status, const int32_t *__restrict__ order, bool scalar_gate,
                    StateSlots slots, bool qk_norm)
{
    using Sm = SimtSmem<D, DV>;
    constexpr int LD = Sm::LD, LA = Sm::LA;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Sm &sm = *reinterpret_cast<Sm *>(smem_raw);

    const int slice = blockIdx.x, h = blockIdx.y;
    const int n = order[blockIdx.z];
    const int tid = threadIdx.x;
    const int j0 = slice * DV;
    int64_t t0, t1;
    seq_range(cu, n, total, t0, t1);
    const float scale = rsqrtf((float)D);

    // state slice S[i][j0 .. j0+DV)
    int64_t si, sf;
    if (!state_entries(slots, n, init_state != nullptr, si, sf) && tid == 0) atomicOr(status, DEV_ERR_SLOT);
    const size_t head_off = (size_t)h * D * D, st_entry = (size_t)H * D * D;
    for (int e = tid; e < D * DV; e += kThreads) {
        const int i = e / DV, j = e % DV;
        sm.S[e] = si >= 0 ? init_state[si * st_entry + head_off + (size_t)i * D + j0 + j] : 0.f;
    }
    bool decay_bad = false;

    for (int64_t c0 = t0; c0 < t1; c0 += kChunk) {
        const int len = (t1 - c0) < kChunk ? (int)(t1 - c0) : kChunk;
        __syncthreads();  // previous chunk finished with shared memory
        // ---- load the chunk (zero rows past the end)
        for (int e = tid; e < kChunk * (D / 4); e += kThreads) {
            const int r = e / (D / 4), i4 = (e % (D / 4)) * 4;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a, c = a;
            if (r < len) {
                const size_t row = ((size_t)(c0 + r) * H + h) * D + i4;
                a = load4_io(q + row);
                b = load4_io(k + row);
                if (scalar_gate) {  // log_alpha [T, H]: one decay for every key channel
                    const float x = log_alpha[(size_t)(c0 + r) * H + h];
                    c = make_float4(x, x, x, x);
                } else {
                    c = *reinterpret_cast<const float4 *>(log_alpha + row);
                }
            }
            *reinterpret_cast<float4 *>(&sm.q[r * LD + i4]) = a;
            *reinterpret_cast<float4 *>(&sm.k[r * LD + i4]) = b;
            *reinterpret_cast<float4 *>(&sm.g[r * LD + i4]) = c;
        }
        for (int e = tid; e < kChunk * (DV / 4); e += kThreads) {
            const int r = e / (DV / 4), j4 = (e % (DV / 4)) * 4;
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < len) a = load4_io(v + ((size_t)(c0 + r) * H + h) * D + j0 + j4);
            *reinterpret_cast<float4 *>(&sm.v[r * DV + j4]) = a;
        }
        if (tid < kChunk) sm.beta[tid] = tid < len ? beta[(size_t)(c0 + tid) * H + h] : 0.f;
        __syncthreads();

        // ---- q / k L2 normalisation, in place in fp32 (one warp per row); nothing below
        // reads q or k before the barrier after a1
        if (qk_norm) {
            const int warp = tid >> 5, lane = tid & 31;
            for (int row = warp; row < 2 * kChunk; row += kThreads / 32) {
                float *x = row < kChunk ? &sm.q[row * LD] : &sm.k[(row - kChunk) * LD];
                float ss = 0.f;
                for (int i = lane; i < D; i += 32) ss += x[i] * x[i];
#pragma unroll
                for (int m = 16; m; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
                const float inv = 1.f / fmaxf(sqrtf(ss), kQkNormEps);
                for (int i = lane; i < D; i += 32) x[i] *= inv;
            }
        }

        // ---- a1: in-chunk cumulative log-decay per channel
        if (tid < D) {
            float acc = 0.f, lo = 0.f, hi = 0.f;
            for (int r = 0; r < kChunk; ++r) {
                acc += sm.g[r * LD + tid];
                sm.g[r * LD + tid] = acc;
                lo = fminf(lo, acc);
                hi = fmaxf(hi, acc);
            }
            sm.glast[tid] = acc;
            if (lo < KDA_MIN_CHUNK_LOG_DECAY || hi > -KDA_MIN_CHUNK_LOG_DECAY) decay_bad = true;
        }
        __syncthreads();

        // ---- a2: decayed operands
        for (int e = tid; e < kChunk * D; e += kThreads) {
            const int r = e / D, i = e % D;
            const float g = sm.g[r * LD + i], kk = sm.k[r * LD + i];
            const float eg = expf(g);
            sm.q[r * LD + i] = scale * sm.q[r * LD + i] * eg;
            sm.g[r * LD + i] = kk * eg;
            sm.ki[r * LD + i] = kk * expf(-g);
            sm.k[r * LD + i] = kk * expf(sm.glast[i] - g);
        }
        __syncthreads();

        // ---- a3: A and Aqk (4x4 register tiles; rows rb+16u, columns sb+16w)
        {
            const int rb = tid / 16, sb = tid % 16;
            float accA[4][4] = {}, accQ[4][4] = {};
            for (int i = 0; i < D; i += 4) {
                float4 kg[4], qg[4], kv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    kg[u] = *reinterpret_cast<const float4 *>(&sm.g[(rb + 16 * u) * LD + i]);
                    qg[u] = *reinterpret_cast<const float4 *>(&sm.q[(rb + 16 * u) * LD + i]);
                    kv[u] = *reinterpret_cast<const float4 *>(&sm.ki[(sb + 16 * u) * LD + i]);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        accA[u][w] += kg[u].x * kv[w].x + kg[u].y * kv[w].y + kg[u].z * kv[w].z +
                                      kg[u].w * kv[w].w;
                        accQ[u][w] += qg[u].x * kv[w].x + qg[u].y * kv[w].y + qg[u].z * kv[w].z +
                                      qg[u].w * kv[w].w;
                    }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    const int r = rb + 16 * u, s = sb + 16 * w;
                    sm.A[r * LA + s] = s < r ? sm.beta[r] * accA[u][w] : 0.f;
                    sm.Aqk[r * LA + s] = s <= r ? accQ[u][w] : 0.f;
                }
        }
        // ---- right-hand side diag(beta)(V - Kg S), in place over V
        {
            const int j = tid % DV;
            for (int r = tid / DV; r < kChunk; r += kThreads / DV) {
                float acc = 0.f;
                for (int i = 0; i < D; ++i) acc += sm.g[r * LD + i] * sm.S[i * DV + j];
                sm.v[r * DV + j] = sm.beta[r] * (sm.v[r * DV + j] - acc);
            }
        }
        __syncthreads();

        // ---- a4-a5: forward substitution (I + A) U = rhs, one lane per value column
        if (tid < DV) {
            const int j = tid;
            for (int r = 1; r < kChunk; ++r) {
                float acc = sm.v[r * DV + j];
                for (int s = 0; s < r; ++s) acc -= sm.A[r * LA + s] * sm.v[s * DV + j];
                sm.v[r * DV + j] = acc;
            }
        }
        __syncthreads();

        // ---- a6: output o = Qg S + Aqk U (skipped when no outputs are wanted)
        if (o) {
            const int j = tid % DV;
            for (int r = tid / DV; r < len; r += kThreads / DV) {
                float acc = 0.f;
                for (int i = 0; i < D; ++i) acc += sm.q[r * LD + i] * sm.S[i * DV + j];
                for (int s = 0; s <= r; ++s) acc += sm.Aqk[r * LA + s] * sm.v[s * DV + j];
                store_io(o + ((size_t)(c0 + r) * H + h) * D + j0 + j, acc);
            }
        }
        __syncthreads();

        // ---- a7: state propagation S <- Diag(e^glast) S + Kd^T U
        {
            const int j = tid % DV;
            for (int i = tid / DV; i < D; i += kThreads / DV) {
                float acc = expf(sm.glast[i]) * sm.S[i * DV + j];
                for (int r = 0; r < kChunk; ++r) acc += sm.k[r * LD + i] * sm.v[r * DV + j];
                sm.S[i * DV + j] = acc;
            }
        }
    }
    __syncthreads();
    for (int e = tid; e < D * DV && sf >= 0; e += kThreads) {
        const int i = e / DV, j = e % DV;
        final_state[sf * st_entry + head_off + (size_t)i * D + j0 + j] = sm.S[e];
    }
    if (decay_bad) atomicOr(status, DEV_ERR_DECAY);
}

template <int D, int DV, typename IO>
cudaError_t launch_simt(const PrefillProblem &p)
{
    constexpr size_t smem = sizeof(SimtSmem<D, DV>);
    auto kern = prefill_simt_kernel<D, DV, IO>;
    static int configured_device = -1;  // attribute is per device context
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (configured_device != dev) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        configured_device = dev;
    }
    dim3 grid(D / DV, p.num_heads, p.num_seqs);
    kern<<<grid, kThreads, smem, p.stream>>>(
        static_cast<const IO *>(p.q), static_cast<const IO *>(p.k), static_cast<const IO *>(p.v),
        p.log_alpha, p.beta, p.cu_seqlens, p.total_tokens, p.num_heads, p.init_state,
        static_cast<IO *>(p.o), p.final_state, p.status, p.order, p.scalar_gate, p.slots, p.qk_l2norm);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_prep(const PrefillProblem &p)
{
    // the ready flag and the copy count of every chunk-head record and, after them, the
    // streamed kernel's claim counter
    const int64_t num_flags = p.flags ? 2 * (int64_t)p.chunk_bound * p.num_heads + 1 : 0;
    prefill_prep_kernel<<<1, 1024, 0, p.stream>>>(p.cu_seqlens, p.num_seqs, p.total_tokens,
                                                  p.status, p.order, p.cc, p.desc, p.chunk_bound,
                                                  p.flags, num_flags);
    return cudaGetLastError();
}

cudaError_t launch_prefill_simt(const PrefillProblem &p)
{
    if (p.d == 128)
        return p.dtype == KDA_DTYPE_BF16 ? launch_simt<128, 32, __nv_bfloat16>(p)
                                         : launch_simt<128, 32, float>(p);
    return p.dtype == KDA_DTYPE_BF16 ? launch_simt<64, 32, __nv_bfloat16>(p)
                                     : launch_simt<64, 32, float>(p);
}

}  // namespace kda
