// prefill_seqsplit.cu -- the sequence-split state pass of the two-kernel prefill.
//
// The chunkwise form makes every chunk's update affine in the state it starts from
// ("K3 attention, three-piece set", KDA paragraphs: chunkwise parallel form, WY
// representation and UT transform; the state is a fixed d_k x d_v matrix per head).
// A run of chunks therefore composes to S_end = M S_start + R, with M the product of the
// chunks' linear parts and R the end state reached from zero.  When a problem has few
// (sequence, head) units the serial state pass leaves most SMs idle; cutting every
// sequence into segments lets the state kernel run
//   1. a transition pass: for each segment but the last of its sequence, R (zero start,
//      the real values) and M (identity start, zero values), all segments at once;
//   2. the combine kernel here: S_start(k + 1) = M_k S_start(k) + R_k in fp32, serial
//      over the few segments of a sequence;
//   3. the state pass proper over all segments at once, each from its true start,
//      writing the outputs and (last segment) the final state.
// The same kernels and records serve both passes; segment boundaries fall on chunk
// boundaries, so no chunk-local work changes.
#include "common.cuh"

namespace kda {

namespace {

constexpr int kD = 128;             // d_k = d_v of the two-kernel path
constexpr int kSplitSMs = 152;      // SMs of a GB300; the transition pass targets one wave
constexpr int kMinSegChunks = 4;    // shortest segment worth a separate start state
constexpr int kPlanThreads = 1024;

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// Exclusive scan of one value per thread over the block, plus the block total.
__device__ int block_exclusive_scan(int x, int &total)
{
    __shared__ int warp_sums[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    int incl = x;
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
    total = warp_sums[31];
    const int before = warp > 0 ? warp_sums[warp - 1] : 0;
    __syncthreads();  // warp_sums is reused by the next call
    return before + incl - x;
}

// One block.  Segment tables from cu_seqlens and the packed chunk numbering cc.
__global__ void __launch_bounds__(kPlanThreads)
seqsplit_plan_kernel(const int32_t *__restrict__ cu, const int32_t *__restrict__ cc, int num_seqs,
                     int64_t total, int H, SeqSplit s, StateSlots user, bool has_init, uint32_t *status)
{
    const int L = s.lseg;
    // segments per sequence, scanned into seg_first
    int carry = 0;
    for (int base = 0; base < num_seqs; base += blockDim.x) {
        const int n = base + threadIdx.x;
        int k = 0;
        if (n < num_seqs) {
            const int chunks = cc[n + 1] - cc[n];
            k = chunks > L ? (chunks + L - 1) / L : 1;
        }
        int tot;
        const int ex = block_exclusive_scan(k, tot);
        if (n < num_seqs) s.seg_first[n] = carry + ex;
        carry += tot;
    }
    const int nv = carry < s.nv_max ? carry : s.nv_max;  // nv_max bounds it by construction
    if (threadIdx.x == 0) s.seg_first[num_seqs] = nv;
    __syncthreads();
    for (int n = threadIdx.x; n < num_seqs; n += blockDim.x) {
        int64_t t0, t1, si, sf;
        seq_range(cu, n, total, t0, t1);
        if (!state_entries(user, n, has_init, si, sf)) atomicOr(status, DEV_ERR_SLOT);
        s.init_src[n] = (int32_t)si;
        const int v0 = s.seg_first[n], v1 = s.seg_first[n + 1];
        for (int v = v0; v < v1 && v < nv; ++v) {
            const int k = v - v0;
            const bool last = v == v1 - 1;
            s.vcu[v] = (int32_t)(t0 + (int64_t)k * L * kChunk);
            s.vcc[v] = cc[n] + k * L;
            s.vorder[v] = v;
            s.fin_a[v] = last ? -1 : v;
            s.init_c[v] = v;
            s.fin_c[v] = last ? (int32_t)sf : -1;
        }
    }
    // the end of the last segment, then an empty sentinel segment for the spare grid slots
    for (int v = nv + threadIdx.x; v <= s.nv_max; v += blockDim.x) {
        s.vcu[v] = (int32_t)total;
        s.vcc[v] = cc[num_seqs];
        if (v < s.nv_max) s.vorder[v] = nv;
        s.fin_a[v] = -1;
        s.init_c[v] = -1;
        s.fin_c[v] = -1;
    }
    if (threadIdx.x == 0) {
        s.vcu[s.nv_max + 1] = (int32_t)total;
        s.vcc[s.nv_max + 1] = cc[num_seqs];
    }
    uint32_t *z = static_cast<uint32_t *>(s.vzero);
    for (int e = threadIdx.x; e < H * kD / 2; e += blockDim.x) z[e] = 0u;
}

// One CTA per (8-column slice, head, sequence): the start state of every segment,
// S_start(0) = the sequence's initial state, S_start(k + 1) = M_k S_start(k) + R_k (fp32).
// M_k is staged transposed in shared memory (a warp loads 32 rows of one column quad, so
// the transposing stores are conflict-free) while the registers already hold M_{k+1}'s
// loads in flight.  Thread: rows 4ib .. 4ib + 3 of column j.
constexpr int kCombThreads = 256, kCols = 8;
__global__ void __launch_bounds__(kCombThreads)
seqsplit_combine_kernel(SeqSplit s, const float *init_state, int H)
{
    extern __shared__ __align__(16) float comb_smem[];
    float *MT = comb_smem;            // [kD][kD]: MT[m][i] = M[i][m]
    float *S = comb_smem + kD * kD;   // [kD][kCols]
    const int j0 = blockIdx.x * kCols, h = blockIdx.y, n = blockIdx.z, tid = threadIdx.x;
    const int v0 = s.seg_first[n];
    const int nseg = min(s.seg_first[n + 1], s.seg_first[gridDim.z]) - v0;
    const int si = s.init_src[n];
    const size_t entry = (size_t)H * kD * kD, head = (size_t)h * kD * kD;
    const int ib = tid >> 3, j = tid & 7;          // compute: rows 4ib.., column j
    const int li = tid & 31, lq = tid >> 5;        // staging: row li + 32 (r & 3), quad lq + 8 (r >> 2)
    for (int e = tid; e < kD * kCols; e += kCombThreads) {
        const int i = e / kCols, c = e % kCols;
        const float x = (init_state && si >= 0) ? init_state[si * entry + head + (size_t)i * kD + j0 + c] : 0.f;
        S[i * kCols + c] = x;
        if (nseg > 0) s.start[v0 * entry + head + (size_t)i * kD + j0 + c] = x;
    }
    float4 mr[16];
    auto load_m = [&](size_t v) {
        const float *Mv = s.M + v * entry + head;
#pragma unroll
        for (int r = 0; r < 16; ++r)
            mr[r] = *reinterpret_cast<const float4 *>(Mv + (size_t)(li + 32 * (r & 3)) * kD + 4 * (lq + 8 * (r >> 2)));
    };
    if (nseg > 1) load_m((size_t)v0);
    for (int k = 0; k + 1 < nseg; ++k) {
        const size_t v = (size_t)(v0 + k);
        __syncthreads();  // the previous step has finished reading MT and S
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const int i = li + 32 * (r & 3), m = 4 * (lq + 8 * (r >> 2));
            MT[(m + 0) * kD + i] = mr[r].x;
            MT[(m + 1) * kD + i] = mr[r].y;
            MT[(m + 2) * kD + i] = mr[r].z;
            MT[(m + 3) * kD + i] = mr[r].w;
        }
        if (k + 2 < nseg) load_m(v + 1);  // in flight during this step's products
        float acc[4];
        const float *Rv = s.R + v * entry + head + j0 + j;
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = Rv[(size_t)(4 * ib + q) * kD];
        __syncthreads();
#pragma unroll 8
        for (int m = 0; m < kD; ++m) {
            const float4 a = *reinterpret_cast<const float4 *>(MT + m * kD + 4 * ib);
            const float b = S[m * kCols + j];
            acc[0] = fmaf(a.x, b, acc[0]);
            acc[1] = fmaf(a.y, b, acc[1]);
            acc[2] = fmaf(a.z, b, acc[2]);
            acc[3] = fmaf(a.w, b, acc[3]);
        }
        __syncthreads();  // every thread has read S_start(k)
        float *dst = s.start + (v + 1) * entry + head + j0 + j;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            S[(4 * ib + q) * kCols + j] = acc[q];
            dst[(size_t)(4 * ib + q) * kD] = acc[q];
        }
    }
}
constexpr size_t kCombSmem = (size_t)(kD * kD + kD * kCols) * sizeof(float);

}  // namespace

int seqsplit_lseg(int num_seqs, int64_t total_tokens, int num_heads)
{
    if (num_seqs <= 0 || num_heads <= 0 || total_tokens <= 0) return 0;
    const int64_t units = (int64_t)num_seqs * num_heads;
    // the transition pass runs 4 CTAs (R and M, two 64-column slices each) per segment and head
    const int64_t kmax = 1 + kSplitSMs / (4 * units);
    const int64_t avg = (total_tokens / kChunk + num_seqs) / num_seqs;  // chunks per sequence
    // The split pays once the serial pass it shortens outweighs the transition pass and the
    // chaining it adds, which takes longer sequences the more units there are.  Timed on one
    // sequence (the two kernels against the split): from about 72 chunks with up to 8 units,
    // about 190 with 16, between 192 and 256 with 19 (T = 4096, 64 chunks: the two kernels
    // 0.085 against 0.099 ms at 4 heads, 0.124 against 0.152 at 19; T = 16384: the split
    // 0.199 against 0.320 ms at 4 heads, 0.460 against 0.473 at 19).
    if (avg < (units <= 8 ? 72 : 15 * units - 50)) return 0;
    int64_t k = avg / kMinSegChunks;
    if (k > kmax) k = kmax;
    if (k < 3) return 0;  // two segments cost as much as they save
    return (int)((avg + k - 1) / k);
}

int seqsplit_nv_max(int lseg, int num_seqs, int64_t total_tokens)
{
    return lseg > 0 ? (int)((total_tokens / kChunk + num_seqs) / lseg + num_seqs + 1) : 0;
}

namespace {
size_t table_bytes(int nv_max, int num_seqs)
{
    return 3 * round256(((size_t)nv_max + 2) * 4) + 3 * round256(((size_t)nv_max + 1) * 4) +
           round256(((size_t)num_seqs + 1) * 4) + round256((size_t)num_seqs * 4);
}
}  // namespace

size_t seqsplit_bytes(int num_seqs, int64_t total_tokens, int num_heads)
{
    const int lseg = seqsplit_lseg(num_seqs, total_tokens, num_heads);
    if (!lseg) return 0;
    const int nv_max = seqsplit_nv_max(lseg, num_seqs, total_tokens);
    return table_bytes(nv_max, num_seqs) + 3 * (size_t)nv_max * num_heads * kD * kD * sizeof(float) +
           round256((size_t)num_heads * kD * 2);
}

void seqsplit_carve(SeqSplit &s, int num_seqs, int64_t total_tokens, int num_heads, char *ws)
{
    s.lseg = seqsplit_lseg(num_seqs, total_tokens, num_heads);
    if (!s.lseg) return;
    s.nv_max = seqsplit_nv_max(s.lseg, num_seqs, total_tokens);
    const size_t big = (size_t)s.nv_max * num_heads * kD * kD * sizeof(float);
    s.R = reinterpret_cast<float *>(ws); ws += big;  // the large buffers first (256-aligned)
    s.M = reinterpret_cast<float *>(ws); ws += big;
    s.start = reinterpret_cast<float *>(ws); ws += big;
    auto take = [&](size_t count) {
        int32_t *q = reinterpret_cast<int32_t *>(ws);
        ws += round256(count * 4);
        return q;
    };
    s.vcu = take((size_t)s.nv_max + 2);
    s.vcc = take((size_t)s.nv_max + 2);
    s.vorder = take((size_t)s.nv_max + 2);
    s.fin_a = take((size_t)s.nv_max + 1);
    s.init_c = take((size_t)s.nv_max + 1);
    s.fin_c = take((size_t)s.nv_max + 1);
    s.seg_first = take((size_t)num_seqs + 1);
    s.init_src = take((size_t)num_seqs);
    s.vzero = ws;
}

cudaError_t launch_seqsplit_plan(const PrefillProblem &p)
{
    const bool has_init = p.init_state != nullptr;
    seqsplit_plan_kernel<<<1, kPlanThreads, 0, p.stream>>>(p.cu_seqlens, p.cc, p.num_seqs, p.total_tokens,
                                                           p.num_heads, p.split, p.slots, has_init, p.status);
    return cudaGetLastError();
}

cudaError_t launch_seqsplit_combine(const PrefillProblem &p)
{
    static int configured_device = -1;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (configured_device != dev) {
        err = cudaFuncSetAttribute(seqsplit_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)kCombSmem);
        if (err != cudaSuccess) return err;
        configured_device = dev;
    }
    dim3 grid(kD / kCols, p.num_heads, p.num_seqs);
    seqsplit_combine_kernel<<<grid, kCombThreads, kCombSmem, p.stream>>>(p.split, p.init_state, p.num_heads);
    return cudaGetLastError();
}

}  // namespace kda
