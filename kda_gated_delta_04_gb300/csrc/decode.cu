// decode.cu -- fused single-token KDA update (one generated token per sequence).
//
// Per (sequence, head) unit, with the state S (d x d, fp32, value channel
// contiguous) read once and written once:
//   a_i = exp(log_alpha_i);  St = Diag(a) S                     (decay key rows)
//   r_k = St^T k;  r_q = St^T q;  kappa = k . q
//   delta = beta (v - r_k)                                      (scaled residual)
//   o = (r_q + kappa delta) / sqrt(d)   == (St + k delta^T)^T q / sqrt(d)
//   S <- St + k delta^T
// The identity o = St^T q + (k.q) delta lets both reductions come from the same
// pass over St held in registers, before the write pass, so S crosses HBM once
// in each direction ("Day 19, linear attention & KDA", sections 2-3: constant
// work per token, decay first and then the delta write; "K3 attention,
// three-piece set": fixed d_k x d_v state per KDA head).
//
// Layout: 256 threads; each thread owns a float4 column quad of P rows; a warp
// reads whole 512-byte (d = 128) or 256-byte (d = 64) rows with 128-bit loads.
// The reduction over rows is done in registers, then across the rows-per-pass
// groups through shared memory.
#include "common.cuh"

namespace kda {
namespace {

// SCALAR: log_alpha holds one value per unit (scalar gate); QKN: q, k arrive raw and are
// L2-normalised here.  Both are template parameters so that the plain kernel carries
// none of their code.
template <int D, typename IO, bool SCALAR, bool QKN>
__global__ void __launch_bounds__(256, 2)
decode_kernel(const IO *__restrict__ q, const IO *__restrict__ k, const IO *__restrict__ v,
              const float *__restrict__ log_alpha, const float *__restrict__ beta,
              float *__restrict__ state, IO *__restrict__ o, const int32_t *__restrict__ slots,
              int H, int num_slots, uint32_t *errors)
{
    constexpr bool scalar_gate = SCALAR, qk_norm = QKN;
    constexpr int TPR = D / 4;      // threads per state row
    constexpr int RPP = 256 / TPR;  // rows per pass
    constexpr int P = D / RPP;      // rows per thread
    const int unit = blockIdx.x;
    const int tid = threadIdx.x;
    const int c4 = tid % TPR;
    const int r0 = tid / TPR;

    __shared__ float s_a[D], s_k[D], s_q[D];
    __shared__ __align__(16) float s_d[D];  // read as float4
    __shared__ __align__(16) float s_rk[RPP][D];
    __shared__ __align__(16) float s_rq[RPP][D];

    size_t sunit = (size_t)unit;  // the unit's state: its own, or its sequence's pool slot
    if (slots) {
        const int b = unit / H, slot = slots[b];
        if (slot < 0 || slot >= num_slots) {
            if (tid == 0 && errors) atomicOr(errors, DEV_ERR_SLOT);
            return;
        }
        sunit = (size_t)slot * H + (unit - b * H);
    }
    float *S = state + sunit * D * D;
    float4 s[P];
#pragma unroll
    for (int p = 0; p < P; ++p)
        s[p] = __ldcs(reinterpret_cast<const float4 *>(S + (size_t)(r0 + p * RPP) * D) + c4);

    if (tid < D) {
        s_a[tid] = expf(scalar_gate ? log_alpha[unit] : log_alpha[(size_t)unit * D + tid]);
        s_k[tid] = load_io(k + (size_t)unit * D + tid);
        s_q[tid] = load_io(q + (size_t)unit * D + tid);
    }
    __syncthreads();

    float4 rk = make_float4(0.f, 0.f, 0.f, 0.f), rq = rk;
#pragma unroll
    for (int p = 0; p < P; ++p) {
        const int i = r0 + p * RPP;
        const float a = s_a[i], ki = s_k[i], qi = s_q[i];
        s[p].x *= a; s[p].y *= a; s[p].z *= a; s[p].w *= a;
        rk.x += s[p].x * ki; rk.y += s[p].y * ki; rk.z += s[p].z * ki; rk.w += s[p].w * ki;
        rq.x += s[p].x * qi; rq.y += s[p].y * qi; rq.z += s[p].z * qi; rq.w += s[p].w * qi;
    }
    reinterpret_cast<float4 *>(&s_rk[r0][0])[c4] = rk;
    reinterpret_cast<float4 *>(&s_rq[r0][0])[c4] = rq;
    __syncthreads();

    if (tid < D) {
        const int j = tid;
        float sk = 0.f, sq = 0.f, kq = 0.f, kk = 0.f, qq = 0.f;
#pragma unroll
        for (int r = 0; r < RPP; ++r) { sk += s_rk[r][j]; sq += s_rq[r][j]; }
        for (int i = 0; i < D; ++i) kq += s_k[i] * s_q[i];
        // raw q, k (qk_norm): every term is linear in q and in k, so the reciprocal norms
        // scale the reductions instead of the vectors (no extra barrier)
        float nk = 1.f, nq = 1.f;
        if (qk_norm) {
            for (int i = 0; i < D; ++i) { kk += s_k[i] * s_k[i]; qq += s_q[i] * s_q[i]; }
            nk = 1.f / fmaxf(sqrtf(kk), kQkNormEps);
            nq = 1.f / fmaxf(sqrtf(qq), kQkNormEps);
        }
        const float scale = rsqrtf((float)D);
        const float d = beta[unit] * (load_io(v + (size_t)unit * D + j) - sk * nk);
        s_d[j] = d * nk;  // the write k^ d^T = k (nk d)^T
        store_io(o + (size_t)unit * D + j, scale * (sq * nq + kq * (nk * nq) * d));
    }
    __syncthreads();

    const float4 d4 = reinterpret_cast<const float4 *>(s_d)[c4];
#pragma unroll
    for (int p = 0; p < P; ++p) {
        const float ki = s_k[r0 + p * RPP];
        float4 x = s[p];
        x.x += ki * d4.x; x.y += ki * d4.y; x.z += ki * d4.z; x.w += ki * d4.w;
        __stcs(reinterpret_cast<float4 *>(S + (size_t)(r0 + p * RPP) * D) + c4, x);
    }
}

template <int D, typename IO, bool SCALAR, bool QKN>
cudaError_t launch_v(const DecodeProblem &p)
{
    const int units = p.batch * p.num_heads;
    decode_kernel<D, IO, SCALAR, QKN><<<units, 256, 0, p.stream>>>(
        static_cast<const IO *>(p.q), static_cast<const IO *>(p.k), static_cast<const IO *>(p.v),
        p.log_alpha, p.beta, p.state, static_cast<IO *>(p.o), p.slots, p.num_heads, p.num_slots, p.errors);
    return cudaGetLastError();
}
template <int D, typename IO>
cudaError_t launch(const DecodeProblem &p)
{
    if (p.scalar_gate) return p.qk_l2norm ? launch_v<D, IO, true, true>(p) : launch_v<D, IO, true, false>(p);
    return p.qk_l2norm ? launch_v<D, IO, false, true>(p) : launch_v<D, IO, false, false>(p);
}

}  // namespace

cudaError_t launch_decode(const DecodeProblem &p)
{
    if (p.batch == 0 || p.num_heads == 0) return cudaSuccess;
    if (p.d == 128)
        return p.dtype == KDA_DTYPE_BF16 ? launch<128, __nv_bfloat16>(p) : launch<128, float>(p);
    return p.dtype == KDA_DTYPE_BF16 ? launch<64, __nv_bfloat16>(p) : launch<64, float>(p);
}

}  // namespace kda
