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
// Layout: 256 threads, 8 warps; warp w owns the value columns [D/8 w, D/8 (w+1)) over
// all D key rows.  Lane = (row lane rl, column quad cq) with CQ = D/32 quads per warp
// and RL = 32/CQ row lanes, so one 128-bit load per lane covers RL whole rows of the
// warp's stripe; a thread keeps the float4 quad of P = D/RL rows (rl, rl + RL, ...).
// Both reductions over the key rows end in the warp: a lane sums its P rows in
// registers, then a butterfly of warp shuffles over the row lanes leaves every lane
// with its columns' S~^T k and S~^T q, so delta, o and the write need no further
// barrier.  k.q is a butterfly over the whole warp.
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
    constexpr int CQ = D / 32;   // column quads per warp (8 warps x CQ quads = D / 4)
    constexpr int RL = 32 / CQ;  // row lanes
    constexpr int P = D / RL;    // rows per thread
    const int unit = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rl = lane / CQ;
    const int c4 = warp * CQ + lane % CQ;  // this thread's column quad

    __shared__ float s_a[D], s_k[D], s_q[D];

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
        s[p] = __ldcs(reinterpret_cast<const float4 *>(S + (size_t)(rl + p * RL) * D) + c4);

    if (tid < D) {
        s_a[tid] = expf(scalar_gate ? log_alpha[unit] : log_alpha[(size_t)unit * D + tid]);
        s_k[tid] = load_io(k + (size_t)unit * D + tid);
        s_q[tid] = load_io(q + (size_t)unit * D + tid);
    }
    __syncthreads();

    float4 rk = make_float4(0.f, 0.f, 0.f, 0.f), rq = rk;
#pragma unroll
    for (int p = 0; p < P; ++p) {
        const int i = rl + p * RL;
        const float a = s_a[i], ki = s_k[i], qi = s_q[i];
        s[p].x *= a; s[p].y *= a; s[p].z *= a; s[p].w *= a;
        rk.x += s[p].x * ki; rk.y += s[p].y * ki; rk.z += s[p].z * ki; rk.w += s[p].w * ki;
        rq.x += s[p].x * qi; rq.y += s[p].y * qi; rq.z += s[p].z * qi; rq.w += s[p].w * qi;
    }
    // k.q (and the squared norms for raw q, k): lane l sums rows l, l + 32, ...
    float kq = 0.f, kk = 0.f, qq = 0.f;
#pragma unroll
    for (int i = lane; i < D; i += 32) {
        const float ki = s_k[i], qi = s_q[i];
        kq += ki * qi;
        if (qk_norm) { kk += ki * ki; qq += qi * qi; }
    }
#pragma unroll
    for (int m = CQ; m < 32; m <<= 1) {  // over the row lanes: the column sums
        rk.x += __shfl_xor_sync(0xffffffffu, rk.x, m); rk.y += __shfl_xor_sync(0xffffffffu, rk.y, m);
        rk.z += __shfl_xor_sync(0xffffffffu, rk.z, m); rk.w += __shfl_xor_sync(0xffffffffu, rk.w, m);
        rq.x += __shfl_xor_sync(0xffffffffu, rq.x, m); rq.y += __shfl_xor_sync(0xffffffffu, rq.y, m);
        rq.z += __shfl_xor_sync(0xffffffffu, rq.z, m); rq.w += __shfl_xor_sync(0xffffffffu, rq.w, m);
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {  // over the whole warp: the dot products
        kq += __shfl_xor_sync(0xffffffffu, kq, m);
        if (qk_norm) {
            kk += __shfl_xor_sync(0xffffffffu, kk, m);
            qq += __shfl_xor_sync(0xffffffffu, qq, m);
        }
    }
    // raw q, k (qk_norm): every term is linear in q and in k, so the reciprocal norms
    // scale the reductions instead of the vectors
    float nk = 1.f, nq = 1.f;
    if (qk_norm) {
        nk = 1.f / fmaxf(sqrtf(kk), kQkNormEps);
        nq = 1.f / fmaxf(sqrtf(qq), kQkNormEps);
    }
    const float scale = rsqrtf((float)D), b = beta[unit];
    const int j = 4 * c4;
    float vj[4];
    load_io4(v + (size_t)unit * D + j, vj);
    const float rkv[4] = {rk.x, rk.y, rk.z, rk.w}, rqv[4] = {rq.x, rq.y, rq.z, rq.w};
    float dl[4], ov[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float d = b * (vj[u] - rkv[u] * nk);
        ov[u] = scale * (rqv[u] * nq + kq * (nk * nq) * d);
        dl[u] = d * nk;  // the write k^ d^T = k (nk d)^T
    }
    if (rl == 0) store_io4(o + (size_t)unit * D + j, ov);

#pragma unroll
    for (int p = 0; p < P; ++p) {
        const float ki = s_k[rl + p * RL];
        float4 x = s[p];
        x.x += ki * dl[0]; x.y += ki * dl[1]; x.z += ki * dl[2]; x.w += ki * dl[3];
        __stcs(reinterpret_cast<float4 *>(S + (size_t)(rl + p * RL) * D) + c4, x);
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
