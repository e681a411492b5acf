// prefill_host.cu -- kda_prefill_host: the prefill from (page-locked) host buffers, with the
// host->device copies of later tokens, the prefill of earlier ones and the device->host copy
// of their outputs overlapped.
//
// The tokens are cut into up to four segments at chunk boundaries of the sequence they fall
// in (64-token multiples from that sequence's start), so every chunk and every serial state
// step is the one kda_prefill would run: the results are bit for bit those of one kda_prefill
// call.  Each sequence's state lives in a device pool entry of its own (its initial state,
// or zero); every segment runs kda_prefill_slots on its tokens with each sequence reading and
// writing its own entry, so a sequence cut by a boundary continues from where the segment
// before left it.  Built on the public calls of this library; no kernel of its own except
// the one that keeps the segments' device-side error words.
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "common.cuh"

namespace {

constexpr int kMaxSegments = 4;
constexpr int64_t kMinSegmentTokens = 1024;  // shorter prompts are not cut
constexpr int kMaxDevices = 64;

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// Segment boundaries bounds[0] = 0 < ... < bounds[n] = total, each one at a 64-token multiple
// from the start of the sequence it falls in.  cu: host [num_seqs + 1] (NULL: one sequence).
// The host->device copies are the critical path and run back to back; what follows the last
// one (that segment's prefill, the copies of its outputs and of the final states) is the only
// exposed part, so the last segment gets 1/16 of the tokens and the others share the rest.
int plan_segments(const int32_t *cu, int num_seqs, int64_t total, int64_t *bounds)
{
    int n = 0;
    bounds[n++] = 0;
    int k = (int)(total / kMinSegmentTokens);
    if (k > kMaxSegments) k = kMaxSegments;
    for (int s = 1; s < k; ++s) {
        const int64_t t = total * 15 * s / (16 * (k - 1));
        int64_t start = 0;  // start of the sequence holding token t
        if (cu) {
            int lo = 0, hi = num_seqs;  // cu[lo] <= t < cu[lo + 1]
            while (hi - lo > 1) {
                const int mid = (lo + hi) / 2;
                if (cu[mid] <= t) lo = mid; else hi = mid;
            }
            start = cu[lo];
        }
        const int64_t b = start + (t - start) / kda::kChunk * kda::kChunk;
        if (b > bounds[n - 1] && b < total) bounds[n++] = b;
    }
    bounds[n] = total;
    return n;
}

struct Segment {
    int64_t a, b;        // tokens [a, b)
    int first, count;    // sequences first .. first + count - 1 (the non-empty ones that meet it)
    size_t cu_off;       // its local cu_seqlens, then its slot list, in the plan array (int32 units)
};

struct Plan {
    std::vector<Segment> seg;
    std::vector<int32_t> ints;  // local cu_seqlens and slot lists of every segment
    size_t off_pool, off_ints, off_in[2], off_out[2], off_ws, bytes;
    size_t in_q, in_la, in_beta;  // offsets inside one input staging buffer (q, k, v back to back)
    size_t ws_bytes;
    int64_t seg_max;
};

bool make_plan(const int32_t *cu, int num_seqs, int64_t total, int H, int d, kda_dtype_t dtype, Plan &p)
{
    int64_t bounds[kMaxSegments + 1];
    const int ns = total > 0 ? plan_segments(cu, num_seqs, total, bounds) : 0;
    auto seq_start = [&](int n) -> int64_t { return cu ? cu[n] : 0; };
    auto seq_end = [&](int n) -> int64_t { return cu ? cu[n + 1] : total; };
    p.seg.clear();
    p.ints.clear();
    p.seg_max = 0;
    p.ws_bytes = 0;
    int n0 = 0;
    for (int s = 0; s < ns; ++s) {
        Segment g{bounds[s], bounds[s + 1], 0, 0, p.ints.size()};
        while (n0 < num_seqs && seq_end(n0) <= g.a) ++n0;  // sequences wholly before the segment
        g.first = n0;
        std::vector<int32_t> lcu{0}, slots;
        for (int n = n0; n < num_seqs && seq_start(n) < g.b; ++n) {
            if (seq_end(n) <= seq_start(n)) continue;  // empty: its entry keeps its initial state
            const int64_t e = seq_end(n) < g.b ? seq_end(n) : g.b;
            lcu.push_back((int32_t)(e - g.a));
            slots.push_back(n);
        }
        g.count = (int)slots.size();
        if (g.count == 0) return false;  // every token belongs to a non-empty sequence
        p.ints.insert(p.ints.end(), lcu.begin(), lcu.end());
        p.ints.insert(p.ints.end(), slots.begin(), slots.end());
        const int64_t len = g.b - g.a;
        if (len > p.seg_max) p.seg_max = len;
        const size_t w = kda_prefill_workspace_size(g.count, len, H, d, d, dtype);
        if (w == 0) return false;
        if (w > p.ws_bytes) p.ws_bytes = w;
        p.seg.push_back(g);
    }
    const size_t esz = dtype == KDA_DTYPE_BF16 ? 2 : 4;
    const size_t row = (size_t)p.seg_max * H * d;
    p.in_q = 0;
    p.in_la = round256(3 * row * esz);
    p.in_beta = p.in_la + round256(row * 4);
    const size_t in_bytes = p.in_beta + round256((size_t)p.seg_max * H * 4);
    size_t off = 0;
    p.off_pool = off = 256;  // bytes 0..255: the error word of the whole call
    off += round256((size_t)num_seqs * H * d * d * 4);
    p.off_ints = off;
    off += round256(p.ints.size() * 4);
    for (int i = 0; i < 2; ++i) { p.off_in[i] = off; off += in_bytes; }
    for (int i = 0; i < 2; ++i) { p.off_out[i] = off; off += round256(row * esz); }
    p.off_ws = off;
    off += p.ws_bytes;
    p.bytes = off;
    return true;
}

// The error word of the whole call collects each segment's (the next segment clears it).
__global__ void or_status_kernel(uint32_t *acc, const uint32_t *seg) { *acc |= *seg; }

// Streams and events of the pipeline, created once per device.
struct DeviceQueues {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t ev[1 + 3 * kMaxSegments] = {};
    bool ready = false;
};
DeviceQueues g_queues[kMaxDevices];
std::mutex g_queue_mutex;

bool queues_for(int dev, DeviceQueues *&q)
{
    if (dev < 0 || dev >= kMaxDevices) return false;
    q = &g_queues[dev];
    if (q->ready) return true;
    if (cudaStreamCreateWithFlags(&q->in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&q->out, cudaStreamNonBlocking) != cudaSuccess)
        return false;
    for (auto &e : q->ev)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return false;
    q->ready = true;
    return true;
}

}  // namespace

extern "C" {

int32_t kda_prefill_host_segments(const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                                  int64_t *bounds, int32_t max_bounds)
{
    if (num_seqs < 0 || total_tokens < 0 || !bounds || max_bounds < kMaxSegments + 1) return -1;
    if (!cu_seqlens && num_seqs != 1) return -1;
    if (total_tokens == 0) return 0;
    return plan_segments(cu_seqlens, num_seqs, total_tokens, bounds);
}

size_t kda_prefill_host_buffer_size(const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                                    int32_t num_heads, int32_t d_k, int32_t d_v, kda_dtype_t dtype)
{
    if (num_seqs <= 0 || total_tokens < 0 || num_heads <= 0 || d_k != d_v || (!cu_seqlens && num_seqs != 1))
        return 0;
    Plan p;
    if (!make_plan(cu_seqlens, num_seqs, total_tokens, num_heads, d_k, dtype, p)) return 0;
    return p.bytes;
}

kda_status_t kda_prefill_host(const void *q, const void *k, const void *v, const float *log_alpha,
                              const float *beta, const int32_t *cu_seqlens, int32_t num_seqs,
                              int64_t total_tokens, int32_t num_heads, int32_t d_k, int32_t d_v,
                              kda_dtype_t dtype, const float *init_state, void *o, float *final_state,
                              void *device_buffer, size_t device_bytes, void *stream, uint32_t flags)
{
    if (num_seqs <= 0 || total_tokens < 0 || num_heads <= 0) return KDA_ERR_INVALID_ARG;
    if (!cu_seqlens && num_seqs != 1) return KDA_ERR_INVALID_ARG;
    if (dtype != KDA_DTYPE_BF16 && dtype != KDA_DTYPE_F32) return KDA_ERR_INVALID_ARG;
    if (d_k != d_v || (d_k != 64 && d_k != 128)) return KDA_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || num_heads > 65535) return KDA_ERR_UNSUPPORTED;
    if (flags & ~(uint32_t)(KDA_FLAG_SCALAR_GATE | KDA_FLAG_QK_L2NORM | KDA_FLAG_NO_SEQ_SPLIT | KDA_FLAG_NO_STREAM |
                            KDA_FLAG_STREAM) ||
        (flags & (KDA_FLAG_STREAM | KDA_FLAG_NO_STREAM)) == (KDA_FLAG_STREAM | KDA_FLAG_NO_STREAM))
        return KDA_ERR_INVALID_ARG;
    if (flags & KDA_FLAG_SCALAR_GATE) return KDA_ERR_UNSUPPORTED;  // log_alpha copies are per channel
    if (total_tokens > 0 && (!q || !k || !v || !log_alpha || !beta)) return KDA_ERR_INVALID_ARG;
    if (!final_state || !device_buffer || (reinterpret_cast<uintptr_t>(device_buffer) & 255u) != 0)
        return KDA_ERR_INVALID_ARG;
    if (cu_seqlens) {  // the host copy is what the plan is made from: check it here
        if (cu_seqlens[0] != 0 || cu_seqlens[num_seqs] != total_tokens) return KDA_ERR_INVALID_ARG;
        for (int n = 0; n < num_seqs; ++n)
            if (cu_seqlens[n + 1] < cu_seqlens[n]) return KDA_ERR_INVALID_ARG;
    }
    Plan p;
    if (!make_plan(cu_seqlens, num_seqs, total_tokens, num_heads, d_k, dtype, p)) return KDA_ERR_UNSUPPORTED;
    if (device_bytes < p.bytes) return KDA_ERR_INVALID_ARG;

    const int H = num_heads, d = d_k;
    const size_t esz = dtype == KDA_DTYPE_BF16 ? 2 : 4;
    const size_t state_bytes = (size_t)num_seqs * H * d * d * 4;
    char *dev = static_cast<char *>(device_buffer);
    float *pool = reinterpret_cast<float *>(dev + p.off_pool);
    int32_t *ints = reinterpret_cast<int32_t *>(dev + p.off_ints);
    uint32_t *word = static_cast<uint32_t *>(device_buffer);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);

    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_queue_mutex);
    DeviceQueues *qs = nullptr;
    if (!queues_for(device, qs)) return KDA_ERR_CUDA;
    cudaEvent_t ev_start = qs->ev[0], *ev_in = qs->ev + 1, *ev_comp = ev_in + kMaxSegments,
                *ev_out = ev_comp + kMaxSegments;
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };

    // the pool starts as the initial states (or zero); the plan goes up once
    if (!ok(cudaMemsetAsync(word, 0, sizeof(uint32_t), cs))) return KDA_ERR_CUDA;
    if (!ok(init_state ? cudaMemcpyAsync(pool, init_state, state_bytes, cudaMemcpyHostToDevice, cs)
                       : cudaMemsetAsync(pool, 0, state_bytes, cs)))
        return KDA_ERR_CUDA;
    if (!p.ints.empty() &&
        !ok(cudaMemcpyAsync(ints, p.ints.data(), p.ints.size() * 4, cudaMemcpyHostToDevice, cs)))
        return KDA_ERR_CUDA;
    if (!ok(cudaEventRecord(ev_start, cs)) || !ok(cudaStreamWaitEvent(qs->in, ev_start, 0)) ||
        !ok(cudaStreamWaitEvent(qs->out, ev_start, 0)))
        return KDA_ERR_CUDA;

    const char *src_q = static_cast<const char *>(q), *src_k = static_cast<const char *>(k),
               *src_v = static_cast<const char *>(v);
    for (size_t s = 0; s < p.seg.size(); ++s) {
        const Segment &g = p.seg[s];
        const int buf = (int)(s & 1);
        const int64_t len = g.b - g.a;
        const size_t tok = (size_t)H * d;  // elements per token of q, k, v, log_alpha
        char *in = dev + p.off_in[buf];
        char *out = dev + p.off_out[buf];
        // inputs of segment s, once segment s - 2 has finished reading this buffer
        if (s >= 2 && !ok(cudaStreamWaitEvent(qs->in, ev_comp[s - 2], 0))) return KDA_ERR_CUDA;
        const size_t nb = (size_t)len * tok * esz;
        if (!ok(cudaMemcpyAsync(in + p.in_q, src_q + (size_t)g.a * tok * esz, nb, cudaMemcpyHostToDevice, qs->in)) ||
            !ok(cudaMemcpyAsync(in + p.in_q + nb, src_k + (size_t)g.a * tok * esz, nb, cudaMemcpyHostToDevice, qs->in)) ||
            !ok(cudaMemcpyAsync(in + p.in_q + 2 * nb, src_v + (size_t)g.a * tok * esz, nb, cudaMemcpyHostToDevice,
                                qs->in)) ||
            !ok(cudaMemcpyAsync(in + p.in_la, log_alpha + (size_t)g.a * tok, (size_t)len * tok * 4,
                                cudaMemcpyHostToDevice, qs->in)) ||
            !ok(cudaMemcpyAsync(in + p.in_beta, beta + (size_t)g.a * H, (size_t)len * H * 4, cudaMemcpyHostToDevice,
                                qs->in)) ||
            !ok(cudaEventRecord(ev_in[s], qs->in)))
            return KDA_ERR_CUDA;
        // the prefill of segment s, once its inputs are in and segment s - 2's outputs are out
        if (!ok(cudaStreamWaitEvent(cs, ev_in[s], 0))) return KDA_ERR_CUDA;
        if (s >= 2 && !ok(cudaStreamWaitEvent(cs, ev_out[s - 2], 0))) return KDA_ERR_CUDA;
        const int32_t *lcu = ints + g.cu_off, *slots = lcu + g.count + 1;
        kda_status_t st = kda_prefill_slots(in + p.in_q, in + p.in_q + nb, in + p.in_q + 2 * nb,
                                            reinterpret_cast<const float *>(in + p.in_la),
                                            reinterpret_cast<const float *>(in + p.in_beta), lcu, g.count, len, H, d,
                                            d, dtype, pool, num_seqs, slots, slots, o ? out : nullptr,
                                            dev + p.off_ws, p.ws_bytes, cs, flags);
        if (st != KDA_OK) return st;
        or_status_kernel<<<1, 1, 0, cs>>>(word, reinterpret_cast<const uint32_t *>(dev + p.off_ws));
        if (!ok(cudaGetLastError()) || !ok(cudaEventRecord(ev_comp[s], cs))) return KDA_ERR_CUDA;
        // its outputs back to the host
        if (!ok(cudaStreamWaitEvent(qs->out, ev_comp[s], 0))) return KDA_ERR_CUDA;
        if (o && !ok(cudaMemcpyAsync(static_cast<char *>(o) + (size_t)g.a * H * d * esz, out, (size_t)len * H * d * esz,
                                     cudaMemcpyDeviceToHost, qs->out)))
            return KDA_ERR_CUDA;
        if (!ok(cudaEventRecord(ev_out[s], qs->out))) return KDA_ERR_CUDA;
    }
    // the final states, after the last segment; the caller's stream then covers every copy
    if (!p.seg.empty() && !ok(cudaStreamWaitEvent(cs, ev_out[p.seg.size() - 1], 0))) return KDA_ERR_CUDA;
    if (!ok(cudaMemcpyAsync(final_state, pool, state_bytes, cudaMemcpyDeviceToHost, cs))) return KDA_ERR_CUDA;
    return KDA_OK;
}

}  // extern "C"
