// prefill_no_alloc.cu -- kda_prefill for callers that cannot allocate device memory.
//
// kda_prefill needs a small device workspace (an error word and the sequence
// schedule).  Some callers cannot provide one: a serving runtime that hands out
// all GPU memory from a pool sized at start-up and refuses allocations after
// that, or a latency-critical path that must not pay for cudaMalloc (which can
// synchronise the device).  This entry point gives them the same prefill with
// the workspace placed in a fixed array that lives inside libkda on every GPU
// that loads the library, until the process exits.  It calls no cudaMalloc,
// cudaFree or allocating library routine.
#include <mutex>

#include "common.cuh"

namespace {

// Covers kda_prefill_workspace_size(KDA_NO_ALLOC_MAX_SEQS, ...): the 256-byte
// header plus the sequence order rounded up to whole 256-byte blocks.
constexpr size_t kScratchBytes = KDA_NO_ALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes >= kda::kWorkspaceHeader +
                                   ((size_t)KDA_NO_ALLOC_MAX_SEQS * sizeof(int32_t) + 1 + 255) /
                                       256 * 256,
              "scratch smaller than the prefill workspace at the maximum sequence count");

// The shared scratch.  In host code this name is only a host-side stand-in for
// the symbol, never a device address: kernels get the address looked up below.
static __device__ __align__(256) unsigned char g_prefill_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];  // device address of g_prefill_scratch, per device
std::mutex g_scratch_mutex;

// Device address of the scratch on the current device, looked up once per device
// (with that device current) and cached.  The cache outlives a cudaDeviceReset, after
// which the module, and so the array, may be loaded at another address: a process
// that resets a device must not call kda_prefill_no_alloc on it again.
kda_status_t scratch_on_current_device(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> guard(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess || !p) return KDA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" kda_status_t kda_prefill_no_alloc(
    const void *q, const void *k, const void *v, const float *log_alpha, const float *beta,
    const int32_t *cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t num_heads,
    int32_t d_k, int32_t d_v, kda_dtype_t dtype, const float *init_state, void *o,
    float *final_state, uint32_t *device_errors, void *stream)
{
    if (num_seqs > KDA_NO_ALLOC_MAX_SEQS) return KDA_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    kda_status_t st = scratch_on_current_device(&scratch);
    if (st != KDA_OK) return st;
    // Same validation and kernels as kda_prefill; its schedule kernel rewrites the
    // error word and the sequence order at the start of every call, so nothing is
    // left over from the previous call that used the scratch.
    st = kda_prefill(q, k, v, log_alpha, beta, cu_seqlens, num_seqs, total_tokens, num_heads, d_k,
                     d_v, dtype, init_state, o, final_state, scratch, kScratchBytes, stream);
    if (st != KDA_OK) return st;
    if (!device_errors) return KDA_OK;
    cudaStream_t strm = static_cast<cudaStream_t>(stream);
    // With no sequences kda_prefill enqueues no kernel, so the scratch still holds the
    // error word of whichever call used it last: report this call's (none) instead.
    const cudaError_t e =
        num_seqs == 0 ? cudaMemsetAsync(device_errors, 0, sizeof(uint32_t), strm)
                      : cudaMemcpyAsync(device_errors, scratch, sizeof(uint32_t),
                                        cudaMemcpyDeviceToDevice, strm);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
