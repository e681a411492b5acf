// selftest.cu -- the library's diagnostics (the pages have no counterpart):
//  kda_selftest_bounded_wait  exercises the kernels' failure path on the device without a
//      fault: a wait on an mbarrier that nothing ever arrives on must give up after its
//      limit, record KDA_DEVICE_ERR_TIMEOUT in the status word and return, leaving the
//      context usable;
//  kda_diag_tensor_phases     measures the prefill kernels' tensor-core product groups on
//      their own (the kernel is in prefill_split.cu, beside the routines it reuses).
#include "common.cuh"
#include "sm100_ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

// One CTA: thread 0 waits (sleeping) and warp 1's lane 0 waits (polling) on a
// barrier that expects one arrival that never comes.
__global__ void bounded_wait_selftest_kernel(uint32_t *status, uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    bool gave_up = false;
    if (threadIdx.x == 0) gave_up = !mbar_wait_ns(&bar, 0, limit_ns);
    if (threadIdx.x == 32) gave_up = !mbar_wait_spin_ns(&bar, 0, limit_ns);
    if (__syncthreads_or(gave_up) && threadIdx.x == 0) atomicOr(status, DEV_ERR_TIMEOUT);
}

}  // namespace
}  // namespace kda

extern "C" kda_status_t kda_selftest_bounded_wait(void *workspace, uint64_t limit_ns, void *stream)
{
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KDA_ERR_INVALID_ARG;
    if (limit_ns == 0 || limit_ns > 1000000000ull) return KDA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess) return KDA_ERR_CUDA;
    kda::bounded_wait_selftest_kernel<<<1, 64, 0, s>>>(static_cast<uint32_t *>(workspace), limit_ns);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

extern "C" kda_status_t kda_diag_tensor_phases(int32_t pass, int32_t reps, void *workspace, void *stream,
                                               double *tflops)
{
    if (pass < 0 || pass > 2 || reps < 1 || reps > (1 << 20) || !tflops) return KDA_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KDA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess) return KDA_ERR_CUDA;
    double t = 0.0;
    if (kda::diag_tensor_phases(pass, reps, static_cast<uint32_t *>(workspace), s, &t) != cudaSuccess)
        return KDA_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (word) return KDA_ERR_TIMEOUT;
    *tflops = t;
    return KDA_OK;
}
