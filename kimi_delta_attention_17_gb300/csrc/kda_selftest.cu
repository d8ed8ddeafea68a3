// kda_selftest_wait_timeout: checks the device-side timeout reporting without
// faulting, trapping or hanging anything. One CTA initialises an mbarrier that
// nothing ever arrives at and waits on it with the kernels' bounded wait (a
// short limit here); the wait gives up, the kernel records KDA_ERR_TIMEOUT in
// the caller's status word exactly as the prefill kernels do in the workspace
// status word, and returns. The context stays usable.
#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

__global__ void __launch_bounds__(32) selftest_timeout(int *status, unsigned limit) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        tc::mbar_fence_init();
    }
    __syncwarp();
    // Nothing arrives: phase 0 never completes.
    const bool ok = tc::mbar_wait(&bar, 0, limit);
    if (threadIdx.x == 0) atomicExch(status, ok ? (int)KDA_OK : (int)KDA_ERR_TIMEOUT);
}

}  // namespace
}  // namespace kda

extern "C" kda_status kda_selftest_wait_timeout(int *status, unsigned int limit,
                                                cudaStream_t stream) {
    if (!status || (reinterpret_cast<uintptr_t>(status) & 3u) != 0 || limit == 0 ||
        limit > (1u << 22))
        return KDA_ERR_INVALID_ARGUMENT;
    kda::selftest_timeout<<<1, 32, 0, stream>>>(status, limit);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
