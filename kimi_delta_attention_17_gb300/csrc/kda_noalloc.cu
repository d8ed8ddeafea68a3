// kda_chunk_fwd_noalloc: the chunkwise prefill for callers that cannot
// allocate device memory themselves (code running where cudaMalloc is
// forbidden or unavailable, e.g. inside a host callback, under an allocator
// that must not be re-entered, or in an embedding that owns all memory
// statically). Its scratch lives in one file-scope device array that the
// module carries; nothing here calls cudaMalloc, cudaFree or any allocating
// library routine.
#include <atomic>

#include "kda_internal.cuh"

namespace {

// The scratch array. Every GPU that loads this library holds these bytes
// until the process exits. In host code `g_noalloc_scratch` is only a
// host-side stand-in for the symbol: its device address is obtained with
// cudaGetSymbolAddress below and only that address is handed to kernels.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_addr[kMaxDevices];

// Resolves (once per device, with that device current) the device address of
// the scratch array.
cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void *p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess) return err;
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" kda_status kda_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                            const float *g, const float *beta, float scale,
                                            const float *init_state, const int32_t *cu_seqlens,
                                            void *out, float *final_state, int B, int T, int H,
                                            int dk, int dv, int num_seqs, kda_dtype dtype,
                                            cudaStream_t stream) {
    const size_t need = kda_chunk_fwd_workspace_size(B, T, H, dk, dv, num_seqs, dtype);
    if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;
    if (need == 0) {
        // Invalid or unsupported sizes: let the regular entry point report
        // which (it returns before touching the device for these).
        return kda_chunk_fwd(q, k, v, g, beta, scale, init_state, cu_seqlens, out, final_state, B,
                             T, H, dk, dv, num_seqs, dtype, nullptr, 0, stream);
    }
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return KDA_ERR_CUDA;
    return kda_chunk_fwd(q, k, v, g, beta, scale, init_state, cu_seqlens, out, final_state, B, T,
                         H, dk, dv, num_seqs, dtype, scratch, (size_t)KDA_NOALLOC_SCRATCH_BYTES,
                         stream);
}
