// kda_chunk_fwd_noalloc: the chunkwise prefill for callers that cannot
// allocate device memory themselves (code running where cudaMalloc is
// forbidden or unavailable, e.g. inside a host callback, under an allocator
// that must not be re-entered, or in an embedding that owns all memory
// statically). Its scratch lives in one file-scope device array that the
// module carries; nothing here calls cudaMalloc, cudaFree or any allocating
// library routine.
#include "kda_internal.cuh"

namespace {

// The scratch array. Every GPU that loads this library holds these bytes
// until the process exits. In host code `g_noalloc_scratch` is only a
// host-side stand-in for the symbol: its device address is obtained with
// cudaGetSymbolAddress below and only that address is handed to kernels.
static __device__ __align__(256) unsigned char g_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

// The device address of the scratch array in the current context. It is
// resolved on every call rather than cached: a context created after a
// cudaDeviceReset (or any other context on the same device) gets its own copy
// of the module, and a cached address would point into the old one. The
// lookup allocates nothing; the first call in a context also loads the
// library's module there.
cudaError_t scratch_address(void **out) {
    void *p = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess) return err;
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
    // The arguments first, exactly as kda_chunk_fwd checks them, so that both
    // entry points report the same error for the same bad call; then the
    // capacity of the fixed scratch.
    const kda_status chk = kda::chunk_fwd_check(q, k, v, g, beta, scale, init_state, cu_seqlens,
                                                out, final_state, B, T, H, dk, dv, num_seqs, dtype,
                                                nullptr);
    if (chk != KDA_OK) return chk;
    const size_t need = kda_chunk_fwd_workspace_size(B, T, H, dk, dv, num_seqs, dtype);
    if (need == 0 || need > (size_t)KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return KDA_ERR_CUDA;
    return kda_chunk_fwd(q, k, v, g, beta, scale, init_state, cu_seqlens, out, final_state, B, T,
                         H, dk, dv, num_seqs, dtype, scratch, (size_t)KDA_NOALLOC_SCRATCH_BYTES,
                         stream);
}

extern "C" kda_status kda_chunk_fwd_noalloc_status(int *status, cudaStream_t stream) {
    if (!status) return KDA_ERR_INVALID_ARGUMENT;
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return KDA_ERR_CUDA;
    // The status word is the first int of the scratch (the workspace layout of
    // kda_chunk_fwd): one 4-byte copy on the caller's stream, nothing allocated.
    return cudaMemcpyAsync(status, scratch, sizeof(int), cudaMemcpyDeviceToHost, stream) ==
                   cudaSuccess
               ? KDA_OK
               : KDA_ERR_CUDA;
}
