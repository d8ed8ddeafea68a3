// Internal declarations shared by the translation units of libkda.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Tokens per chunk of the chunkwise prefill.
constexpr int kChunk = 64;

// One chunk of one sequence: tokens [bos, bos + len) of sequence `seq`,
// the `idx`-th chunk of that sequence. seq < 0 marks an unused slot.
struct ChunkEntry {
    int seq;
    int bos;
    int len;
    int idx;
};

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Upper bound on chunk slots: exact for fixed-length batches, and for packed
// sequences sum_n ceil(len_n / 64) <= ceil(T / 64) + num_seqs.
inline long long max_chunk_slots(int B, int T, int num_seqs, bool packed) {
    const long long per = (T + kChunk - 1) / kChunk;
    return packed ? per + num_seqs : (long long)B * per;
}

// Grid over (head, chunk slot) with heads fastest; slots fold over y and z
// because gridDim.y is limited to 65535.
inline dim3 head_slot_grid(int H, long long slots) {
    const long long y = slots < 65535 ? slots : 65535;
    return dim3((unsigned)H, (unsigned)(y > 0 ? y : 1), (unsigned)((slots + y - 1) / (y > 0 ? y : 1)));
}

// Workspace layout: a 256-byte header whose first int is the device status
// word (0, or a kda_status a kernel left after a bounded wait gave up), then
// the chunk table, the per-sequence first-slot offsets, and the per-path
// regions.
constexpr size_t kWsHeader = 256;
// Workspace head: the status word, the chunk table, then seq_first_slot
// [num_seqs + 1] followed by seq_order [num_seqs] (the state passes' sequence
// order, longest first).
inline size_t table_bytes(long long slots, int num_seqs) {
    return kWsHeader + align_up((size_t)slots * sizeof(ChunkEntry), 256) +
           align_up((size_t)(2 * num_seqs + 1) * sizeof(int), 256);
}

// State-pass CTAs per (sequence, head) at most (d_v tiles), for the 1-D grids.
constexpr int kMaxStateTiles = 8;

// Segmented state pass (tensor-core path, fixed-length batches): the number
// of segments per sequence is capped so that chains x segments <= this bound,
// which also bounds the buffers the workspace reserves for it.
constexpr long long kSegChainBound = 32;

// Most segments a call with these sizes may use (1: the serial chain only).
inline int seg_limit(int B, int T, int H, int num_seqs, bool packed, bool tc_path) {
    if (packed || !tc_path || B <= 0 || H <= 0 || num_seqs != B) return 1;
    const long long chains = (long long)num_seqs * H;
    const long long nchunks = (T + kChunk - 1) / kChunk;
    long long p = kSegChainBound / chains;
    if (p > nchunks) p = nchunks;
    return p >= 2 ? (int)p : 1;
}

// Bytes of the segment buffers for `segs` segments: per (sequence, head,
// segment) the map [E | M] (d x 2d fp32) and the entering state (d x d fp32).
inline size_t seg_bytes(long long chains, int segs, int d) {
    return segs >= 2 ? (size_t)chains * segs * (size_t)d * d * 3 * sizeof(float) : 0;
}

// Validated kda_options, passed to the kernels by value.
struct Prologue {
    int decay;    // kda_decay: layout of g
    int gate;     // kda_gate: meaning of g's values
    float lower;  // KDA_GATE_BOUNDED: lower bound of log a
    int l2norm;   // normalise q and k per (token, head)
};
constexpr float kL2Eps = 1e-6f;  // x / sqrt(sum x^2 + kL2Eps)

// log a from a value of g under the gate transform (KDA_DECAY_NONE never calls
// this). log sigmoid(z) = min(z, 0) - log(1 + e^-|z|) avoids overflow; the
// fast exp/log are accurate to ~1e-7 absolute here, far inside the tolerances.
__device__ __forceinline__ float log_decay(float z, const Prologue &p) {
    if (p.gate == KDA_GATE_LOGSIGMOID) return fminf(z, 0.f) - __logf(1.f + __expf(-fabsf(z)));
    if (p.gate == KDA_GATE_BOUNDED) return p.lower * __fdividef(1.f, 1.f + __expf(-z));
    return z;
}
// a itself (= exp(log_decay)) where only the factor is needed: sigmoid(z) for
// the log-sigmoid gate without a logarithm.
__device__ __forceinline__ float decay_factor(float z, const Prologue &p) {
    if (p.gate == KDA_GATE_LOGSIGMOID) return __fdividef(1.f, 1.f + __expf(-z));
    if (p.gate == KDA_GATE_BOUNDED) return __expf(p.lower * __fdividef(1.f, 1.f + __expf(-z)));
    return expf(z);
}

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// The argument checks of kda_chunk_fwd_opt other than the workspace's, in the
// same order (host only; no CUDA call). KDA_OK when the call may proceed.
kda_status chunk_fwd_check(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, float scale, const float *init_state,
                           const int32_t *cu_seqlens, void *out, float *final_state, int B, int T,
                           int H, int dk, int dv, int num_seqs, kda_dtype dtype,
                           const kda_options *options);

// Fills `table` and `seq_first_slot` from cu_seqlens (device) or, when
// cu_seqlens is NULL, from num_seqs sequences of length T_fixed, and clears
// the status word.
cudaError_t launch_chunk_table(const int32_t *cu_seqlens, int num_seqs, int T_fixed, long long tokens,
                               long long slots, ChunkEntry *table, int *seq_first_slot,
                               int *status, cudaStream_t stream);

// fp32 SIMT prefill (any storage dtype; the reference-precision path).
size_t simt_region_bytes(int d);
cudaError_t launch_prefill_simt(const void *q, const void *k, const void *v, const float *g,
                                const float *beta, float scale, const float *init_state,
                                const int32_t *cu_seqlens, void *out, float *final_state,
                                int T_fixed, int H, int d, int num_seqs, kda_dtype dtype,
                                long long slots, const ChunkEntry *table,
                                const int *seq_first_slot, float *region, const int *status,
                                const Prologue &pro, cudaStream_t stream, cudaEvent_t *events);

// Output gate and RMS normalisation applied to the prefill's outputs (z NULL:
// none): out = w o / sqrt(mean(o^2) + eps) sigmoid(z) per (token, head).
struct GateParams {
    const void *z;   // gate logits [tokens][H][dv], storage dtype
    const float *w;  // [dv] or NULL
    float eps;
};

// Tensor-core prefill (bf16 storage, d = 128).
size_t tc_region_bytes();
cudaError_t launch_prefill_tc(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, float scale, const float *init_state,
                              const int32_t *cu_seqlens, void *out, float *final_state,
                              int T_fixed, long long tokens, int H, int num_seqs, long long slots,
                              const ChunkEntry *table, const int *seq_first_slot,
                              unsigned char *region, int *status, const Prologue &pro,
                              int segments, int seg_max, float *seg_ws, const GateParams &gate,
                              int fused, cudaStream_t stream, cudaEvent_t *events);

// Records events[i] (when non-NULL) on the stream: the prefill marks the
// start (0), the end of the chunk table (1), of the intra-chunk phase (2) and
// of the state pass (3).
inline cudaError_t mark(cudaEvent_t *events, int i, cudaStream_t stream) {
    return (events && events[i]) ? cudaEventRecord(events[i], stream) : cudaSuccess;
}

// Output gate + RMS normalisation over rows of dv values (rows = tokens * H).
cudaError_t launch_output_gate_rmsnorm(const void *o, const void *z, const float *w, float eps,
                                       void *out, long long rows, int dv, kda_dtype dtype,
                                       cudaStream_t stream);

// Decode step.
cudaError_t launch_decode(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, float scale, float *state, void *out, int N, int H,
                          int d, kda_dtype dtype, const Prologue &pro, cudaStream_t stream);

}  // namespace kda
