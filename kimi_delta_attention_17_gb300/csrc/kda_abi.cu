// The C ABI of libkda.so: argument validation, workspace sizing, the chunk
// table, and dispatch to the prefill and decode kernels. Every argument check
// happens here, on the host, before any CUDA call.
#include <math.h>

#include "kda_internal.cuh"

namespace kda {
namespace {

// Builds the chunk table on the device (cu_seqlens lives there; reading it on
// the host would need a synchronising copy). One CTA: an exclusive scan of
// per-sequence chunk counts, then each sequence writes its own slots; the
// slots past the last used one are marked unused. It also writes the order in
// which the state passes take the sequences: each state-pass CTA walks one
// sequence's chunks in series, so a mixed-length batch finishes soonest when
// the longest chains are dispatched first (longest-processing-time order;
// ties by index). Up to kOrderMaxSeqs packed sequences are ranked, by a
// count over shared memory; beyond that, and for fixed-length batches, the
// order is the identity. Packed offsets are checked first (cu_seqlens[0] = 0,
// non-decreasing, cu_seqlens[num_seqs] = tokens): on a violation the status
// word reads KDA_ERR_INVALID_ARGUMENT, the table is empty and the state
// passes, which read the status word first, do nothing.
constexpr int kTableThreads = 1024;
constexpr int kOrderMaxSeqs = 1024;

__global__ void __launch_bounds__(kTableThreads)
chunk_table_kernel(const int32_t *__restrict__ cu_seqlens, int num_seqs, int T_fixed,
                   long long tokens, long long slots, ChunkEntry *__restrict__ table,
                   int *__restrict__ seq_first_slot, int *__restrict__ seq_order,
                   int *__restrict__ status) {
    __shared__ int part[kTableThreads];
    __shared__ int nch[kOrderMaxSeqs];
    const int tid = threadIdx.x;
    if (tid == 0) *status = 0;
    // Sequences [lo, hi) belong to this thread.
    const int per = (num_seqs + kTableThreads - 1) / kTableThreads;
    const int lo = min(num_seqs, tid * per), hi = min(num_seqs, lo + per);
    bool bad = false;
    if (cu_seqlens) {
        for (int n = lo; n < hi; ++n) bad |= cu_seqlens[n + 1] < cu_seqlens[n];
        if (tid == 0) bad |= cu_seqlens[0] != 0 || (long long)cu_seqlens[num_seqs] != tokens;
    }
    if (__syncthreads_or(bad)) {
        if (tid == 0) {
            *status = (int)KDA_ERR_INVALID_ARGUMENT;
            seq_first_slot[num_seqs] = 0;  // no used slot: phase 1 has no item
        }
        for (int n = tid; n < num_seqs; n += kTableThreads) {
            seq_first_slot[n] = 0;
            seq_order[n] = n;
        }
        for (long long s = tid; s < slots; s += kTableThreads) {
            ChunkEntry e;
            e.seq = -1;
            e.bos = 0;
            e.len = 0;
            e.idx = 0;
            table[s] = e;
        }
        return;
    }
    auto seq_bounds = [&](int n, int &bos, int &len) {
        if (cu_seqlens) {
            bos = cu_seqlens[n];
            len = cu_seqlens[n + 1] - bos;
        } else {
            bos = n * T_fixed;
            len = T_fixed;
        }
    };
    const bool rank = cu_seqlens != nullptr && num_seqs <= kOrderMaxSeqs;
    int mine = 0;
    for (int n = lo; n < hi; ++n) {
        int bos, len;
        seq_bounds(n, bos, len);
        const int c = (len + kChunk - 1) / kChunk;
        mine += c;
        if (rank) nch[n] = c;
    }
    part[tid] = mine;
    __syncthreads();
    for (int n = lo; n < hi; ++n) {
        int r = n;
        if (rank) {
            const int c = nch[n];
            r = 0;
            for (int m = 0; m < num_seqs; ++m) r += nch[m] > c || (nch[m] == c && m < n);
        }
        seq_order[r] = n;
    }
    // Inclusive Hillis-Steele scan over the per-thread totals.
    for (int off = 1; off < kTableThreads; off <<= 1) {
        const int add = tid >= off ? part[tid - off] : 0;
        __syncthreads();
        part[tid] += add;
        __syncthreads();
    }
    int slot = part[tid] - mine;
    for (int n = lo; n < hi; ++n) {
        int bos, len;
        seq_bounds(n, bos, len);
        seq_first_slot[n] = slot;
        slot += (len + kChunk - 1) / kChunk;
    }
    const int used = part[kTableThreads - 1];
    if (tid == 0) seq_first_slot[num_seqs] = used;
    __syncthreads();  // every sequence's first slot is in place
    // The entries, spread over all threads (one sequence of many chunks would
    // otherwise be one thread's serial loop). Slot s belongs to the last
    // sequence whose first slot is <= s (an empty sequence shares its first
    // slot with the next one, which is later).
    const int nch_fixed = (T_fixed + kChunk - 1) / kChunk;
    for (long long s = tid; s < slots; s += kTableThreads) {
        ChunkEntry e;
        e.seq = -1;
        e.bos = 0;
        e.len = 0;
        e.idx = 0;
        if (s < used) {
            int n;
            if (!cu_seqlens) {
                n = (int)(s / nch_fixed);
            } else {
                int a = 0, b = num_seqs - 1;  // seq_first_slot[a] <= s holds throughout
                while (a < b) {
                    const int m = (a + b + 1) >> 1;
                    if (seq_first_slot[m] <= s) a = m; else b = m - 1;
                }
                n = a;
            }
            int bos, len;
            seq_bounds(n, bos, len);
            const int c = (int)(s - seq_first_slot[n]);
            e.seq = n;
            e.bos = bos + c * kChunk;
            e.len = min(kChunk, len - c * kChunk);
            e.idx = c;
        }
        table[s] = e;
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dims_ok(int dk, int dv) { return dk == dv && (dk == 64 || dk == 128); }

// The tensor-core path serves bf16 storage with d = 128; the fp32 SIMT path
// serves everything else (fp32 storage, and d = 64).
bool use_tc(int d, kda_dtype dtype) { return dtype == KDA_DTYPE_BF16 && d == 128; }

// Bytes of the per-path region that follows the chunk table.
size_t path_region_bytes(long long slots, int H, int d, kda_dtype dtype) {
    return (size_t)slots * (size_t)H * (use_tc(d, dtype) ? tc_region_bytes() : simt_region_bytes(d));
}

}  // namespace

cudaError_t launch_chunk_table(const int32_t *cu_seqlens, int num_seqs, int T_fixed, long long tokens,
                               long long slots, ChunkEntry *table, int *seq_first_slot,
                               int *status, cudaStream_t stream) {
    chunk_table_kernel<<<1, kTableThreads, 0, stream>>>(cu_seqlens, num_seqs, T_fixed, tokens, slots,
                                                        table, seq_first_slot,
                                                        seq_first_slot + num_seqs + 1, status);
    return cudaGetLastError();
}

}  // namespace kda

using namespace kda;

extern "C" const char *kda_status_string(kda_status status) {
    switch (status) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARGUMENT: return "KDA_ERR_INVALID_ARGUMENT";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
    }
    return "KDA_ERR_UNKNOWN";
}

extern "C" size_t kda_chunk_fwd_workspace_size(int B, int T, int H, int dk, int dv, int num_seqs,
                                               kda_dtype dtype) {
    if (B <= 0 || T < 0 || H <= 0 || num_seqs <= 0) return 0;
    if (!dims_ok(dk, dv)) return 0;
    if (dtype != KDA_DTYPE_F32 && dtype != KDA_DTYPE_BF16) return 0;
    const bool packed = num_seqs != B;
    if (packed && B != 1) return 0;
    const long long slots = max_chunk_slots(B, T, num_seqs, packed);
    const int segs = seg_limit(B, T, H, num_seqs, packed, use_tc(dk, dtype));
    return table_bytes(slots, num_seqs) +
           align_up(path_region_bytes(slots, H, dk, dtype), 256) +
           seg_bytes((long long)num_seqs * H, segs, dk);
}

namespace {

// Checks kda_options and turns them into the kernels' Prologue (NULL: the
// defaults of kda_chunk_fwd / kda_decode_step).
bool make_prologue(const kda_options *o, Prologue *p) {
    *p = Prologue{KDA_DECAY_CHANNEL, KDA_GATE_LOG, 0.f, 0};
    if (!o) return true;
    if (o->decay != KDA_DECAY_CHANNEL && o->decay != KDA_DECAY_SCALAR && o->decay != KDA_DECAY_NONE)
        return false;
    if (o->gate != KDA_GATE_LOG && o->gate != KDA_GATE_LOGSIGMOID && o->gate != KDA_GATE_BOUNDED)
        return false;
    if (o->gate == KDA_GATE_BOUNDED && !(o->gate_lower >= -10.f && o->gate_lower < 0.f)) return false;
    if (o->segments < 0) return false;
    if (o->fused < -1 || o->fused > 1) return false;
    *p = Prologue{(int)o->decay, (int)o->gate, o->gate == KDA_GATE_BOUNDED ? o->gate_lower : 0.f,
                  o->l2norm_qk ? 1 : 0};
    return true;
}

// g is required unless there is no decay; per-channel g is 16-byte aligned,
// per-head g 4-byte aligned.
bool g_ok(const float *g, const Prologue &p, bool required) {
    if (p.decay == KDA_DECAY_NONE) return true;
    if (required && !g) return false;
    const uintptr_t a = reinterpret_cast<uintptr_t>(g);
    return (a & (p.decay == KDA_DECAY_CHANNEL ? 15u : 3u)) == 0;
}

}  // namespace

// Every check of a prefill call's arguments except those of the workspace, in
// the order kda_chunk_fwd applies them (host only, no CUDA call).
kda_status kda::chunk_fwd_check(const void *q, const void *k, const void *v, const float *g,
                                const float *beta, float scale, const float *init_state,
                                const int32_t *cu_seqlens, void *out, float *final_state, int B,
                                int T, int H, int dk, int dv, int num_seqs, kda_dtype dtype,
                                const kda_options *options) {
    Prologue pro;
    if (!make_prologue(options, &pro)) return KDA_ERR_INVALID_ARGUMENT;
    if (dtype != KDA_DTYPE_F32 && dtype != KDA_DTYPE_BF16) return KDA_ERR_INVALID_ARGUMENT;
    if (B <= 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0 || num_seqs <= 0)
        return KDA_ERR_INVALID_ARGUMENT;
    if (!isfinite(scale)) return KDA_ERR_INVALID_ARGUMENT;
    if (cu_seqlens ? B != 1 : num_seqs != B) return KDA_ERR_INVALID_ARGUMENT;
    if ((long long)B * T * H * (dk > dv ? dk : dv) >= (1LL << 40)) return KDA_ERR_INVALID_ARGUMENT;
    if ((long long)B * T >= (1LL << 31) - kChunk) return KDA_ERR_INVALID_ARGUMENT;
    if ((long long)num_seqs * H * kMaxStateTiles >= (1LL << 31)) return KDA_ERR_UNSUPPORTED;
    const bool have_tokens = (long long)B * T > 0;
    if (have_tokens && (!q || !k || !v || !beta || !out)) return KDA_ERR_INVALID_ARGUMENT;
    if (!g_ok(g, pro, have_tokens)) return KDA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
        !aligned16(init_state) || !aligned16(final_state))
        return KDA_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(beta) & 3u) != 0) return KDA_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(cu_seqlens) & 3u) != 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!dims_ok(dk, dv)) return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

namespace {

kda_status chunk_fwd_impl(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, float scale, const float *init_state,
                          const int32_t *cu_seqlens, void *out, float *final_state, int B, int T,
                          int H, int dk, int dv, int num_seqs, kda_dtype dtype,
                          const kda_options *options, void *workspace, size_t workspace_bytes,
                          cudaStream_t stream, cudaEvent_t *events,
                          const GateParams &gate = GateParams{nullptr, nullptr, 0.f}) {
    const kda_status chk = chunk_fwd_check(q, k, v, g, beta, scale, init_state, cu_seqlens, out,
                                           final_state, B, T, H, dk, dv, num_seqs, dtype, options);
    if (chk != KDA_OK) return chk;
    Prologue pro;
    make_prologue(options, &pro);
    const size_t need = kda_chunk_fwd_workspace_size(B, T, H, dk, dv, num_seqs, dtype);
    if (!workspace || workspace_bytes < need) return KDA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return KDA_ERR_WORKSPACE;

    // The same slot bound as kda_chunk_fwd_workspace_size (one packed sequence
    // is bounded like a fixed-length batch of one).
    const bool packed = cu_seqlens != nullptr;
    const long long slots = max_chunk_slots(B, T, num_seqs, num_seqs != B);
    char *ws = static_cast<char *>(workspace);
    int *status = reinterpret_cast<int *>(ws);
    ChunkEntry *table = reinterpret_cast<ChunkEntry *>(ws + kWsHeader);
    int *seq_first_slot = reinterpret_cast<int *>(
        ws + kWsHeader + align_up((size_t)slots * sizeof(ChunkEntry), 256));
    char *region = ws + table_bytes(slots, num_seqs);
    const int seg_max = seg_limit(B, T, H, num_seqs, packed, use_tc(dk, dtype));
    float *seg_ws = seg_max >= 2 ? reinterpret_cast<float *>(
                                       region + align_up(path_region_bytes(slots, H, dk, dtype), 256))
                                 : nullptr;
    const int T_fixed = packed ? 0 : T;

    if (events && events[0] && cudaEventRecord(events[0], stream) != cudaSuccess) return KDA_ERR_CUDA;
    cudaError_t err = launch_chunk_table(cu_seqlens, num_seqs, T_fixed, (long long)B * T, slots, table,
                                         seq_first_slot, status, stream);
    if (err != cudaSuccess) return KDA_ERR_CUDA;
    if (use_tc(dk, dtype))
        err = launch_prefill_tc(q, k, v, g, beta, scale, init_state, cu_seqlens, out, final_state,
                                T_fixed, (long long)B * T, H, num_seqs, slots, table, seq_first_slot,
                                reinterpret_cast<unsigned char *>(region), status, pro,
                                options ? options->segments : 0, seg_max, seg_ws, gate,
                                options ? options->fused : 0, stream, events);
    else {
        err = launch_prefill_simt(q, k, v, g, beta, scale, init_state, cu_seqlens, out,
                                  final_state, T_fixed, H, dk, num_seqs, dtype, slots, table,
                                  seq_first_slot, reinterpret_cast<float *>(region), status, pro,
                                  stream, events);
        // The fp32 path applies the output gate as a pass over its outputs.
        if (err == cudaSuccess && gate.z)
            err = launch_output_gate_rmsnorm(out, gate.z, gate.w, gate.eps, out, (long long)B * T * H,
                                             dv, dtype, stream);
    }
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace

extern "C" kda_status kda_chunk_fwd(const void *q, const void *k, const void *v, const float *g,
                                    const float *beta, float scale, const float *init_state,
                                    const int32_t *cu_seqlens, void *out, float *final_state,
                                    int B, int T, int H, int dk, int dv, int num_seqs,
                                    kda_dtype dtype, void *workspace, size_t workspace_bytes,
                                    cudaStream_t stream) {
    return chunk_fwd_impl(q, k, v, g, beta, scale, init_state, cu_seqlens, out, final_state, B, T,
                          H, dk, dv, num_seqs, dtype, nullptr, workspace, workspace_bytes, stream,
                          nullptr);
}

extern "C" kda_status kda_chunk_fwd_timed(const void *q, const void *k, const void *v,
                                          const float *g, const float *beta, float scale,
                                          const float *init_state, const int32_t *cu_seqlens,
                                          void *out, float *final_state, int B, int T, int H,
                                          int dk, int dv, int num_seqs, kda_dtype dtype,
                                          void *workspace, size_t workspace_bytes,
                                          cudaStream_t stream, cudaEvent_t *events) {
    return chunk_fwd_impl(q, k, v, g, beta, scale, init_state, cu_seqlens, out, final_state, B, T,
                          H, dk, dv, num_seqs, dtype, nullptr, workspace, workspace_bytes, stream,
                          events);
}

extern "C" kda_status kda_chunk_fwd_opt(const void *q, const void *k, const void *v,
                                        const float *g, const float *beta, float scale,
                                        const float *init_state, const int32_t *cu_seqlens,
                                        void *out, float *final_state, int B, int T, int H, int dk,
                                        int dv, int num_seqs, kda_dtype dtype,
                                        const kda_options *options, void *workspace,
                                        size_t workspace_bytes, cudaStream_t stream,
                                        cudaEvent_t *events) {
    return chunk_fwd_impl(q, k, v, g, beta, scale, init_state, cu_seqlens, out, final_state, B, T,
                          H, dk, dv, num_seqs, dtype, options, workspace, workspace_bytes, stream,
                          events);
}

extern "C" kda_status kda_chunk_fwd_gated(const void *q, const void *k, const void *v,
                                          const float *g, const float *beta, float scale,
                                          const float *init_state, const int32_t *cu_seqlens,
                                          const void *z, const float *weight, float eps, void *out,
                                          float *final_state, int B, int T, int H, int dk, int dv,
                                          int num_seqs, kda_dtype dtype,
                                          const kda_options *options, void *workspace,
                                          size_t workspace_bytes, cudaStream_t stream,
                                          cudaEvent_t *events) {
    if (!(eps > 0.f) || !isfinite(eps)) return KDA_ERR_INVALID_ARGUMENT;
    if ((long long)B * T > 0 && !z) return KDA_ERR_INVALID_ARGUMENT;
    if (!aligned16(z) || (reinterpret_cast<uintptr_t>(weight) & 3u) != 0)
        return KDA_ERR_INVALID_ARGUMENT;
    if ((long long)B * T <= 0) z = nullptr;  // nothing to gate
    return chunk_fwd_impl(q, k, v, g, beta, scale, init_state, cu_seqlens, out, final_state, B, T,
                          H, dk, dv, num_seqs, dtype, options, workspace, workspace_bytes, stream,
                          events, GateParams{z, weight, eps});
}

namespace {

kda_status decode_impl(const void *q, const void *k, const void *v, const float *g,
                       const float *beta, float scale, float *state, void *out, int N, int H,
                       int dk, int dv, kda_dtype dtype, const kda_options *options,
                       cudaStream_t stream) {
    Prologue pro;
    if (!make_prologue(options, &pro)) return KDA_ERR_INVALID_ARGUMENT;
    if (dtype != KDA_DTYPE_F32 && dtype != KDA_DTYPE_BF16) return KDA_ERR_INVALID_ARGUMENT;
    if (N < 0 || H <= 0 || dk <= 0 || dv <= 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!isfinite(scale)) return KDA_ERR_INVALID_ARGUMENT;
    if ((long long)N * H >= (1LL << 31)) return KDA_ERR_INVALID_ARGUMENT;
    if (N > 0 && (!q || !k || !v || !beta || !state || !out)) return KDA_ERR_INVALID_ARGUMENT;
    if (!g_ok(g, pro, N > 0)) return KDA_ERR_INVALID_ARGUMENT;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(state) || !aligned16(out))
        return KDA_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(beta) & 3u) != 0) return KDA_ERR_INVALID_ARGUMENT;
    if (!dims_ok(dk, dv)) return KDA_ERR_UNSUPPORTED;
    const cudaError_t err =
        launch_decode(q, k, v, g, beta, scale, state, out, N, H, dk, dtype, pro, stream);
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace

extern "C" kda_status kda_decode_step(const void *q, const void *k, const void *v, const float *g,
                                      const float *beta, float scale, float *state, void *out,
                                      int N, int H, int dk, int dv, kda_dtype dtype,
                                      cudaStream_t stream) {
    return decode_impl(q, k, v, g, beta, scale, state, out, N, H, dk, dv, dtype, nullptr, stream);
}

extern "C" kda_status kda_decode_step_opt(const void *q, const void *k, const void *v,
                                          const float *g, const float *beta, float scale,
                                          float *state, void *out, int N, int H, int dk, int dv,
                                          kda_dtype dtype, const kda_options *options,
                                          cudaStream_t stream) {
    return decode_impl(q, k, v, g, beta, scale, state, out, N, H, dk, dv, dtype, options, stream);
}

extern "C" kda_status kda_output_gate_rmsnorm(const void *o, const void *z, const float *weight,
                                              float eps, void *out, long long tokens, int H,
                                              int dv, kda_dtype dtype, cudaStream_t stream) {
    if (dtype != KDA_DTYPE_F32 && dtype != KDA_DTYPE_BF16) return KDA_ERR_INVALID_ARGUMENT;
    if (tokens < 0 || H <= 0 || !(eps > 0.f) || !isfinite(eps)) return KDA_ERR_INVALID_ARGUMENT;
    if (tokens * H >= (1LL << 34)) return KDA_ERR_INVALID_ARGUMENT;  // grid of rows / 8 blocks
    if (tokens > 0 && (!o || !z || !out)) return KDA_ERR_INVALID_ARGUMENT;
    if (!aligned16(o) || !aligned16(z) || !aligned16(out)) return KDA_ERR_INVALID_ARGUMENT;
    if ((reinterpret_cast<uintptr_t>(weight) & 3u) != 0) return KDA_ERR_INVALID_ARGUMENT;
    if (dv != 64 && dv != 128) return KDA_ERR_UNSUPPORTED;
    const cudaError_t err =
        launch_output_gate_rmsnorm(o, z, weight, eps, out, tokens * H, dv, dtype, stream);
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
