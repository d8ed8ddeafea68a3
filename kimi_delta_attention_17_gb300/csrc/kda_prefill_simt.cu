// fp32 SIMT chunkwise prefill: the reference-precision path (fp32 storage
// dtype) and an independent check of the tensor-core path.
//
// The chunk algebra is the one derived in "Understanding Kimi Delta
// Attention", sections "The triangular system" and "Putting the chunks
// together". For one chunk of n <= 64 tokens with incoming state S0, G the
// in-chunk cumulative log-decay and q already multiplied by the query scale:
//
//   A_ij = -beta_i sum_c k_ic k_jc exp(G_ic - G_jc)   (j < i)
//   H_ij =         sum_c q_ic k_jc exp(G_ic - G_jc)   (j <= i)
//   T    = (I - A)^{-1}                                (forward substitution)
//   W    = T Diag(beta) L,  L_j = k_j o exp(G_j)
//   U    = T Diag(beta) V
//   Z    = U - W S0,   O = Qbar S0 + H Z,   Qbar_i = q_i o exp(G_i)
//   S1   = Diag(exp(G_n)) S0 + Kbar^T Z,   Kbar_j = k_j o exp(G_n - G_j)
//
// The output is regrouped so that the state pass needs only products with S0:
//   O = (Qbar - H W) S0 + H U = Q' S0 + Ou.
// Phase 1 (one CTA per chunk and head, all chunks in parallel) computes
// W, Q', Kbar, U, Ou and exp(G_n) into the workspace; phase 2 (one CTA per
// sequence, head and 16-column slab of the state) walks the chunks in order:
//   Z = U - W S,  O = Ou + Q' S,  S <- Diag(exp(G_n)) S + Kbar^T Z.
//
// Here every pair decay exp(G_i - G_j) with j <= i is formed directly (its
// exponent is <= 0, so it cannot overflow). Padded tokens of a ragged last
// chunk carry k = q = v = 0, beta = 0, g = 0: identity transitions whose rows
// of W, U, Q', Ou and Kbar are zero and whose outputs are not stored.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;

template <int D>
__host__ __device__ constexpr size_t region_floats() {
    return (size_t)5 * kChunk * D + D;
}

// Offsets inside one (chunk slot, head) region, in floats.
template <int D> struct Region {
    static constexpr size_t W = 0;
    static constexpr size_t Qp = (size_t)kChunk * D;
    static constexpr size_t Kb = (size_t)2 * kChunk * D;
    static constexpr size_t U = (size_t)3 * kChunk * D;
    static constexpr size_t Ou = (size_t)4 * kChunk * D;
    static constexpr size_t Gam = (size_t)5 * kChunk * D;
};

template <int D>
constexpr size_t prep_smem_bytes() {
    // k, q, G, v rows padded to D+1; A, T, H 64x64; beta 64.
    return sizeof(float) * ((size_t)4 * kChunk * (D + 1) + 3 * kChunk * kChunk + kChunk);
}

template <int D, typename InT>
__global__ void __launch_bounds__(kThreads)
simt_chunk_prep(const InT *__restrict__ q, const InT *__restrict__ k, const InT *__restrict__ v,
                const float *__restrict__ g, const float *__restrict__ beta, float scale,
                const ChunkEntry *__restrict__ table, long long nslots, int H,
                float *__restrict__ ws, Prologue pro) {
    constexpr int P = D + 1;  // padded row stride
    const int h = blockIdx.x;  // heads fastest: resident CTAs read whole token rows
    const long long slot = (long long)blockIdx.z * gridDim.y + blockIdx.y;
    if (slot >= nslots) return;
    const ChunkEntry ce = table[slot];
    if (ce.seq < 0) return;
    const int tid = threadIdx.x;

    extern __shared__ float sm[];
    float *ks = sm;
    float *qs = ks + kChunk * P;
    float *Gs = qs + kChunk * P;
    float *vs = Gs + kChunk * P;
    float *As = vs + kChunk * P;
    float *Ts = As + kChunk * kChunk;
    float *Hs = Ts + kChunk * kChunk;
    float *bs = Hs + kChunk * kChunk;

    for (int idx = tid; idx < kChunk * D; idx += kThreads) {
        const int i = idx / D, c = idx % D;
        float kv = 0.f, qv = 0.f, gv = 0.f, vv = 0.f;
        if (i < ce.len) {
            const size_t tok = (size_t)(ce.bos + i) * H + h;
            const size_t off = tok * D + c;
            kv = to_f32(k[off]);
            qv = to_f32(q[off]);  // scaled below, after any normalisation
            // log a_t per channel, one per head (broadcast), or none.
            if (pro.decay == KDA_DECAY_CHANNEL) gv = log_decay(g[off], pro);
            else if (pro.decay == KDA_DECAY_SCALAR) gv = log_decay(g[tok], pro);
            vv = to_f32(v[off]);
        }
        ks[i * P + c] = kv;
        qs[i * P + c] = qv;
        Gs[i * P + c] = gv;
        vs[i * P + c] = vv;
    }
    if (tid < kChunk) bs[tid] = tid < ce.len ? beta[(size_t)(ce.bos + tid) * H + h] : 0.f;
    __syncthreads();
    // q (and, when asked, q and k normalised per token): row r of k or q by
    // one thread, x / sqrt(sum x^2 + eps), then the query scale.
    if (tid < 2 * kChunk) {
        const int r = tid & (kChunk - 1);
        float *row = (tid < kChunk ? ks : qs) + r * P;
        float f = tid < kChunk ? 1.f : scale;
        if (pro.l2norm) {
            float ss = 0.f;
            for (int c = 0; c < D; ++c) ss += row[c] * row[c];
            f *= rsqrtf(ss + kL2Eps);
        }
        if (f != 1.f)
            for (int c = 0; c < D; ++c) row[c] *= f;
    }
    __syncthreads();

    // In-chunk cumulative log-decay, one thread per key channel.
    if (tid < D) {
        float acc = 0.f;
        for (int i = 0; i < kChunk; ++i) {
            acc += Gs[i * P + tid];
            Gs[i * P + tid] = acc;
        }
    }
    __syncthreads();

    // A (strictly lower) and H (lower, inclusive): one (i, j) pair per thread pass.
    for (int p = tid; p < kChunk * kChunk; p += kThreads) {
        const int i = p / kChunk, j = p % kChunk;
        float a = 0.f, hq = 0.f;
        if (j <= i) {
            for (int c = 0; c < D; ++c) {
                const float kj = ks[j * P + c] * expf(Gs[i * P + c] - Gs[j * P + c]);
                a += ks[i * P + c] * kj;
                hq += qs[i * P + c] * kj;
            }
        }
        As[p] = j < i ? -bs[i] * a : 0.f;
        Hs[p] = hq;
    }
    __syncthreads();

    // T = (I - A)^{-1}: column `col` by forward substitution,
    // T_i,col = [i == col] + sum_{col <= j < i} A_ij T_j,col.
    if (tid < kChunk) {
        const int col = tid;
        for (int i = 0; i < kChunk; ++i) {
            float acc = i == col ? 1.f : 0.f;
            for (int j = col; j < i; ++j) acc += As[i * kChunk + j] * Ts[j * kChunk + col];
            Ts[i * kChunk + col] = i < col ? 0.f : acc;
        }
    }

    float *reg = ws + ((size_t)slot * H + h) * region_floats<D>();
    // Kbar and exp(G_n) (G is flat past the last real token, so row 63 holds G_n).
    for (int idx = tid; idx < kChunk * D; idx += kThreads) {
        const int i = idx / D, c = idx % D;
        reg[Region<D>::Kb + idx] = ks[i * P + c] * expf(Gs[(kChunk - 1) * P + c] - Gs[i * P + c]);
    }
    if (tid < D) reg[Region<D>::Gam + tid] = expf(Gs[(kChunk - 1) * P + tid]);
    __syncthreads();

    // In place: ks <- Diag(beta) L,  qs <- Qbar,  vs <- Diag(beta) V.
    for (int idx = tid; idx < kChunk * D; idx += kThreads) {
        const int i = idx / D, c = idx % D;
        const float e = expf(Gs[i * P + c]);
        ks[i * P + c] *= bs[i] * e;
        qs[i * P + c] *= e;
        vs[i * P + c] *= bs[i];
    }
    __syncthreads();

    // W = T (B L),  U = T (B V).
    for (int idx = tid; idx < kChunk * D; idx += kThreads) {
        const int i = idx / D, c = idx % D;
        float w = 0.f, u = 0.f;
        for (int j = 0; j <= i; ++j) {
            const float t = Ts[i * kChunk + j];
            w += t * ks[j * P + c];
            u += t * vs[j * P + c];
        }
        reg[Region<D>::W + idx] = w;
        reg[Region<D>::U + idx] = u;
    }
    __syncthreads();

    // Q' = Qbar - H W,  Ou = H U (W and U read back from this block's writes).
    for (int idx = tid; idx < kChunk * D; idx += kThreads) {
        const int i = idx / D, c = idx % D;
        float qp = qs[i * P + c], ou = 0.f;
        for (int j = 0; j <= i; ++j) {
            const float hh = Hs[i * kChunk + j];
            qp -= hh * reg[Region<D>::W + j * D + c];
            ou += hh * reg[Region<D>::U + j * D + c];
        }
        reg[Region<D>::Qp + idx] = qp;
        reg[Region<D>::Ou + idx] = ou;
    }
}

constexpr int kSlabCols = 16;

template <int D>
constexpr size_t pass_smem_bytes() {
    // [W; Q'] 128 x (D+1), Kbar 64 x (D+1), S D x 16, U/Ou/Z 64 x 16, gamma D.
    return sizeof(float) * ((size_t)3 * kChunk * (D + 1) + (size_t)D * kSlabCols +
                            (size_t)3 * kChunk * kSlabCols + D);
}

template <int D, typename OutT>
__global__ void __launch_bounds__(kThreads)
simt_state_pass(const float *__restrict__ ws, const int *__restrict__ seq_first_slot,
                const int *__restrict__ seq_order, const int32_t *__restrict__ cu_seqlens,
                int T_fixed, const float *init_state, OutT *__restrict__ out, float *final_state,
                int H, const int *__restrict__ status) {
    // A call whose chunk table was refused (or that already failed) does
    // nothing; the decision is taken once for the whole CTA.
    if (__syncthreads_or(threadIdx.x == 0 && *status != 0)) return;
    constexpr int P = D + 1;
    // 1-D grid, sequences slowest in seq_order (longest first), then heads,
    // then the column slabs of one head.
    constexpr int kTiles = D / kSlabCols;
    const int per_seq = H * kTiles;
    const int r = (int)blockIdx.x / per_seq, rem = (int)blockIdx.x - r * per_seq;
    const int h = rem / kTiles, j0 = (rem - h * kTiles) * kSlabCols;
    const int n = seq_order[r];
    const int tid = threadIdx.x;
    int bos, len;
    if (cu_seqlens) {
        bos = cu_seqlens[n];
        len = cu_seqlens[n + 1] - bos;
    } else {
        bos = n * T_fixed;
        len = T_fixed;
    }
    const int nchunks = (len + kChunk - 1) / kChunk;
    const int slot0 = seq_first_slot[n];

    extern __shared__ float sm[];
    float *A1 = sm;                        // [128][P]: rows 0-63 W, 64-127 Q'
    float *Kb = A1 + 2 * kChunk * P;       // [64][P]
    float *S = Kb + kChunk * P;            // [D][16]
    float *Us = S + D * kSlabCols;         // [64][16]
    float *Os = Us + kChunk * kSlabCols;   // [64][16]
    float *Zs = Os + kChunk * kSlabCols;   // [64][16]
    float *gam = Zs + kChunk * kSlabCols;  // [D]

    const size_t st_off = ((size_t)n * H + h) * D * D;
    for (int idx = tid; idx < D * kSlabCols; idx += kThreads) {
        const int c = idx / kSlabCols, j = idx % kSlabCols;
        S[idx] = init_state ? init_state[st_off + (size_t)c * D + j0 + j] : 0.f;
    }

    for (int ch = 0; ch < nchunks; ++ch) {
        const float *reg = ws + ((size_t)(slot0 + ch) * H + h) * region_floats<D>();
        __syncthreads();
        for (int idx = tid; idx < kChunk * D; idx += kThreads) {
            const int i = idx / D, c = idx % D;
            A1[i * P + c] = reg[Region<D>::W + idx];
            A1[(kChunk + i) * P + c] = reg[Region<D>::Qp + idx];
            Kb[i * P + c] = reg[Region<D>::Kb + idx];
        }
        for (int idx = tid; idx < kChunk * kSlabCols; idx += kThreads) {
            const int i = idx / kSlabCols, j = idx % kSlabCols;
            Us[idx] = reg[Region<D>::U + i * D + j0 + j];
            Os[idx] = reg[Region<D>::Ou + i * D + j0 + j];
        }
        if (tid < D) gam[tid] = reg[Region<D>::Gam + tid];
        __syncthreads();

        const int clen = min(kChunk, len - ch * kChunk);
        for (int o = tid; o < 2 * kChunk * kSlabCols; o += kThreads) {
            const int r = o / kSlabCols, j = o % kSlabCols;
            float acc = 0.f;
            for (int c = 0; c < D; ++c) acc += A1[r * P + c] * S[c * kSlabCols + j];
            if (r < kChunk) {
                Zs[r * kSlabCols + j] = Us[r * kSlabCols + j] - acc;
            } else if (r - kChunk < clen) {
                const int i = r - kChunk;
                out[((size_t)(bos + ch * kChunk + i) * H + h) * D + j0 + j] =
                    from_f32<OutT>(Os[i * kSlabCols + j] + acc);
            }
        }
        __syncthreads();
        for (int o = tid; o < D * kSlabCols; o += kThreads) {
            const int c = o / kSlabCols, j = o % kSlabCols;
            float acc = 0.f;
            for (int i = 0; i < kChunk; ++i) acc += Kb[i * P + c] * Zs[i * kSlabCols + j];
            S[o] = gam[c] * S[o] + acc;
        }
    }
    __syncthreads();
    if (final_state) {
        for (int idx = tid; idx < D * kSlabCols; idx += kThreads) {
            const int c = idx / kSlabCols, j = idx % kSlabCols;
            final_state[st_off + (size_t)c * D + j0 + j] = S[idx];
        }
    }
}

template <int D, typename InT>
cudaError_t launch_t(const void *q, const void *k, const void *v, const float *g,
                     const float *beta, float scale, const float *init_state,
                     const int32_t *cu_seqlens, void *out, float *final_state, int T_fixed, int H,
                     int num_seqs, long long slots, const ChunkEntry *table,
                     const int *seq_first_slot, float *region, const int *status,
                     const Prologue &pro, cudaStream_t stream, cudaEvent_t *events) {
    constexpr size_t s1 = prep_smem_bytes<D>();
    constexpr size_t s2 = pass_smem_bytes<D>();
    // The shared-memory opt-ins, once per device and instance (nothing but
    // launches then reaches the stream, so a call can be graph-captured).
    static bool ready[64];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!ready[dev]) {
        err = cudaFuncSetAttribute(simt_chunk_prep<D, InT>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
        if (err != cudaSuccess) return err;
        err = cudaFuncSetAttribute(simt_state_pass<D, InT>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2);
        if (err != cudaSuccess) return err;
        ready[dev] = true;
    }
    if ((err = mark(events, 1, stream)) != cudaSuccess) return err;
    if (slots > 0) {
        simt_chunk_prep<D, InT><<<head_slot_grid(H, slots), kThreads, s1, stream>>>(
            static_cast<const InT *>(q), static_cast<const InT *>(k), static_cast<const InT *>(v), g,
            beta, scale, table, slots, H, region, pro);
        err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    if ((err = mark(events, 2, stream)) != cudaSuccess) return err;
    if (num_seqs > 0) {
        static_assert(D / kSlabCols <= kMaxStateTiles, "grid bound checked with kMaxStateTiles");
        simt_state_pass<D, InT><<<(unsigned)num_seqs * H * (D / kSlabCols), kThreads, s2, stream>>>(
            region, seq_first_slot, seq_first_slot + num_seqs + 1, cu_seqlens, T_fixed, init_state,
            static_cast<InT *>(out), final_state, H, status);
        err = cudaGetLastError();
        if (err != cudaSuccess) return err;
    }
    return mark(events, 3, stream);
}

}  // namespace

size_t simt_region_bytes(int d) {
    return d == 128 ? region_floats<128>() * sizeof(float) : region_floats<64>() * sizeof(float);
}

cudaError_t launch_prefill_simt(const void *q, const void *k, const void *v, const float *g,
                                const float *beta, float scale, const float *init_state,
                                const int32_t *cu_seqlens, void *out, float *final_state,
                                int T_fixed, int H, int d, int num_seqs, kda_dtype dtype,
                                long long slots, const ChunkEntry *table,
                                const int *seq_first_slot, float *region, const int *status,
                                const Prologue &pro, cudaStream_t stream, cudaEvent_t *events) {
#define KDA_SIMT_ARGS q, k, v, g, beta, scale, init_state, cu_seqlens, out, final_state, T_fixed, H, \
                      num_seqs, slots, table, seq_first_slot, region, status, pro, stream, events
    if (dtype == KDA_DTYPE_BF16)
        return d == 128 ? launch_t<128, __nv_bfloat16>(KDA_SIMT_ARGS)
                        : launch_t<64, __nv_bfloat16>(KDA_SIMT_ARGS);
    return d == 128 ? launch_t<128, float>(KDA_SIMT_ARGS) : launch_t<64, float>(KDA_SIMT_ARGS);
#undef KDA_SIMT_ARGS
}

}  // namespace kda
