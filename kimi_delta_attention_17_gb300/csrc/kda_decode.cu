// Single-token recurrent decode step, fused into one pass over the state.
//
// Per (sequence, head), with a = exp(g), the update of "Understanding Kimi
// Delta Attention" (box "KDA: Retain, predict, correct") reads
//     S' = Diag(a) S + k e^T,  e = beta (v - (Diag(a) S)^T k),  o = S'^T (s q).
// Expanding the read, S'^T (s q) = S^T (a o s q) + (s q^T k) e, so the old
// state is read exactly once: both reductions over the key channels,
//     vhat = S^T (a o k)   and   p = S^T (a o s q),
// come from the same registers, then e and o follow, then S' is written.
//
// The step is pure HBM streaming (64 KiB read + 64 KiB written per head at
// d = 128 against ~1.3 KiB of token inputs). One CTA of 128 threads owns a
// 32-column slab of one head's state: 16 row groups x 8 column quads, each
// thread holding d/16 float4 rows of the slab in registers; all loads are
// issued before any arithmetic and each warp touches 4 full 128-byte rows.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kDecodeThreads = 128;
constexpr int kSlab = 32;  // state columns per CTA

// Instances: kVar 0 is the plain step (per-channel log-decay in g, no
// normalisation) and 2 the KDA layer's own prologue (per-channel decay from
// gate logits through the log-sigmoid, q and k normalised), each compiled
// with its options fixed; 1 takes every option at run time.
constexpr int kDecPlain = 0, kDecRuntime = 1, kDecGated = 2;
template <int D, typename InT, int kVar>
__global__ void __launch_bounds__(kDecodeThreads, 7)
decode_step_kernel(const InT *__restrict__ q, const InT *__restrict__ k, const InT *__restrict__ v,
                   const float *__restrict__ g, const float *__restrict__ beta, float scale,
                   float *__restrict__ state, InT *__restrict__ out, Prologue pro) {
    constexpr bool kOpts = kVar != kDecPlain;
    if (kVar == kDecGated) pro = Prologue{KDA_DECAY_CHANNEL, KDA_GATE_LOGSIGMOID, 0.f, 1};
    constexpr int R = D / 16;  // rows per thread
    const int nh = blockIdx.x;           // (sequence, head) flattened
    const int col0 = blockIdx.y * kSlab;  // first state column of this slab
    const int tid = threadIdx.x;
    const int cq = tid & 7;   // column quad within the slab
    const int rg = tid >> 3;  // row group 0..15; rows rg + 16 m

    float *S = state + (size_t)nh * D * D + col0 + 4 * cq;
    float4 s[R];
#pragma unroll
    for (int m = 0; m < R; ++m)
        s[m] = *reinterpret_cast<const float4 *>(S + (size_t)(rg + 16 * m) * D);

    const size_t tok = (size_t)nh * D;
    // Decay of this head: per channel, one per head, or none (log a = 0).
    const float ah = kOpts && pro.decay == KDA_DECAY_SCALAR ? decay_factor(g[nh], pro) : 1.f;
    // All row loads first (one uniform branch around g), so that they are in
    // flight together.
    float zr[R], kin[R], qin[R];
    const bool chan = !kOpts || pro.decay == KDA_DECAY_CHANNEL;
    if (chan) {
#pragma unroll
        for (int m = 0; m < R; ++m) zr[m] = g[tok + rg + 16 * m];
    }
#pragma unroll
    for (int m = 0; m < R; ++m) {
        kin[m] = to_f32(k[tok + rg + 16 * m]);
        qin[m] = to_f32(q[tok + rg + 16 * m]);
    }
    float av[R], ak[R], aq[R], kr[R];
    float qk = 0.f, kss = 0.f, qss = 0.f;  // q.k and the squared norms of raw k and q
#pragma unroll
    for (int m = 0; m < R; ++m) {
        const float a = !kOpts ? expf(zr[m]) : chan ? decay_factor(zr[m], pro)
                                                    : ah;  // per head, or 1 without decay
        const float kk = kin[m];
        const float q0 = qin[m];
        const float qq = scale * q0;
        av[m] = a;
        kr[m] = kk;
        ak[m] = a * kk;
        aq[m] = a * qq;
        qk += qq * kk;
        if (kOpts) {
            kss += kk * kk;
            qss += q0 * q0;
        }
    }
    float4 vh = make_float4(0.f, 0.f, 0.f, 0.f), po = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < R; ++m) {
        vh.x += ak[m] * s[m].x; vh.y += ak[m] * s[m].y; vh.z += ak[m] * s[m].z; vh.w += ak[m] * s[m].w;
        po.x += aq[m] * s[m].x; po.y += aq[m] * s[m].y; po.z += aq[m] * s[m].z; po.w += aq[m] * s[m].w;
    }
    // Sum over the 4 row groups of this warp (lanes 8 apart) ...
#pragma unroll
    for (int off = 8; off < 32; off <<= 1) {
        vh.x += __shfl_xor_sync(0xffffffffu, vh.x, off);
        vh.y += __shfl_xor_sync(0xffffffffu, vh.y, off);
        vh.z += __shfl_xor_sync(0xffffffffu, vh.z, off);
        vh.w += __shfl_xor_sync(0xffffffffu, vh.w, off);
        po.x += __shfl_xor_sync(0xffffffffu, po.x, off);
        po.y += __shfl_xor_sync(0xffffffffu, po.y, off);
        po.z += __shfl_xor_sync(0xffffffffu, po.z, off);
        po.w += __shfl_xor_sync(0xffffffffu, po.w, off);
        qk += __shfl_xor_sync(0xffffffffu, qk, off);
        if (kOpts) {
            kss += __shfl_xor_sync(0xffffffffu, kss, off);
            qss += __shfl_xor_sync(0xffffffffu, qss, off);
        }
    }
    // ... then over the 4 warps.
    constexpr int NR = kOpts ? 11 : 9;  // reduced values per column quad
    __shared__ float red[4][8][NR];
    const int warp = tid >> 5, lane = tid & 31;
    if (lane < 8) {
        float *r = red[warp][lane];
        r[0] = vh.x; r[1] = vh.y; r[2] = vh.z; r[3] = vh.w;
        r[4] = po.x; r[5] = po.y; r[6] = po.z; r[7] = po.w;
        r[8] = qk;
        if (kOpts) {
            r[NR - 2] = kss;
            r[NR - 1] = qss;
        }
    }
    __syncthreads();
    float tot[NR];
#pragma unroll
    for (int i = 0; i < NR; ++i) tot[i] = red[0][cq][i] + red[1][cq][i] + red[2][cq][i] + red[3][cq][i];
    if (kOpts && pro.l2norm) {
        // The reads are linear in k and q: normalising afterwards scales vhat by
        // 1/|k|, the decayed query read by 1/|q|, q.k by both, and the write by 1/|k|.
        const float rk = rsqrtf(tot[NR - 2] + kL2Eps), rq = rsqrtf(tot[NR - 1] + kL2Eps);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            tot[i] *= rk;
            tot[4 + i] *= rq;
        }
        tot[8] *= rk * rq;
#pragma unroll
        for (int m = 0; m < R; ++m) kr[m] *= rk;
    }

    const float b = beta[nh];
    const size_t vo = (size_t)nh * D + col0 + 4 * cq;
    float e[4], o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        e[i] = b * (to_f32(v[vo + i]) - tot[i]);
        o[i] = tot[4 + i] + tot[8] * e[i];
    }
    if (rg == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) out[vo + i] = from_f32<InT>(o[i]);
    }
#pragma unroll
    for (int m = 0; m < R; ++m) {
        const float a = av[m];
        float4 n;
        n.x = a * s[m].x + kr[m] * e[0];
        n.y = a * s[m].y + kr[m] * e[1];
        n.z = a * s[m].z + kr[m] * e[2];
        n.w = a * s[m].w + kr[m] * e[3];
        *reinterpret_cast<float4 *>(S + (size_t)(rg + 16 * m) * D) = n;
    }
}

template <int D, typename InT>
cudaError_t launch_decode_t(const void *q, const void *k, const void *v, const float *g,
                            const float *beta, float scale, float *state, void *out, int N, int H,
                            const Prologue &pro, cudaStream_t stream) {
    dim3 grid((unsigned)(N * H), D / kSlab);
    const bool chan = pro.decay == KDA_DECAY_CHANNEL;
    const int var = chan && pro.gate == KDA_GATE_LOG && !pro.l2norm              ? kDecPlain
                    : chan && pro.gate == KDA_GATE_LOGSIGMOID && pro.l2norm ? kDecGated
                                                                               : kDecRuntime;
#define KDA_DECODE_LAUNCH(V)                                                                   \
    decode_step_kernel<D, InT, V><<<grid, kDecodeThreads, 0, stream>>>(                          \
        static_cast<const InT *>(q), static_cast<const InT *>(k), static_cast<const InT *>(v), g, \
        beta, scale, state, static_cast<InT *>(out), pro)
    switch (var) {
        case kDecPlain: KDA_DECODE_LAUNCH(kDecPlain); break;
        case kDecGated: KDA_DECODE_LAUNCH(kDecGated); break;
        default: KDA_DECODE_LAUNCH(kDecRuntime); break;
    }
#undef KDA_DECODE_LAUNCH
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, float scale, float *state, void *out, int N, int H,
                          int d, kda_dtype dtype, const Prologue &pro, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    if (dtype == KDA_DTYPE_BF16) {
        return d == 128 ? launch_decode_t<128, __nv_bfloat16>(q, k, v, g, beta, scale, state, out, N, H, pro, stream)
                        : launch_decode_t<64, __nv_bfloat16>(q, k, v, g, beta, scale, state, out, N, H, pro, stream);
    }
    return d == 128 ? launch_decode_t<128, float>(q, k, v, g, beta, scale, state, out, N, H, pro, stream)
                    : launch_decode_t<64, float>(q, k, v, g, beta, scale, state, out, N, H, pro, stream);
}

}  // namespace kda
