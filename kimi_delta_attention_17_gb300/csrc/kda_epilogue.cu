// Output gate and RMS normalisation of the token outputs, per (token, head):
// out = w * o / sqrt(mean(o^2) + eps) * sigmoid(z) ("Understanding Kimi Delta
// Attention", closing remarks: output gating and RMS normalisation of the
// heads' outputs).
//
// Each row of d_v values is spread over the lanes that cover it in 16-byte
// pieces (8 lanes for d_v = 64 bf16, 16 for d_v = 128 bf16 or 64 fp32, 32 for
// 128 fp32), so that a warp holds several rows; every lane first issues the
// loads of its pieces of kEpiPasses rows, then finishes each row (sum of
// squares by a butterfly within the row's lanes, scale, gate, store). Pure HBM
// streaming: o and z read once, out written once; the loads in flight per
// lane are what keep HBM busy.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kEpiWarps = 8;   // warps per CTA
constexpr int kEpiPasses = 4;  // rows in flight per lane

template <typename T>
__device__ __forceinline__ void unpack16(const uint4 &r, float *x);
template <>
__device__ __forceinline__ void unpack16<__nv_bfloat16>(const uint4 &r, float *x) {
    const uint32_t u[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(u[i] << 16);
        x[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
}
template <>
__device__ __forceinline__ void unpack16<float>(const uint4 &r, float *x) {
    x[0] = __uint_as_float(r.x); x[1] = __uint_as_float(r.y);
    x[2] = __uint_as_float(r.z); x[3] = __uint_as_float(r.w);
}
template <typename T>
__device__ __forceinline__ uint4 pack16(const float *x);
template <>
__device__ __forceinline__ uint4 pack16<__nv_bfloat16>(const float *x) {
    uint32_t u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
        u[i] = *reinterpret_cast<const uint32_t *>(&h);
    }
    return make_uint4(u[0], u[1], u[2], u[3]);
}
template <>
__device__ __forceinline__ uint4 pack16<float>(const float *x) {
    return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                      __float_as_uint(x[3]));
}

template <int D, typename T>
struct EpiShape {
    static constexpr int E = 16 / (int)sizeof(T);  // values per 16-byte piece
    static constexpr int L = D / E;                // lanes per row
    static constexpr int RPW = 32 / L;             // rows per warp and pass
    static constexpr int rows_per_cta = kEpiWarps * RPW * kEpiPasses;
    static_assert(L >= 1 && L <= 32 && 32 % L == 0, "a row must fit a warp in 16-byte pieces");
};

template <int D, typename T>
__global__ void __launch_bounds__(32 * kEpiWarps)
output_gate_rmsnorm(const T *__restrict__ o, const T *__restrict__ z, const float *__restrict__ w,
                    float eps, T *out, long long rows) {
    using S = EpiShape<D, T>;
    constexpr int E = S::E, L = S::L, RPW = S::RPW;
    const int lane = threadIdx.x & 31, sub = lane / L, li = lane % L;
    const long long row0 = ((long long)blockIdx.x * kEpiWarps + (threadIdx.x >> 5)) * (RPW * kEpiPasses);
    float wv[E];
#pragma unroll
    for (int i = 0; i < E; ++i) wv[i] = w ? w[E * li + i] : 1.f;
    uint4 ro[kEpiPasses], rz[kEpiPasses];
#pragma unroll
    for (int p = 0; p < kEpiPasses; ++p) {
        const long long row = row0 + p * RPW + sub;
        if (row < rows) {
            const size_t off = (size_t)row * D + E * li;
            ro[p] = *reinterpret_cast<const uint4 *>(o + off);
            rz[p] = *reinterpret_cast<const uint4 *>(z + off);
        } else {
            ro[p] = make_uint4(0, 0, 0, 0);
            rz[p] = make_uint4(0, 0, 0, 0);
        }
    }
#pragma unroll
    for (int p = 0; p < kEpiPasses; ++p) {
        float x[E], g[E];
        unpack16<T>(ro[p], x);
        unpack16<T>(rz[p], g);
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < E; ++i) ss += x[i] * x[i];
#pragma unroll
        for (int m = L / 2; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
        const float r = rsqrtf(ss * (1.f / D) + eps);
#pragma unroll
        for (int i = 0; i < E; ++i) x[i] = wv[i] * x[i] * r * __fdividef(1.f, 1.f + __expf(-g[i]));
        const long long row = row0 + p * RPW + sub;
        if (row < rows) *reinterpret_cast<uint4 *>(out + (size_t)row * D + E * li) = pack16<T>(x);
    }
}

template <int D, typename T>
cudaError_t launch_epi(const void *o, const void *z, const float *w, float eps, void *out,
                       long long rows, cudaStream_t stream) {
    constexpr long long per = EpiShape<D, T>::rows_per_cta;
    const long long blocks = (rows + per - 1) / per;
    output_gate_rmsnorm<D, T><<<(unsigned)blocks, 32 * kEpiWarps, 0, stream>>>(
        static_cast<const T *>(o), static_cast<const T *>(z), w, eps, static_cast<T *>(out), rows);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_output_gate_rmsnorm(const void *o, const void *z, const float *w, float eps,
                                       void *out, long long rows, int dv, kda_dtype dtype,
                                       cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    if (dtype == KDA_DTYPE_BF16)
        return dv == 128 ? launch_epi<128, __nv_bfloat16>(o, z, w, eps, out, rows, stream)
                         : launch_epi<64, __nv_bfloat16>(o, z, w, eps, out, rows, stream);
    return dv == 128 ? launch_epi<128, float>(o, z, w, eps, out, rows, stream)
                     : launch_epi<64, float>(o, z, w, eps, out, rows, stream);
}

}  // namespace kda
