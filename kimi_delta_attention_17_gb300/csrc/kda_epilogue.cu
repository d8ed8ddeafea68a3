// Output gate and RMS normalisation of the token outputs, per (token, head):
// out = w * o / sqrt(mean(o^2) + eps) * sigmoid(z) ("Understanding Kimi Delta
// Attention", closing remarks: output gating and RMS normalisation of the
// heads' outputs).
//
// One warp per (token, head) row of d_v values: each lane moves d_v / 32
// consecutive values (16 or 8 bytes in bf16), the sum of squares is a warp
// butterfly, and the row is written back scaled. Pure HBM streaming: the row
// of o and of z read once, out written once.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kEpiWarps = 8;  // rows per CTA

template <int V, typename T> struct Vec;  // V consecutive values
template <> struct Vec<4, __nv_bfloat16> { using type = uint2; };
template <> struct Vec<2, __nv_bfloat16> { using type = uint32_t; };
template <> struct Vec<4, float> { using type = float4; };
template <> struct Vec<2, float> { using type = float2; };

template <int V, typename T>
__device__ __forceinline__ void load_row(const T *p, float (&x)[V]) {
    const typename Vec<V, T>::type r = *reinterpret_cast<const typename Vec<V, T>::type *>(p);
    const T *e = reinterpret_cast<const T *>(&r);
#pragma unroll
    for (int i = 0; i < V; ++i) x[i] = to_f32(e[i]);
}
template <int V, typename T>
__device__ __forceinline__ void store_row(T *p, const float (&x)[V]) {
    typename Vec<V, T>::type r;
    T *e = reinterpret_cast<T *>(&r);
#pragma unroll
    for (int i = 0; i < V; ++i) e[i] = from_f32<T>(x[i]);
    *reinterpret_cast<typename Vec<V, T>::type *>(p) = r;
}

template <int D, typename T>
__global__ void __launch_bounds__(32 * kEpiWarps)
output_gate_rmsnorm(const T *__restrict__ o, const T *__restrict__ z, const float *__restrict__ w,
                    float eps, T *out, long long rows) {
    constexpr int V = D / 32;
    const long long row = (long long)blockIdx.x * kEpiWarps + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    const size_t off = (size_t)row * D + V * lane;
    float x[V], g[V];
    load_row<V>(o + off, x);
    load_row<V>(z + off, g);
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < V; ++i) ss += x[i] * x[i];
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
    const float r = rsqrtf(ss * (1.f / D) + eps);
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const float wi = w ? w[V * lane + i] : 1.f;
        x[i] = wi * x[i] * r * __fdividef(1.f, 1.f + __expf(-g[i]));
    }
    store_row<V>(out + off, x);
}

template <int D, typename T>
cudaError_t launch_epi(const void *o, const void *z, const float *w, float eps, void *out,
                       long long rows, cudaStream_t stream) {
    const long long blocks = (rows + kEpiWarps - 1) / kEpiWarps;
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
