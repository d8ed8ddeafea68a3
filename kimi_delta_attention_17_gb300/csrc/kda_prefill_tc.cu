// Tensor-core chunkwise prefill for bf16 q/k/v with d_k = d_v = 128 (sm_103a:
// tcgen05.mma with TMEM accumulators, 1-D bulk copies for the state pass).
//
// The algebra is the chunkwise form of "Understanding Kimi Delta Attention"
// (sections "The triangular system" and "Putting the chunks together"), with
// the output regrouped as O = (Qbar - H W) S0 + H U = Q' S0 + Ou so that the
// serial state pass only multiplies by the state:
//
//   phase 1 (every chunk and head in parallel, one CTA each):
//     G      in-chunk cumulative log-decay (registers, one thread per channel)
//     A, H   decay-gated K K^T and Q K^T, from ONE tcgen05.mma (below)
//     T      (I - A)^{-1}: blocked forward substitution in fp32 shared memory
//     W = (T B) L,  U = (T B) V                 two MMAs, B = Diag(beta)
//     Q' = Qbar - H W,  Ou = H U                two MMAs
//     Kbar^T, exp(G_n)                          elementwise
//   phase 2 (one CTA per sequence, head and 32-column slab of the state,
//   chunks in order, state in registers):
//     [W S; Q' S] = [W; Q'] S                   one MMA, M = 128
//     Z = U - W S,  O = Ou + Q' S
//     S <- Diag(exp(G_n)) S + Kbar^T Z          one MMA
//
// Decay absorption with secondary chunking ("Kimi Delta Attention: a half-life
// per channel", section "What changes in the kernel"): the per-channel pair
// decay exp(G_i - G_j) factors through a reference r as
//     exp(G_i - G_r) * exp(G_r - G_j),
// which turns the gated products into plain matmuls of rescaled rows. Each
// 16-token block I of the chunk has its reference at its 8th token, r(I); a
// row i in block I is scaled by E_i = exp(G_i - G_r(I)) and a column j in
// block J <= I by exp(G_r(I) - G_j) = exp(G_r(I) - G_r(J)) / E_j. Every factor
// spans at most 8 tokens of decay where it can exceed 1, so nothing overflows
// fp32 for per-token log-decays down to about -10 (the factors that shrink
// may underflow to zero, exactly where the true product is negligible). The
// ten (I, J) column versions stack into one B operand of 160 rows, and the
// K-tilde / Q-tilde rows into one A operand of 128 rows, so a single
// M=128, N=160, K=128 MMA yields every block of A (rows 0-63) and H (rows
// 64-127) at once; each row keeps the columns of its own versions.
//
// Operands are written by threads into no-swizzle canonical layouts: one
// thread per key channel writes 16-byte runs along the token axis (MN-major
// tiles when the contraction runs over channels, K-major when it runs over
// tokens). Accumulators are read back with tcgen05.ld (thread t = TMEM lane t).
#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int D = 128;   // d_k = d_v on this path
constexpr int C = kChunk;
constexpr int kTN = 32;  // state columns per phase-2 CTA

// Workspace region of one (chunk slot, head), byte offsets.
struct TcRegion {
    static constexpr size_t A1 = 0;        // [W; Q'] bf16, MN-major, 128 tokens x 128 ch
    static constexpr size_t A2 = 32768;    // Kbar^T bf16, K-major, 128 ch x 64 tokens
    static constexpr size_t U = 49152;     // fp32 [D/kTN][64][kTN], rows swizzled
    static constexpr size_t Ou = 81920;    // same layout as U
    static constexpr size_t Gam = 114688;  // fp32 [128] exp(G_n)
    static constexpr size_t bytes = 115200;
};
// Descriptor strides of the workspace tiles (and of their shared-memory copies).
constexpr uint32_t kA1Lbo = 128, kA1Sbo = 2048;  // MN-major: channel cores adjacent
constexpr uint32_t kA2Lbo = 2048, kA2Sbo = 128;  // K-major: channel groups adjacent

// Position of U/Ou element (token i, column j within a kTN slab): float4
// groups of a row are XOR-swizzled by (i & 7) so that one thread per row
// reads its row without bank conflicts.
__device__ __forceinline__ int slab_idx(int i, int j) {
    return i * kTN + ((((j >> 2) ^ (i & 7))) << 2) + (j & 3);
}

// ---------------------------------------------------------------- phase 1
// Shared memory of the intra-chunk kernel (bytes).
constexpr int kP1R1 = 0;        // 36 KiB: [Ktilde; Qtilde] -> A, T fp32 -> L^T, V^T -> W^T, U^T
constexpr int kP1R2 = 36864;    // 40 KiB: column versions -> H, T*B, scratch X
constexpr int kP1E = 77824;     // 32 KiB: E fp32 [64][128]
constexpr int kP1Beta = 110592; // 64 floats
constexpr int kP1Bar = 110848;  // mbarrier
constexpr int kP1Tmem = 110856; // TMEM base address
constexpr int kP1Smem = 110880;
constexpr int kAS = 65;         // row stride (floats) of A and T in shared memory

// (I, J) of column version v = I (I + 1) / 2 + J.
__device__ __forceinline__ constexpr int ver_I(int v) { return v < 1 ? 0 : v < 3 ? 1 : v < 6 ? 2 : 3; }
__device__ __forceinline__ constexpr int ver_J(int v) { return v - ver_I(v) * (ver_I(v) + 1) / 2; }

__device__ __forceinline__ float ldbf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

__global__ void __launch_bounds__(128, 2)
tc_intra_chunk(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
               const __nv_bfloat16 *__restrict__ v, const float *__restrict__ g,
               const float *__restrict__ beta, float scale, const ChunkEntry *__restrict__ table,
               long long nslots, int H, unsigned char *__restrict__ ws, int *__restrict__ status) {
    extern __shared__ __align__(1024) unsigned char sm[];
    // Heads vary fastest across the grid, so CTAs resident together read whole
    // token rows ([token][head][channel]) rather than one head's slice of many.
    const int h = blockIdx.x;
    const long long slot = (long long)blockIdx.z * gridDim.y + blockIdx.y;
    if (slot >= nslots) return;
    const ChunkEntry ce = table[slot];
    if (ce.seq < 0) return;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int c = tid;  // key/value channel owned by this thread
    unsigned char *R1 = sm + kP1R1;
    unsigned char *R2 = sm + kP1R2;
    float *Es = reinterpret_cast<float *>(sm + kP1E);
    float *beta_s = reinterpret_cast<float *>(sm + kP1Beta);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + kP1Bar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + kP1Tmem);
    unsigned char *reg = ws + ((size_t)slot * H + h) * TcRegion::bytes;

    if (warp == 0) tmem_alloc<256>(tslot);
    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_fence_init();
    }

    const int len = ce.len;
    const size_t row0 = (size_t)ce.bos * H + h;  // token row of the chunk's first token
    auto at = [&](int i) { return (row0 + (size_t)i * H) * D + c; };

    // ---- cumulative log-decay, block references, E_i = exp(G_i - G_r(block i)).
    float G[C];
#pragma unroll
    for (int i = 0; i < C; ++i) G[i] = i < len ? __ldg(g + at(i)) : 0.f;
#pragma unroll
    for (int i = 1; i < C; ++i) G[i] += G[i - 1];
    const float Rf[4] = {G[7], G[23], G[39], G[55]};
    const float Gend = G[C - 1];
#pragma unroll
    for (int i = 0; i < C; ++i) Es[i * D + c] = __expf(G[i] - Rf[i >> 4]);
    float P[4], Y[4];
#pragma unroll
    for (int I = 0; I < 4; ++I) {
        P[I] = __expf(Rf[I]);         // exp(G_r(I)) from the chunk start
        Y[I] = __expf(Gend - Rf[I]);  // exp(G_n - G_r(I))
    }
    float X[4][4];  // exp(G_r(I) - G_r(J)), J <= I
#pragma unroll
    for (int I = 0; I < 4; ++I)
#pragma unroll
        for (int J = 0; J < 4; ++J) X[I][J] = J < I ? __expf(Rf[I] - Rf[J]) : 1.f;
    if (tid < C) beta_s[tid] = tid < len ? beta[row0 + (size_t)tid * H] : 0.f;

    // ---- operands of the gated K K^T / Q K^T product, and Kbar^T.
    // A operand (MN-major, 128 rows x 128 channels): rows i = Ktilde_i, 64+i = s Qtilde_i.
    // B operand (MN-major, 160 rows): row 16 v(I,J) + (j mod 16) = k_j exp(G_r(I) - G_j).
#pragma unroll
    for (int ig = 0; ig < 8; ++ig) {
        float kk[8], qq[8], e[8], f[8], t8[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int i = ig * 8 + r;
            kk[r] = i < len ? ldbf(k + at(i)) : 0.f;
            qq[r] = i < len ? scale * ldbf(q + at(i)) : 0.f;
            e[r] = Es[i * D + c];
            f[r] = 1.f / e[r];
        }
        const uint32_t a_off = (uint32_t)ig * kA1Sbo + (uint32_t)(c >> 3) * 128u + (uint32_t)(c & 7) * 16u;
#pragma unroll
        for (int r = 0; r < 8; ++r) t8[r] = kk[r] * e[r];
        *reinterpret_cast<uint4 *>(R1 + a_off) = pack8(t8);
#pragma unroll
        for (int r = 0; r < 8; ++r) t8[r] = qq[r] * e[r];
        *reinterpret_cast<uint4 *>(R1 + a_off + 8 * kA1Sbo) = pack8(t8);
        const int J = ig >> 1;
#pragma unroll
        for (int I = 0; I < 4; ++I) {
            if (I < J) continue;
            const int n0 = 16 * (I * (I + 1) / 2 + J) + (ig & 1) * 8;
#pragma unroll
            for (int r = 0; r < 8; ++r) t8[r] = kk[r] * f[r] * X[I][J];
            *reinterpret_cast<uint4 *>(R2 + (uint32_t)(n0 >> 3) * kA1Sbo + (uint32_t)(c >> 3) * 128u +
                                       (uint32_t)(c & 7) * 16u) = pack8(t8);
        }
        // Kbar^T row c, tokens 8 ig .. 8 ig + 7: k_j exp(G_n - G_j).
#pragma unroll
        for (int r = 0; r < 8; ++r) t8[r] = kk[r] * f[r] * Y[J];
        *reinterpret_cast<uint4 *>(reg + TcRegion::A2 + kmaj(c, ig * 8, kA2Lbo, kA2Sbo)) = pack8(t8);
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

    if (tid == 0) {
        const uint32_t id = idesc_bf16(128, 160, 1, 1);
#pragma unroll
        for (int s = 0; s < D / 16; ++s)
            mma_bf16(tmem, desc(smem_u32(R1) + s * 2 * kA1Lbo, kA1Lbo, kA1Sbo),
                     desc(smem_u32(R2) + s * 2 * kA1Lbo, kA1Lbo, kA1Sbo), id, s > 0);
        commit(bar);
    }
    bool ok = __syncthreads_and(mbar_wait(bar, 0));
    fence_after();
    if (!ok) goto fail;

    {
        // ---- A (fp32, for the solve) and H (bf16 B operand, K-major [i][j]).
        float *As = reinterpret_cast<float *>(R1);
        float *Ts = reinterpret_cast<float *>(R1 + 16640);
        unsigned char *Hs = R2;                  // K-major [N = i][K = j]: LBO 1024, SBO 128
        unsigned char *TBs = R2 + 8192;          // same layout
        float *Xs = reinterpret_cast<float *>(R2 + 16384);
        const int i = tid & 63, Iblk = i >> 4;
        const bool isH = tid >= 64;
        const float bi = beta_s[i];
#pragma unroll
        for (int vv = 0; vv < 10; ++vv) {
            const bool warp_uses = (warp & 1) ? vv >= 3 : vv < 3;  // warp-uniform
            if (!warp_uses) continue;
            float x[16];
            tmem_ld16(tmem + lane_base + vv * 16, x);
            tmem_wait_ld();
            if (ver_I(vv) != Iblk) continue;
            const int J = ver_J(vv);
            if (!isH) {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int j = 16 * J + jj;
                    As[i * kAS + j] = j < i ? -bi * x[jj] : 0.f;
                }
            } else {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    float t8[8];
#pragma unroll
                    for (int r = 0; r < 8; ++r) t8[r] = (16 * J + 8 * hf + r <= i) ? x[8 * hf + r] : 0.f;
                    *reinterpret_cast<uint4 *>(Hs + kmaj(i, 16 * J + 8 * hf, 1024, 128)) = pack8(t8);
                }
            }
        }
#pragma unroll
        for (int J = 0; J < 4; ++J) {
            if (J <= Iblk) continue;
            if (!isH) {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) As[i * kAS + 16 * J + jj] = 0.f;
            } else {
                const uint4 z = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4 *>(Hs + kmaj(i, 16 * J, 1024, 128)) = z;
                *reinterpret_cast<uint4 *>(Hs + kmaj(i, 16 * J + 8, 1024, 128)) = z;
            }
        }
        fence_before();
        __syncthreads();

        // ---- T = (I - A)^{-1}. Diagonal 16x16 blocks by forward substitution
        // (thread = column), then T_IJ = T_II sum_{K=J}^{I-1} A_IK T_KJ by levels.
        if (tid < 64) {
            const int I = tid >> 4, col = tid;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int ii = 16 * I + r;
                float acc = ii == col ? 1.f : 0.f;
#pragma unroll
                for (int rr = 0; rr < r; ++rr) acc += As[ii * kAS + 16 * I + rr] * x[rr];
                x[r] = ii < col ? 0.f : acc;
                Ts[ii * kAS + col] = x[r];
            }
        }
        __syncthreads();
#pragma unroll
        for (int L = 1; L <= 3; ++L) {
            const int npairs = 4 - L;
            for (int o = tid; o < npairs * 256; o += 128) {
                const int p = o >> 8, r = (o >> 4) & 15, cc = o & 15;
                const int J = p, I = J + L;
                float acc = 0.f;
                for (int K = J; K < I; ++K)
#pragma unroll
                    for (int kk = 0; kk < 16; ++kk)
                        acc += As[(16 * I + r) * kAS + 16 * K + kk] * Ts[(16 * K + kk) * kAS + 16 * J + cc];
                Xs[p * 256 + r * 16 + cc] = acc;
            }
            __syncthreads();
            for (int o = tid; o < npairs * 256; o += 128) {
                const int p = o >> 8, r = (o >> 4) & 15, cc = o & 15;
                const int J = p, I = J + L;
                float acc = 0.f;
#pragma unroll
                for (int kk = 0; kk < 16; ++kk)
                    acc += Ts[(16 * I + r) * kAS + 16 * I + kk] * Xs[p * 256 + kk * 16 + cc];
                Ts[(16 * I + r) * kAS + 16 * J + cc] = acc;
            }
            __syncthreads();
        }

        // ---- T B (bf16 B operand, K-major [N = i][K = j]).
        {
            const int hf = tid >> 6;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const int jb = 32 * hf + 8 * q4;
                float t8[8];
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int j = jb + r;
                    t8[r] = j <= i ? Ts[i * kAS + j] * beta_s[j] : 0.f;
                }
                *reinterpret_cast<uint4 *>(TBs + kmaj(i, jb, 1024, 128)) = pack8(t8);
            }
        }
        __syncthreads();

        // ---- L^T and V^T (A operands, K-major [M = channel][K = token]) into R1.
#pragma unroll
        for (int jg = 0; jg < 8; ++jg) {
            float t8[8], u8[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int j = jg * 8 + r;
                t8[r] = j < len ? ldbf(k + at(j)) * Es[j * D + c] * P[jg >> 1] : 0.f;
                u8[r] = j < len ? ldbf(v + at(j)) : 0.f;
            }
            *reinterpret_cast<uint4 *>(R1 + kmaj(c, jg * 8, kA2Lbo, kA2Sbo)) = pack8(t8);
            *reinterpret_cast<uint4 *>(R1 + 16384 + kmaj(c, jg * 8, kA2Lbo, kA2Sbo)) = pack8(u8);
        }
        fence_async_smem();
        fence_before();
        __syncthreads();
        fence_after();
        if (tid == 0) {
            const uint32_t id = idesc_bf16(128, 64, 0, 0);
#pragma unroll
            for (int s = 0; s < C / 16; ++s) {
                const uint64_t b = desc(smem_u32(TBs) + s * 2 * 1024, 1024, 128);
                mma_bf16(tmem + 0, desc(smem_u32(R1) + s * 2 * kA2Lbo, kA2Lbo, kA2Sbo), b, id, s > 0);
                mma_bf16(tmem + 64, desc(smem_u32(R1 + 16384) + s * 2 * kA2Lbo, kA2Lbo, kA2Sbo), b, id,
                         s > 0);
            }
            commit(bar);
        }
        ok = __syncthreads_and(mbar_wait(bar, 1));
        fence_after();
        if (!ok) goto fail;

        // ---- W, U: workspace copies for the state pass, and W^T, U^T operands.
        float *Uw = reinterpret_cast<float *>(reg + TcRegion::U) + (size_t)(c / kTN) * C * kTN;
#pragma unroll
        for (int part = 0; part < 4; ++part) {
            float w16[16], u16[16];
            tmem_ld16(tmem + lane_base + 16 * part, w16);
            tmem_ld16(tmem + lane_base + 64 + 16 * part, u16);
            tmem_wait_ld();
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int i0 = 16 * part + 8 * hf;
                const uint4 wp = pack8(w16 + 8 * hf);
                *reinterpret_cast<uint4 *>(reg + TcRegion::A1 + mnmaj(i0, c, kA1Lbo, kA1Sbo)) = wp;
                *reinterpret_cast<uint4 *>(R1 + kmaj(c, i0, kA2Lbo, kA2Sbo)) = wp;
                *reinterpret_cast<uint4 *>(R1 + 16384 + kmaj(c, i0, kA2Lbo, kA2Sbo)) = pack8(u16 + 8 * hf);
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) Uw[slab_idx(16 * part + r, c % kTN)] = u16[r];
        }
        fence_async_smem();
        fence_before();
        __syncthreads();
        fence_after();
        if (tid == 0) {
            const uint32_t id = idesc_bf16(128, 64, 0, 0);
#pragma unroll
            for (int s = 0; s < C / 16; ++s) {
                const uint64_t b = desc(smem_u32(Hs) + s * 2 * 1024, 1024, 128);
                mma_bf16(tmem + 128, desc(smem_u32(R1) + s * 2 * kA2Lbo, kA2Lbo, kA2Sbo), b, id, s > 0);
                mma_bf16(tmem + 192, desc(smem_u32(R1 + 16384) + s * 2 * kA2Lbo, kA2Lbo, kA2Sbo), b, id,
                         s > 0);
            }
            commit(bar);
        }
        ok = __syncthreads_and(mbar_wait(bar, 0));
        fence_after();
        if (!ok) goto fail;

        // ---- Q' = Qbar - H W (rows 64..127 of A1) and Ou = H U.
        float *Ow = reinterpret_cast<float *>(reg + TcRegion::Ou) + (size_t)(c / kTN) * C * kTN;
#pragma unroll
        for (int part = 0; part < 4; ++part) {
            float d16[16], o16[16], t16[16];
            tmem_ld16(tmem + lane_base + 128 + 16 * part, d16);
            tmem_ld16(tmem + lane_base + 192 + 16 * part, o16);
            tmem_wait_ld();
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const int ii = 16 * part + r;
                const float qb = ii < len ? scale * ldbf(q + at(ii)) * Es[ii * D + c] * P[part] : 0.f;
                t16[r] = qb - d16[r];
                Ow[slab_idx(ii, c % kTN)] = o16[r];
            }
            *reinterpret_cast<uint4 *>(reg + TcRegion::A1 + mnmaj(64 + 16 * part, c, kA1Lbo, kA1Sbo)) =
                pack8(t16);
            *reinterpret_cast<uint4 *>(reg + TcRegion::A1 + mnmaj(64 + 16 * part + 8, c, kA1Lbo, kA1Sbo)) =
                pack8(t16 + 8);
        }
        reinterpret_cast<float *>(reg + TcRegion::Gam)[c] = __expf(Gend);
    }
    fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc<256>(tmem);
    return;

fail:
    if (tid == 0) atomicExch(status, (int)KDA_ERR_TIMEOUT);
    mbar_wait(bar, 0);  // bounded: let any MMA still in flight finish before freeing TMEM
    mbar_wait(bar, 1);
    fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc<256>(*tslot);
}

// ---------------------------------------------------------------- phase 2
constexpr int kBufBytes = 66560;  // one chunk's A1, A2, U slab, Ou slab, gamma (65 KiB)
constexpr int kBufA2 = 32768, kBufU = 49152, kBufOu = 57344, kBufGam = 65536;
constexpr uint32_t kLoadBytes = 32768 + 16384 + 8192 + 8192 + 512;
constexpr int kP2B1 = 2 * kBufBytes;            // S (hi | lo) bf16, MN-major [K = ch][N = 64]
constexpr int kP2B2 = kP2B1 + 16384;            // Z hi, Z lo bf16, MN-major [K = token][N = 32]
constexpr int kP2Bar = kP2B2 + 8192;            // 3 mbarriers
constexpr int kP2Tmem = kP2Bar + 24;
constexpr int kP2Smem = kP2Tmem + 8;
constexpr uint32_t kB1Lbo = 128, kB1Sbo = 2048;
constexpr uint32_t kB2Lbo = 128, kB2Sbo = 1024;

__global__ void __launch_bounds__(128, 1)
tc_state_pass(const unsigned char *__restrict__ ws, const int *__restrict__ seq_first_slot,
              const int32_t *__restrict__ cu_seqlens, int T_fixed, const float *init_state,
              __nv_bfloat16 *__restrict__ out, float *final_state, int H, int *__restrict__ status) {
    extern __shared__ __align__(1024) unsigned char sm[];
    const int n = blockIdx.x, h = blockIdx.y, jt = blockIdx.z, j0 = jt * kTN;
    const int tid = threadIdx.x, warp = tid >> 5;
    int bos, len;
    if (cu_seqlens) {
        bos = cu_seqlens[n];
        len = cu_seqlens[n + 1] - bos;
    } else {
        bos = n * T_fixed;
        len = T_fixed;
    }
    const int nchunks = (len + C - 1) / C;
    const int slot0 = seq_first_slot[n];
    unsigned char *B1 = sm + kP2B1;
    unsigned char *B2 = sm + kP2B2;
    uint64_t *bar_load = reinterpret_cast<uint64_t *>(sm + kP2Bar);  // [2]
    uint64_t *bar_mma = bar_load + 2;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + kP2Tmem);

    // Thread c owns state row c of the slab, columns j0 .. j0 + 31.
    const int c = tid;
    const size_t st_off = (((size_t)n * H + h) * D + c) * D + j0;
    float S[kTN];
    if (init_state) {
#pragma unroll
        for (int j = 0; j < kTN; j += 4) {
            const float4 t = *reinterpret_cast<const float4 *>(init_state + st_off + j);
            S[j] = t.x; S[j + 1] = t.y; S[j + 2] = t.z; S[j + 3] = t.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < kTN; ++j) S[j] = 0.f;
    }
    auto put_state = [&]() {
        // B1 rows n = j (hi) and 32 + j (lo), K-row = channel c.
#pragma unroll
        for (int jg = 0; jg < kTN / 8; ++jg) {
            float hi[8], lo[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const float x = S[8 * jg + r];
                hi[r] = __bfloat162float(__float2bfloat16_rn(x));
                lo[r] = x - hi[r];
            }
            *reinterpret_cast<uint4 *>(B1 + mnmaj(8 * jg, c, kB1Lbo, kB1Sbo)) = pack8(hi);
            *reinterpret_cast<uint4 *>(B1 + mnmaj(kTN + 8 * jg, c, kB1Lbo, kB1Sbo)) = pack8(lo);
        }
    };
    put_state();

    if (warp == 0) tmem_alloc<128>(tslot);
    if (tid == 0) {
        mbar_init(bar_load, 1);
        mbar_init(bar_load + 1, 1);
        mbar_init(bar_mma, 1);
        mbar_fence_init();
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

    auto issue_load = [&](int ch, int b) {
        const unsigned char *r = ws + ((size_t)(slot0 + ch) * H + h) * TcRegion::bytes;
        unsigned char *dst = sm + b * kBufBytes;
        mbar_expect_tx(bar_load + b, kLoadBytes);
        bulk_g2s(dst, r + TcRegion::A1, 32768, bar_load + b);
        bulk_g2s(dst + kBufA2, r + TcRegion::A2, 16384, bar_load + b);
        bulk_g2s(dst + kBufU, r + TcRegion::U + (size_t)jt * C * kTN * 4, C * kTN * 4, bar_load + b);
        bulk_g2s(dst + kBufOu, r + TcRegion::Ou + (size_t)jt * C * kTN * 4, C * kTN * 4, bar_load + b);
        bulk_g2s(dst + kBufGam, r + TcRegion::Gam, 512, bar_load + b);
    };
    if (tid == 0 && nchunks > 0) issue_load(0, 0);

    uint32_t mma_phase = 0;
    bool ok = true;
    for (int ch = 0; ch < nchunks; ++ch) {
        const int b = ch & 1;
        unsigned char *buf = sm + b * kBufBytes;
        if (tid == 0 && ch + 1 < nchunks) issue_load(ch + 1, b ^ 1);
        ok = __syncthreads_and(mbar_wait(bar_load + b, (ch >> 1) & 1));
        if (!ok) break;
        // [W S; Q' S] with S = S_hi + S_lo: N = 64 (hi columns 0-31, lo 32-63).
        if (tid == 0) {
            fence_after();
            const uint32_t id = idesc_bf16(128, 2 * kTN, 1, 1);
#pragma unroll
            for (int s = 0; s < D / 16; ++s)
                mma_bf16(tmem, desc(smem_u32(buf) + s * 2 * kA1Lbo, kA1Lbo, kA1Sbo),
                         desc(smem_u32(B1) + s * 2 * kB1Lbo, kB1Lbo, kB1Sbo), id, s > 0);
            commit(bar_mma);
        }
        ok = __syncthreads_and(mbar_wait(bar_mma, mma_phase));
        mma_phase ^= 1;
        fence_after();
        if (!ok) break;
        {
            float hi[16], lo[16], d[kTN];
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                tmem_ld16(tmem + lane_base + 16 * part, hi);
                tmem_ld16(tmem + lane_base + kTN + 16 * part, lo);
                tmem_wait_ld();
#pragma unroll
                for (int r = 0; r < 16; ++r) d[16 * part + r] = hi[r] + lo[r];
            }
            const int i = tid & 63;
            if (tid < 64) {
                const float *Us = reinterpret_cast<const float *>(buf + kBufU);
#pragma unroll
                for (int jg = 0; jg < kTN / 8; ++jg) {
                    float zh[8], zl[8];
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const int j = 8 * jg + r;
                        const float z = Us[slab_idx(i, j)] - d[j];
                        zh[r] = __bfloat162float(__float2bfloat16_rn(z));
                        zl[r] = z - zh[r];
                    }
                    *reinterpret_cast<uint4 *>(B2 + mnmaj(8 * jg, i, kB2Lbo, kB2Sbo)) = pack8(zh);
                    *reinterpret_cast<uint4 *>(B2 + 4096 + mnmaj(8 * jg, i, kB2Lbo, kB2Sbo)) = pack8(zl);
                }
            } else {
                const float *Os = reinterpret_cast<const float *>(buf + kBufOu);
                const int clen = min(C, len - ch * C);
                if (i < clen) {
                    __nv_bfloat16 *dst = out + ((size_t)(bos + ch * C + i) * H + h) * D + j0;
#pragma unroll
                    for (int jg = 0; jg < kTN / 8; ++jg) {
                        float o8[8];
#pragma unroll
                        for (int r = 0; r < 8; ++r) o8[r] = Os[slab_idx(i, 8 * jg + r)] + d[8 * jg + r];
                        *reinterpret_cast<uint4 *>(dst + 8 * jg) = pack8(o8);
                    }
                }
            }
        }
        fence_async_smem();
        fence_before();
        __syncthreads();
        if (tid == 0) {
            fence_after();
            const uint32_t id = idesc_bf16(128, kTN, 0, 1);
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int s = 0; s < C / 16; ++s)
                    mma_bf16(tmem + 2 * kTN,
                             desc(smem_u32(buf + kBufA2) + s * 2 * kA2Lbo, kA2Lbo, kA2Sbo),
                             desc(smem_u32(B2 + part * 4096) + s * 2 * kB2Lbo, kB2Lbo, kB2Sbo), id,
                             part > 0 || s > 0);
            commit(bar_mma);
        }
        ok = __syncthreads_and(mbar_wait(bar_mma, mma_phase));
        mma_phase ^= 1;
        fence_after();
        if (!ok) break;
        {
            const float gam = reinterpret_cast<const float *>(buf + kBufGam)[c];
            float d16[16];
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                tmem_ld16(tmem + lane_base + 2 * kTN + 16 * part, d16);
                tmem_wait_ld();
#pragma unroll
                for (int r = 0; r < 16; ++r) S[16 * part + r] = gam * S[16 * part + r] + d16[r];
            }
            put_state();
        }
        fence_async_smem();
        fence_before();
        __syncthreads();
    }
    if (!ok) {
        if (tid == 0) atomicExch(status, (int)KDA_ERR_TIMEOUT);
        // Bounded waits for the copies and MMAs that may still be in flight.
        mbar_wait(bar_load, 0);
        mbar_wait(bar_load + 1, 0);
        mbar_wait(bar_mma, mma_phase);
    } else if (final_state) {
#pragma unroll
        for (int j = 0; j < kTN; j += 4)
            *reinterpret_cast<float4 *>(final_state + st_off + j) = make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
    fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc<128>(tmem);
}

}  // namespace

size_t tc_region_bytes() { return TcRegion::bytes; }

cudaError_t launch_prefill_tc(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, float scale, const float *init_state,
                              const int32_t *cu_seqlens, void *out, float *final_state,
                              int T_fixed, int H, int num_seqs, long long slots,
                              const ChunkEntry *table, const int *seq_first_slot,
                              unsigned char *region, int *status, cudaStream_t stream,
                              cudaEvent_t *events) {
    cudaError_t err = cudaFuncSetAttribute(tc_intra_chunk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kP1Smem);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(tc_state_pass, cudaFuncAttributeMaxDynamicSharedMemorySize, kP2Smem);
    if (err != cudaSuccess) return err;
    if ((err = mark(events, 1, stream)) != cudaSuccess) return err;
    if (slots > 0) {
        tc_intra_chunk<<<head_slot_grid(H, slots), 128, kP1Smem, stream>>>(
            static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
            static_cast<const __nv_bfloat16 *>(v), g, beta, scale, table, slots, H, region, status);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    if ((err = mark(events, 2, stream)) != cudaSuccess) return err;
    if (num_seqs > 0) {
        tc_state_pass<<<dim3(num_seqs, H, D / kTN), 128, kP2Smem, stream>>>(
            region, seq_first_slot, cu_seqlens, T_fixed, init_state,
            static_cast<__nv_bfloat16 *>(out), final_state, H, status);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    return mark(events, 3, stream);
}

}  // namespace kda
