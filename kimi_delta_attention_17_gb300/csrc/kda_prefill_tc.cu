// Tensor-core chunkwise prefill for bf16 q/k/v with d_k = d_v = 128 (sm_103a:
// tcgen05.mma with TMEM accumulators, tensor-map and 1-D bulk copies).
//
// The algebra is the chunkwise form of "Understanding Kimi Delta Attention"
// (sections "The triangular system" and "Putting the chunks together"):
//
//   phase 1 (every chunk and head in parallel; persistent, one CTA per SM,
//   whose two halves work on consecutive items: the elementwise steps of
//   item n + 1 beside the solve and W of item n):
//     G      in-chunk cumulative log-decay (registers, one thread per channel)
//     A, H   decay-gated K K^T and Q K^T, from ONE tcgen05.mma (below)
//     T      (I - A)^{-1}: blocked forward substitution in fp32 shared memory
//     W = (T B) L                               one MMA, B = Diag(beta)
//     s Qbar, Kbar^T, exp(G_n)                  elementwise
//   phase 2 (one CTA per sequence, head and 32- or 64-column slab of the
//   state, chunks in order, state in registers, warp-specialised):
//     U = (T B) V                               one MMA, a chunk ahead
//     [s Qbar S; W S] = [s Qbar; W] S           one MMA, M = 128
//     Z = U - W S                               elementwise
//     S <- Diag(exp(G_n)) S + Kbar^T Z          one MMA
//     O = s Qbar S + H Z                        one MMA into the first one's rows
//   (with few (sequence, head) chains the chunks are cut into segments whose
//   affine maps are composed before the segments run in parallel: SegPass)
//
// Decay absorption with secondary chunking ("Kimi Delta Attention: a half-life
// per channel", section "What changes in the kernel"): the per-channel pair
// decay exp(G_i - G_j) factors through a reference r as
//     exp(G_i - G_r) * exp(G_r - G_j),
// which turns the gated products into plain matmuls of rescaled rows. Each
// 16-token block I of the chunk has its reference at its 8th token, r(I); a
// row i in block I is scaled by E_i = exp(G_i - G_r(I)) and a column j in
// block J <= I by exp(G_r(I) - G_r(J)) / E_j. Every factor that can exceed 1
// spans at most 8 tokens of one block's decay, so while no channel decays by
// more than kSteepNats within a 16-token block every factor stays far inside
// fp32 and bf16 range (the factors that shrink may underflow to zero, exactly
// where the true product is negligible). An item with a steeper block takes
// the steep-decay form: rows referenced to the point before their block,
// columns to their block's last token (every factor then <= 1), and the
// diagonal blocks, which no single reference splits safely, formed directly
// in fp32 with the pair decay exp(G_i - G_j). The
// ten (I, J) column versions stack into one B operand of 160 rows, and the
// K-tilde / Q-tilde rows into one A operand of 128 rows, so a single
// M=128, N=160, K=128 MMA yields every block of A (rows 0-63) and H (rows
// 64-127) at once; each row keeps the columns of its own versions.
//
// Operands are written by threads into no-swizzle canonical layouts: one
// thread per key channel writes 16-byte runs along the token axis (MN-major
// tiles when the contraction runs over channels, K-major when it runs over
// tokens). Accumulators are read back with tcgen05.ld (thread t = TMEM lane t).
#include <cstring>
#include <cuda.h>  // CUtensorMap (the encoder is fetched at run time; no libcuda link)

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

using namespace tc;

constexpr int D = 128;   // d_k = d_v on this path
constexpr int C = kChunk;
constexpr int kTN = 32;  // state columns per phase-2 CTA

// Workspace region of one (chunk slot, head), byte offsets. Everything a
// state-pass CTA needs from it is shared by the head's four CTAs and moves in
// one bulk copy (an SM completes about one bulk copy per 900 cycles whatever
// its size, up to 64 KiB: copies must be few and large); each CTA forms its
// own 32-column slab of U = (T B) V from (T B) here and the value rows it
// loads itself.
struct TcRegion {
    static constexpr size_t A1 = 0;        // [s Qbar; W] bf16, MN-major, 128 tokens x 128 ch
    static constexpr size_t A2 = 32768;    // Kbar^T bf16, K-major, 128 ch x 64 tokens
    static constexpr size_t Gam = 49152;   // fp32 [128] exp(G_n)
    static constexpr size_t HT = 49664;    // [H; T B] bf16, K-major [row][token j] (LBO 2048, SBO 128)
    static constexpr size_t bytes = 66048;
};
static_assert(TcRegion::bytes % 256 == 0, "regions stay 256-byte aligned");
// Descriptor strides of the workspace tiles (and of their shared-memory copies).
constexpr uint32_t kA1Lbo = 128, kA1Sbo = 2048;  // MN-major: channel cores adjacent
constexpr uint32_t kA2Lbo = 2048, kA2Sbo = 128;  // K-major: channel groups adjacent

// ---------------------------------------------------------------- phase 1
// Persistent: one CTA of 16 warps per SM walks the (chunk slot, head) items,
// heads fastest, as a two-stage pipeline over two items. Warps 0-7 (the
// elementwise side) take the raw rows of item n + 1 (q, k bf16 and g fp32:
// three tensor-map tiles in staging) to the MMA operands and the workspace
// rows that need no solve, then issue its A/H product; meanwhile warps 8-15
// (the solve side) read back item n's A and H, run the triangular solve and
// the W product and write the rest of its region. The elementwise pass is
// bound by instruction issue and the solve by its dependent stages (MMA round
// trips, barriers, a shuffle chain), so each fills the other's idle issue
// slots. Elementwise thread (c, hb) owns key/value channel c and the 16-token
// blocks hb and 3 - hb; solve-side warp w reads TMEM lanes 32 (w mod 4) to
// 32 (w mod 4) + 31. What the two sides hand over is double-buffered by item
// parity: the TMEM
// accumulators (two 256-column halves), L^T, beta and the steep flag.
constexpr int kP1Threads = 512;
constexpr int kP1E = 256, kP1S = 256;   // elementwise side: threads 0-255; solve side: 256-511
constexpr int kBarE = 1, kBarSv = 2;    // their named barriers
struct P1 {  // shared-memory offsets, bytes
    static constexpr int q = 0, k = 16384, g = 32768;  // staging rows of one chunk
    static constexpr int am = 65536;    // [Ktilde; s Qtilde] bf16, MN-major 128 x 128
    static constexpr int bm = 98304;    // column versions bf16, MN-major 160 x 128
    static constexpr int lt = 139264;   // [2] L^T bf16, K-major [channel][token], 16 KiB each
    static constexpr int As = 172032;   // fp32 [64][68]: A; the solve overwrites it with T
    static constexpr int TBs = 189440;  // bf16 K-major [i][j]: T Diag(beta)
    static constexpr int Ms = 197632;   // fp32 [6][16][kMS]: M_IK = T_II A_IK
    static constexpr int Rs = 205312;   // fp32 [3][16][kMS]: partial sums of T_IJ
    static constexpr int beta = 209152; // fp32 [2][64] by item parity
    static constexpr int bar = 209664;  // 10 mbarriers (see intra_chunk_body)
    static constexpr int tmem = 209744;
    static constexpr int flags = 209760;  // int [2] steep, by item parity; int error flag
    static constexpr int exch = 209776; // fp32 [2][4][128]: block totals and local references of G
    static constexpr int gsc = 213872;  // fp32 [64]: per-head log-decay of the item's tokens
    static constexpr int fac = 214128;  // fp32 [2 (k, q)][64]: reciprocal norms (q's times the scale)
    static constexpr int dg = 214640;   // fp32 [2 (A, H)][64][16]: diagonal blocks of steep items
    static constexpr int bytes = 222832;
    static constexpr int Ts = As;       // T (fp32 [64][68]) takes A's place
};
constexpr int kMS = 20;  // row stride (floats) of the M / R blocks: 8 rows hit 8 bank groups
static_assert(P1::As + 64 * 68 * 4 == P1::TBs && P1::Rs + 3 * 16 * kMS * 4 == P1::beta &&
              P1::lt + 2 * 16384 == P1::As && P1::dg + 2 * 64 * 16 * 4 == P1::bytes,
              "phase-1 shared-memory regions are disjoint");
static_assert(P1::bytes <= 232448, "phase-1 shared memory exceeds 227 KiB");
constexpr int kAS = 68;  // row stride (floats) of A and T: 16-byte rows, 8 rows hit 8 bank groups
// Largest total decay, in nats, of one channel over a 16-token block for which
// the block-centred references are used: every factor then stays within
// e^64 ~ 6e27, far inside fp32 and bf16 range. An item in which some channel's
// block decays more takes the steep-decay form.
constexpr float kSteepNats = 64.f;

// (I, J) of column version v = I (I + 1) / 2 + J.
__host__ __device__ constexpr int ver_I(int v) { return v < 1 ? 0 : v < 3 ? 1 : v < 6 ? 2 : 3; }
__host__ __device__ constexpr int ver_J(int v) { return v - ver_I(v) * (ver_I(v) + 1) / 2; }

__device__ __forceinline__ void st16(unsigned char *p, const float *x) {
    *reinterpret_cast<uint4 *>(p) = pack8(x);
}

// Phase 1 keeps its cumulative log-decays in base-2 units (nats times
// log2 e), so that every decay factor is one hardware 2^x.
constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Steep item (kSteepNats): the diagonal 16 x 16 blocks of A and H in fp32,
// sum_c x_ic k_jc 2^(G_ic - G_jc) (G in base-2 units) with the pair decay formed directly (its
// exponent is <= 0 wherever j <= i), into P1::dg as raw sums (the readback
// applies -beta and the causal masks). Reads the staged q, k rows, the
// reciprocal norms and the in-block log-decay prefixes that replaced g in
// staging. Elementwise-side thread t (t < 256): row i = t / 4 and the 32
// channels of group t mod 4; the four groups of a row combine by shuffles. Kept out of line: it runs only for steep items and the
// kernel's common path must stay within the instruction cache.
__device__ __noinline__ void steep_diagonal_blocks(unsigned char *sm, int tid, int len, int l2norm,
                                                   float scale) {
    const __nv_bfloat16 *qs = reinterpret_cast<const __nv_bfloat16 *>(sm + P1::q);
    const __nv_bfloat16 *ks = reinterpret_cast<const __nv_bfloat16 *>(sm + P1::k);
    const float *gG = reinterpret_cast<const float *>(sm + P1::g);
    const float *fac_s = reinterpret_cast<const float *>(sm + P1::fac);
    float *dgA = reinterpret_cast<float *>(sm + P1::dg), *dgH = dgA + 64 * 16;
    const int i = tid >> 2, cg = tid & 3, i0 = i & ~15;
    const float fki = l2norm ? fac_s[i] : 1.f, fqi = l2norm ? fac_s[C + i] : scale;
#pragma unroll 1
    for (int jj = 0; jj < 16; ++jj) {
        const int j = i0 + jj;
        const float fkj = j < len ? (l2norm ? fac_s[j] : 1.f) : 0.f;
        float a = 0.f, hq = 0.f;
#pragma unroll
        for (int hf = 0; hf < 4; ++hf) {
            const int c0 = 32 * cg + 8 * hf;
            const uint4 kiw = *reinterpret_cast<const uint4 *>(ks + i * D + c0);
            const uint4 qiw = *reinterpret_cast<const uint4 *>(qs + i * D + c0);
            const uint4 kjw = *reinterpret_cast<const uint4 *>(ks + j * D + c0);
            const float4 gi0 = *reinterpret_cast<const float4 *>(gG + i * D + c0);
            const float4 gi1 = *reinterpret_cast<const float4 *>(gG + i * D + c0 + 4);
            const float4 gj0 = *reinterpret_cast<const float4 *>(gG + j * D + c0);
            const float4 gj1 = *reinterpret_cast<const float4 *>(gG + j * D + c0 + 4);
            const uint32_t ki[4] = {kiw.x, kiw.y, kiw.z, kiw.w};
            const uint32_t qi[4] = {qiw.x, qiw.y, qiw.z, qiw.w};
            const uint32_t kj[4] = {kjw.x, kjw.y, kjw.z, kjw.w};
            const float gi[8] = {gi0.x, gi0.y, gi0.z, gi0.w, gi1.x, gi1.y, gi1.z, gi1.w};
            const float gj[8] = {gj0.x, gj0.y, gj0.z, gj0.w, gj1.x, gj1.y, gj1.z, gj1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t sh = (e & 1) ? 0u : 16u;  // element 2m sits in the low half
                const float kie = __uint_as_float((ki[e >> 1] << sh) & 0xFFFF0000u);
                const float qie = __uint_as_float((qi[e >> 1] << sh) & 0xFFFF0000u);
                const float kje = __uint_as_float((kj[e >> 1] << sh) & 0xFFFF0000u);
                const float w = kje * ex2(gi[e] - gj[e]);
                a += kie * w;
                hq += qie * w;
            }
        }
#pragma unroll
        for (int m = 1; m < 4; m <<= 1) {
            a += __shfl_xor_sync(0xffffffffu, a, m);
            hq += __shfl_xor_sync(0xffffffffu, hq, m);
        }
        if (cg == 0) {
            const bool in = i < len;
            dgA[i * 16 + jj] = in ? fki * fkj * a : 0.f;
            dgH[i * 16 + jj] = in ? fqi * fkj * hq : 0.f;
        }
    }
}

// Instances: kVar fixes the options at compile time, so that each common
// form is compiled without the code of the others (the kernel must stay
// within the instruction cache): 0 per-channel log-decay (KDA), 2 one
// log-decay per head (Gated DeltaNet), 3 no decay (DeltaNet), all with g
// holding log a and no normalisation; 4 per-channel decay from gate logits
// through the log-sigmoid with q and k normalised (the KDA layer's own
// prologue); 1 takes every option at run time.
constexpr int kVarChannel = 0, kVarRuntime = 1, kVarScalar = 2, kVarNone = 3, kVarGated = 4;
// How a phase-1 CTA walks the items: its rank among the phase-1 CTAs and
// their count; in the fused prefill also the ready flags it sets and the item
// order (ilv > 1: chunk-major over ilv fixed-length sequences of nch chunks
// each, so that chunk c of every sequence is ready at about the same time).
struct P1Walk {
    int rank, count;
    int *ready;  // [slot][H]: 1 once the item's region is written; NULL: no flags
    int ilv, nch;
};

// The item order's slot index -> the table slot.
__device__ __forceinline__ int p1_phys(const P1Walk &wk, int s) {
    return wk.ilv > 1 ? (s % wk.ilv) * wk.nch + s / wk.ilv : s;
}


// Phase 1 for the threads 0 .. kP1Threads - 1 of a CTA (its barriers count
// exactly those threads, so a larger CTA may run it with the rest idle).
//
// Hand-over between the two sides (mbarriers; phase k of a barrier pair
// [item parity] belongs to item 2 k + parity):
//   bar_ld       q, k of item n landed in staging (tensor-map copies)
//   bar_ldg      g of item n landed in staging (issued as soon as the item
//                before has summed its own, unless that item was steep)
//   bar_ah[2]    item n's A/H product done: the solve side may read it, the
//                elementwise side may overwrite the operands (am, bm)
//   bar_e[2]     the elementwise side is done with item n (beta, the steep
//                flag, L^T and its workspace rows written)
//   bar_w        the W product of the solve side's item done
//   bar_rb       item n's A/H read back (the steep blocks' scratch is free)
//   bar_sf[2]    the solve side is done with item n: its TMEM half, L^T and
//                beta slots may take item n + 2
template <int kVar>
__device__ __forceinline__ void intra_chunk_body(const CUtensorMap *tm_q, const CUtensorMap *tm_k,
                                                 const CUtensorMap *tm_g, const float *__restrict__ g_head,
                                                 Prologue pro, const float *__restrict__ beta, float scale,
                                                 const ChunkEntry *__restrict__ table,
                                                 const int *__restrict__ used_slots, long long nslots,
                                                 int H, unsigned char *__restrict__ ws,
                                                 int *__restrict__ status, const P1Walk wk) {
    extern __shared__ __align__(1024) unsigned char sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t *bar_ld = reinterpret_cast<uint64_t *>(sm + P1::bar);
    uint64_t *bar_ah = bar_ld + 1;
    uint64_t *bar_e = bar_ah + 2;
    uint64_t *bar_w = bar_e + 2;
    uint64_t *bar_rb = bar_w + 1;
    uint64_t *bar_sf = bar_rb + 1;
    uint64_t *bar_ldg = bar_sf + 2;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + P1::tmem);
    int *steep_s = reinterpret_cast<int *>(sm + P1::flags);
    volatile int *err = reinterpret_cast<volatile int *>(sm + P1::flags + 8);
    float *betas = reinterpret_cast<float *>(sm + P1::beta);
    // Slots [0, used) of the table hold every chunk, in order; the rest are empty.
    const int used = (int)min((long long)*used_slots, nslots);
    // Items are (slot, head) pairs, heads fastest; CTA b takes items b, b + grid,
    // ...: stepping by the grid in (slot, head) form keeps 64-bit divisions off
    // the item path. Both sides walk the same items.
    const int step_s = (int)(wk.count / H), step_h = (int)(wk.count % H);
    auto phys = [&](int s) { return p1_phys(wk, s); };
    auto advance = [&](int &sl, int &hh) {
        sl += step_s;
        hh += step_h;
        if (hh >= H) {
            hh -= H;
            ++sl;
        }
    };
    // Bounded waits: a completed phase returns at once; otherwise the CTA's
    // error flag is read first and the wait is skipped once either side has
    // given up. A timeout raises the flag and the call's status.
    auto wait = [&](uint64_t *bar, uint32_t parity) {
        if (mbar_test(bar, parity)) return true;
        if (*err) return false;
        if (!mbar_wait(bar, parity)) {
            *err = 1;
            atomicExch(status, (int)KDA_ERR_TIMEOUT);
            return false;
        }
        return true;
    };

    if (warp == 0) tmem_alloc<512>(tslot);
    if (tid == 0) {
        mbar_init(bar_ld, 1);
        mbar_init(bar_ldg, 1);
        mbar_init(bar_w, 1);
        mbar_init(bar_rb, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_ah + b, 1);
            mbar_init(bar_e + b, 1);
            mbar_init(bar_sf + b, 1);
        }
        *err = 0;
        mbar_fence_init();
    }
    fence_before();
    bar_sync(0, kP1Threads);
    fence_after();
    const uint32_t tmem = *tslot;

    if (kVar == kVarChannel) pro = Prologue{KDA_DECAY_CHANNEL, KDA_GATE_LOG, 0.f, 0};
    if (kVar == kVarScalar) pro = Prologue{KDA_DECAY_SCALAR, KDA_GATE_LOG, 0.f, 0};
    if (kVar == kVarNone) pro = Prologue{KDA_DECAY_NONE, KDA_GATE_LOG, 0.f, 0};
    if (kVar == kVarGated) pro = Prologue{KDA_DECAY_CHANNEL, KDA_GATE_LOGSIGMOID, 0.f, 1};

    if (tid < kP1E) {
        // ============================================ elementwise side
        // Channel c and blocks hb, 3 - hb: the earlier a block, the more
        // column versions it writes, so each thread takes one early and one late.
        const int c = tid & 127, hb = tid >> 7;
        // Operand descriptors, built once: a K step adds a constant to the
        // address field (byte address / 16).
        const uint64_t d_am = desc(smem_u32(sm + P1::am), kA1Lbo, kA1Sbo);
        const uint64_t d_bm = desc(smem_u32(sm + P1::bm), kA1Lbo, kA1Sbo);
        // One thread fetches an item: 3-D TMA tiles (128 channels x 1 head x
        // 64 tokens) land as dense [token][channel] rows, q and k on one
        // barrier and g on another. Tokens past the end of the tensor read as
        // zeros; tokens of the next sequence are masked by len.
        const bool g_tile = pro.decay == KDA_DECAY_CHANNEL;  // g arrives as a tile only per channel
        auto issue_qk = [&](int hh, const ChunkEntry e) {
            mbar_expect_tx(bar_ld, 64u * 2u * 256u);
            tma_load_3d(sm + P1::q, tm_q, 0, hh, e.bos, bar_ld);
            tma_load_3d(sm + P1::k, tm_k, 0, hh, e.bos, bar_ld);
        };
        auto issue_g = [&](int hh, const ChunkEntry e) {
            mbar_expect_tx(bar_ldg, 64u * 512u);
            tma_load_3d(sm + P1::g, tm_g, 0, hh, e.bos, bar_ldg);
        };
        // Each item's table entry and beta values are read one item ahead, so
        // that no global load latency sits on the item's path.
        auto beta_of = [&](int hh, const ChunkEntry &e) {
            return tid < C && tid < e.len ? beta[(size_t)(e.bos + tid) * H + hh] : 0.f;
        };
        // The per-head decay value of token tid (Gated DeltaNet form), read the
        // same way; it becomes log a (log_decay) when it is stored for its item.
        auto ghead_of = [&](int hh, const ChunkEntry &e) {
            return pro.decay == KDA_DECAY_SCALAR && tid < C && tid < e.len
                       ? g_head[(size_t)(e.bos + tid) * H + hh]
                       : 0.f;
        };
        float *gs = reinterpret_cast<float *>(sm + P1::g);
        const __nv_bfloat16 *qs = reinterpret_cast<const __nv_bfloat16 *>(sm + P1::q);
        const __nv_bfloat16 *ks = reinterpret_cast<const __nv_bfloat16 *>(sm + P1::k);
        float *gsc_s = reinterpret_cast<float *>(sm + P1::gsc);  // written one item ahead
        float *tot_s = reinterpret_cast<float *>(sm + P1::exch);
        float *ref_s = tot_s + 4 * D;
        float *fac_s = reinterpret_cast<float *>(sm + P1::fac);

        int sl = (int)(wk.rank / H), hc = (int)(wk.rank % H);  // this item
        ChunkEntry ce{};
        float bcur = 0.f;
        int ld_issued = 0, g_issued = 0, ah_issued = 0;  // copies / products issued (thread 0)
        // Fused prefill (thread 0): the ready flags of the two items in the
        // solve side's hands, by parity. Item n - 2's flag is released as soon
        // as the solve side is done with it (bar_sf, which this thread waits
        // for anyway); the region's writes by both sides precede that barrier
        // (this side's through its own barriers), so the release makes them
        // visible before the flag. A release waits for stores in flight to
        // reach L2, which this side's idle wait absorbs.
        long long flag0 = -1, flag1 = -1;  // even, odd items
        bool g_next = false;  // thread 0: the next item's g is on its way
        if (sl < used) {
            ce = table[phys(sl)];
            if (tid == 0) {
                issue_qk(hc, ce);
                ld_issued = 1;
                if (g_tile) {
                    issue_g(hc, ce);
                    g_issued = 1;
                }
            }
            bcur = beta_of(hc, ce);
            if (pro.decay == KDA_DECAY_SCALAR && tid < C)
                gsc_s[tid] = tid < ce.len ? log_decay(ghead_of(hc, ce), pro) : 0.f;
        }
        int sn = sl, hn = hc;  // the next item
        advance(sn, hn);
        ChunkEntry en = sn < used ? table[phys(sn)] : ce;
        bar_sync(kBarE, kP1E);  // the first item's per-head decays
        int n = 0;              // items done by this side
        while (sl < used) {
            const int len = ce.len;
            const int par = n & 1;
            int snn = sn, hnn = hn;  // the item after next
            ChunkEntry enn;
            float bn, gn;
            unsigned char *reg = ws + ((size_t)phys(sl) * H + hc) * TcRegion::bytes;
            if (g_tile) wait(bar_ldg, (uint32_t)par);  // a failure shows in the error flag after the barrier
            if (tid == 0) {
                // Item n - 2's TMEM half, L^T and beta slots, and the operands
                // item n - 1's product read, are free before anything is written.
                if (n >= 2 && wait(bar_sf + par, (uint32_t)((n - 2) >> 1) & 1) && wk.ready)
                    st_release_gpu(wk.ready + (par ? flag1 : flag0), 1);
                if (n >= 1) wait(bar_ah + (par ^ 1), (uint32_t)((n - 1) >> 1) & 1);
                const long long f = (long long)phys(sl) * H + hc;
                flag0 = par ? flag0 : f;
                flag1 = par ? f : flag1;
            }

            // Cumulative log-decay of channel c over each of the thread's two
            // blocks, kept in registers (G0, G1: in-block prefixes) for the
            // factor loop, so that staging may take the next item's g as soon
            // as every thread has summed this one's. Block totals and in-block
            // references (token 7 of each block) go to the exchange, so that
            // every thread has the absolute references R_I = G_{16 I + 7} and
            // the chunk total. In-block factors need only the local prefixes
            // (the block's offset cancels in G_i - G_r).
            float G0[16], G1[16], accb[2];
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
                const int b = bb == 0 ? hb : 3 - hb;
                float *G = bb == 0 ? G0 : G1;
                float acc = 0.f;
                if (pro.decay == KDA_DECAY_CHANNEL && pro.gate == KDA_GATE_LOG) {
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        const int tok = 16 * b + t;
                        acc = fmaf(tok < len ? gs[tok * D + c] : 0.f, kLog2e, acc);
                        G[t] = acc;
                    }
                } else if (pro.decay == KDA_DECAY_CHANNEL) {
                    // Gate logits become log a in registers as they are summed;
                    // the 16 transforms are independent, so they issue back to back.
                    float gv[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t) gv[t] = gs[(16 * b + t) * D + c];
                    if (pro.gate == KDA_GATE_LOGSIGMOID) {
                        // log2 sigmoid(x) = min(x, 0) log2 e - log2(1 + 2^(-|x| log2 e)),
                        // already in the base-2 units of G.
#pragma unroll
                        for (int t = 0; t < 16; ++t)
                            gv[t] = fmaf(fminf(gv[t], 0.f), kLog2e, -lg2(1.f + ex2(-fabsf(gv[t]) * kLog2e)));
#pragma unroll
                        for (int t = 0; t < 16; ++t) {
                            acc += 16 * b + t < len ? gv[t] : 0.f;
                            G[t] = acc;
                        }
                    } else {
#pragma unroll
                        for (int t = 0; t < 16; ++t) gv[t] = pro.lower * __fdividef(1.f, 1.f + __expf(-gv[t]));
#pragma unroll
                        for (int t = 0; t < 16; ++t) {
                            acc = fmaf(16 * b + t < len ? gv[t] : 0.f, kLog2e, acc);
                            G[t] = acc;
                        }
                    }
                } else if (pro.decay == KDA_DECAY_SCALAR) {
                    // One decay per head: every channel's prefix is the same.
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        acc = fmaf(gsc_s[16 * b + t], kLog2e, acc);
                        G[t] = acc;
                    }
                } else {
#pragma unroll
                    for (int t = 0; t < 16; ++t) G[t] = 0.f;
                }
                tot_s[b * D + c] = acc;
                ref_s[b * D + c] = G[7];
                accb[bb] = acc;
            }
            // A block's total decay bounds every factor of its references (the
            // log-decay is non-increasing within the block); over kSteepNats
            // anywhere, the whole item takes the steep-decay form (the decision
            // is uniform over the side). The reads of staged g are ordered
            // before the copy that may refill it right after this barrier.
            fence_async_smem();
            const bool steep =
                bar_or(kBarE, kP1E, fminf(accb[0], accb[1]) < -kSteepNats * kLog2e) != 0;
            if (*err) break;
            // The next item's g, unless a steep item still needs staging's g
            // rows for its in-block prefixes.
            if (tid == 0 && g_tile && !steep && sn < used) {
                issue_g(hn, en);
                ++g_issued;
                g_next = true;
            }
            // The table entry of the item after next and the next item's beta,
            // read here: the next barrier is the whole factor pass away.
            advance(snn, hnn);
            enn = snn < used ? table[phys(snn)] : en;
            bn = sn < used ? beta_of(hn, en) : 0.f;
            gn = sn < used ? ghead_of(hn, en) : 0.f;
            if (tid < C) betas[par * C + tid] = bcur;
            if (tid == 0) steep_s[par] = steep ? 1 : 0;
            // References of every block for this channel, as cumulative
            // log-decays from the chunk start: rows (K-tilde, Q-tilde, L, Qbar)
            // are scaled relative to Rr, columns (the versions, Kbar) relative
            // to Rc. Normally both are the block's 8th token (no factor spans
            // more than 8 tokens). In a steep item rows take the point before
            // the block's first token and columns its last token, so that every
            // factor is exp(x) with x <= 0; the diagonal blocks, which no single
            // reference can split safely, are then formed directly below.
            float Rr[4], Rc[4], off = 0.f;
#pragma unroll
            for (int I = 0; I < 4; ++I) {
                const float rf = ref_s[I * D + c], tt = tot_s[I * D + c];
                Rr[I] = steep ? off : off + rf;
                Rc[I] = steep ? off + tt : off + rf;
                off += tt;
            }
            const float Gend = off;
            unsigned char *ltp = sm + P1::lt + par * 16384;
            wait(bar_ld, (uint32_t)par);  // q, k (a failure skips the rest below)
            if (pro.l2norm) {
                // Reciprocal norms of k and q per token (the query scale folded
                // in): two threads per (tensor, token) each sum 64 channels of
                // the staged row, in 16-byte pieces rotated by the token so that
                // a warp's reads spread over the banks; one shuffle combines them.
                const int pair = tid >> 1, part = tid & 1;
                const int tsr = pair >> 6, tok = pair & 63;  // tensor 0: k, 1: q
                const __nv_bfloat16 *row = (tsr ? qs : ks) + tok * D;
                float ss = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int piece = 8 * part + ((j + tok) & 7);  // 8 channels
                    const uint4 w = *reinterpret_cast<const uint4 *>(row + 8 * piece);
                    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float lo = __uint_as_float(u[e] << 16), hi = __uint_as_float(u[e] & 0xFFFF0000u);
                        ss += lo * lo + hi * hi;
                    }
                }
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                if (part == 0) fac_s[pair] = rsqrtf(ss + kL2Eps) * (tsr ? scale : 1.f);
                // Every thread reads the norms below; the rows are cleared past
                // a ragged chunk's length only after every norm has been summed.
                bar_sync(kBarE, kP1E);
            }
            if (len < C) {
                // A ragged chunk: the staged q, k rows past len (the next
                // sequence's, or zeros past the tensor) are cleared, each thread
                // its own entries, which are all it reads below.
                __nv_bfloat16 *qw = reinterpret_cast<__nv_bfloat16 *>(sm + P1::q);
                __nv_bfloat16 *kw = reinterpret_cast<__nv_bfloat16 *>(sm + P1::k);
#pragma unroll 1
                for (int bb = 0; bb < 2; ++bb) {
                    const int b = bb == 0 ? hb : 3 - hb;
                    for (int t = 16 * b; t < 16 * b + 16; ++t)
                        if (t >= len) {
                            qw[t * D + c] = __float2bfloat16(0.f);
                            kw[t * D + c] = __float2bfloat16(0.f);
                        }
                }
            }
            // Runtime loops over the thread's two blocks and their two 8-token
            // groups (one copy of the body keeps the kernel within the
            // instruction cache).
#pragma unroll 1
            for (int bb = 0; bb < 2; ++bb) {
                const int b = bb == 0 ? hb : 3 - hb;
                // Per-block constants: the block's references, exp of the row
                // one from the chunk start and of the column one to the chunk
                // end, and the factors exp(Rr_I - Rc_b) of the later blocks'
                // versions (the own block's version: 1, or 0 in a steep item).
                const float Rrs = b == 0 ? Rr[0] : b == 1 ? Rr[1] : b == 2 ? Rr[2] : Rr[3];
                const float Rcs = b == 0 ? Rc[0] : b == 1 ? Rc[1] : b == 2 ? Rc[2] : Rc[3];
                // The same references relative to the block start.
                const float refb = bb ? G1[7] : G0[7], totb = bb ? G1[15] : G0[15];
                const float Rlr = steep ? 0.f : refb, Rlc = steep ? totb : refb;
                // (The query scale s rides on the s Qbar rows' factor; the
                // solve side applies it to H.)
                const float Ps = ex2(Rrs), Ys = ex2(Gend - Rcs), PsQ = Ps * (pro.l2norm ? 1.f : scale);
                float Xv[4];
#pragma unroll
                for (int I = 0; I < 4; ++I) Xv[I] = I > b ? ex2(Rr[I] - Rcs) : (steep ? 0.f : 1.f);
#pragma unroll 1
                for (int ig = 0; ig < 2; ++ig) {
                    const int i0 = 16 * b + 8 * ig;  // first token of the group
                    float kv[8], qv[8], E[8], kF[8], t8[8], Gi[8];
#pragma unroll
                    for (int r = 0; r < 8; ++r)
                        Gi[r] = bb ? (ig ? G1[8 + r] : G1[r]) : (ig ? G0[8 + r] : G0[r]);
                    if (steep) {
                        // The in-block log-decay prefixes replace g in staging
                        // (each thread its own entries) for the diagonal blocks.
#pragma unroll
                        for (int r = 0; r < 8; ++r) gs[(i0 + r) * D + c] = Gi[r];
                    }
                    // Staged rows past len are zero (see above), so no masks here.
                    float fk8[8], fq8[8];  // the group's norm factors, four 16-byte loads
                    if (pro.l2norm) {
#pragma unroll
                        for (int h4 = 0; h4 < 2; ++h4) {
                            const float4 a4 = *reinterpret_cast<const float4 *>(fac_s + i0 + 4 * h4);
                            const float4 b4 = *reinterpret_cast<const float4 *>(fac_s + C + i0 + 4 * h4);
                            fk8[4 * h4] = a4.x; fk8[4 * h4 + 1] = a4.y; fk8[4 * h4 + 2] = a4.z; fk8[4 * h4 + 3] = a4.w;
                            fq8[4 * h4] = b4.x; fq8[4 * h4 + 1] = b4.y; fq8[4 * h4 + 2] = b4.z; fq8[4 * h4 + 3] = b4.w;
                        }
                    }
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const int i = i0 + r;
                        kv[r] = __bfloat162float(ks[i * D + c]);
                        qv[r] = __bfloat162float(qs[i * D + c]);
                        if (pro.l2norm) {
                            kv[r] *= fk8[r];
                            qv[r] *= fq8[r];
                        }
                        E[r] = ex2(Gi[r] - Rlr);
                        kF[r] = kv[r] * ex2(Rlc - Gi[r]);
                    }
#pragma unroll
                    for (int r = 0; r < 8; ++r) t8[r] = kv[r] * E[r];
                    st16(sm + P1::am + mnmaj(i0, c, kA1Lbo, kA1Sbo), t8);
#pragma unroll
                    for (int r = 0; r < 8; ++r) t8[r] = qv[r] * E[r];
                    st16(sm + P1::am + mnmaj(64 + i0, c, kA1Lbo, kA1Sbo), t8);
#pragma unroll
                    for (int I = 0; I < 4; ++I) {
                        if (I < b) continue;
                        const int n0 = 16 * (I * (I + 1) / 2 + b) + 8 * ig;
#pragma unroll
                        for (int r = 0; r < 8; ++r) t8[r] = kF[r] * Xv[I];
                        st16(sm + P1::bm + mnmaj(n0, c, kA1Lbo, kA1Sbo), t8);
                    }
#pragma unroll
                    for (int r = 0; r < 8; ++r) t8[r] = kF[r] * Ys;
                    st16(reg + TcRegion::A2 + kmaj(c, i0, kA2Lbo, kA2Sbo), t8);
#pragma unroll
                    for (int r = 0; r < 8; ++r) t8[r] = kv[r] * E[r] * Ps;
                    st16(ltp + kmaj(c, i0, kA2Lbo, kA2Sbo), t8);
                    // s Qbar, rows 0-63 of the state-pass operand [s Qbar; W].
#pragma unroll
                    for (int r = 0; r < 8; ++r) t8[r] = qv[r] * E[r] * PsQ;
                    st16(reg + TcRegion::A1 + mnmaj(i0, c, kA1Lbo, kA1Sbo), t8);
                }
            }
            if (hb == 0) reinterpret_cast<float *>(reg + TcRegion::Gam)[c] = ex2(Gend);
            if (steep) {
                // Steep item: the diagonal blocks formed directly, once the
                // solve side has read back the previous item's.
                if (tid == 0 && n >= 1) wait(bar_rb, (uint32_t)(n - 1) & 1);
                bar_sync(kBarE, kP1E);
                steep_diagonal_blocks(sm, tid, len, pro.l2norm, pro.l2norm ? scale : 1.f);
            }
            // The next item's per-head log-decays (this item's were read above).
            if (pro.decay == KDA_DECAY_SCALAR && tid < C)
                gsc_s[tid] = sn < used && tid < en.len ? log_decay(gn, pro) : 0.f;
            // The operands (and this side's reads of staging) are ordered before
            // the product and the copies that refill staging.
            fence_async_smem();
            bar_sync(kBarE, kP1E);
            if (tid == 0 && !*err) {
                fence_after();
                if (sn < used) {
                    issue_qk(hn, en);
                    ++ld_issued;
                    if (g_tile && !g_next) {
                        issue_g(hn, en);
                        ++g_issued;
                    }
                }
                g_next = false;
                // A / H = gated K K^T and Q K^T (M=128, N=160, K=128) into this
                // item's TMEM half.
                const uint32_t id = idesc_bf16(128, 160, 1, 1);
#pragma unroll
                for (int s = 0; s < D / 16; ++s)
                    mma_bf16(tmem + (uint32_t)(par * 256), d_am + s * (2 * kA1Lbo >> 4),
                             d_bm + s * (2 * kA1Lbo >> 4), id, s > 0);
                commit(bar_ah + par);
                ++ah_issued;
                mbar_arrive(bar_e + par);
            }
            ++n;
            sl = sn;
            hc = hn;
            ce = en;
            sn = snn;
            hn = hnn;
            en = enn;
            bcur = bn;
        }
        if (tid == 0) {
            // Bounded waits for copies and products that may still be in flight
            // after an error (at once otherwise).
            if (ld_issued > 0) mbar_wait(bar_ld, (uint32_t)(ld_issued - 1) & 1);
            if (g_issued > 0) mbar_wait(bar_ldg, (uint32_t)(g_issued - 1) & 1);
            if (ah_issued >= 1) mbar_wait(bar_ah + ((ah_issued - 1) & 1), (uint32_t)((ah_issued - 1) >> 1) & 1);
            // The flags of the last two items, once the solve side is done with
            // them (after an error the state pass gives up on its own).
            for (int k = n - 2; k < n; ++k)
                if (k >= 0 && wait(bar_sf + (k & 1), (uint32_t)(k >> 1) & 1) && wk.ready && !*err)
                    st_release_gpu(wk.ready + ((k & 1) ? flag1 : flag0), 1);
        }
    } else {
        // ============================================ solve side
        const int st = tid - kP1E, sw = st >> 5;  // thread and warp within the side
        const int quad = warp & 3;                // TMEM lane quadrant of this warp
        const uint32_t lane_base = (uint32_t)(32 * quad) << 16;
        const uint64_t d_lt = desc(smem_u32(sm + P1::lt), kA2Lbo, kA2Sbo);
        const uint64_t d_tb = desc(smem_u32(sm + P1::TBs), 1024, 128);
        float *As = reinterpret_cast<float *>(sm + P1::As);
        float *Ts = reinterpret_cast<float *>(sm + P1::Ts);
        float *Ms = reinterpret_cast<float *>(sm + P1::Ms);
        float *Rs = reinterpret_cast<float *>(sm + P1::Rs);
        int sl = (int)(wk.rank / H), hc = (int)(wk.rank % H);
        int n = 0, w_issued = 0;
        while (sl < used) {
            const int par = n & 1;
            unsigned char *reg = ws + ((size_t)phys(sl) * H + hc) * TcRegion::bytes;
            const uint32_t tb = tmem + (uint32_t)(par * 256);
            wait(bar_e + par, (uint32_t)(n >> 1) & 1);
            wait(bar_ah + par, (uint32_t)(n >> 1) & 1);
            fence_after();
            __syncwarp();  // tcgen05.ld is warp-collective: reconverge after the per-lane waits
            const bool steep = steep_s[par] != 0;
            const float *beta_n = betas + par * C;

            // ================= read back A (rows 0-63) and H (rows 64-127)
            {
                unsigned char *Hs = reg + TcRegion::HT;  // H goes straight to the workspace (rows 0-63)
                const int lr = 32 * quad + lane, i = lr & 63, Iblk = i >> 4;
                const bool isH = lr >= 64;
                const int g2 = sw >> 2;               // which of the quadrant's two warps
                const bool upper = (quad & 1) != 0;   // rows 32-63: blocks 2, 3
                const float bi = beta_n[i];
                // The query scale s (not applied to the staged Q-tilde rows unless
                // the normalisation folded it into q's norm factor).
                const float hsc = pro.l2norm ? 1.f : scale;
                // Versions of this warp's rows (blocks 0-1: versions 0-2; blocks
                // 2-3: versions 3-9), split between the quadrant's two warps; a
                // runtime loop keeps the code small enough for the instruction cache.
                const int v0 = upper ? (g2 ? 7 : 3) : (g2 ? 2 : 0);
                const int nv = upper ? (g2 ? 3 : 4) : (g2 ? 1 : 2);
#pragma unroll 1
                for (int k = 0; k < nv; ++k) {
                    const int vv = v0 + k;  // warp-uniform
                    float x[16];
                    tmem_ld16(tb + lane_base + vv * 16, x);
                    tmem_wait_ld();
                    if (ver_I(vv) != Iblk) continue;
                    const int J = ver_J(vv);
                    if (steep && J == Iblk) {  // formed directly in the elementwise pass
                        const float *src = reinterpret_cast<const float *>(sm + P1::dg) + (isH ? 64 * 16 : 0) + i * 16;
#pragma unroll
                        for (int f = 0; f < 4; ++f) {
                            const float4 d4 = *reinterpret_cast<const float4 *>(src + 4 * f);
                            x[4 * f] = d4.x; x[4 * f + 1] = d4.y; x[4 * f + 2] = d4.z; x[4 * f + 3] = d4.w;
                        }
                    }
                    if (!isH) {
#pragma unroll
                        for (int f = 0; f < 4; ++f) {
                            float a4[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int j = 16 * J + 4 * f + e;
                                a4[e] = j < i ? -bi * x[4 * f + e] : 0.f;
                            }
                            *reinterpret_cast<float4 *>(As + i * kAS + 16 * J + 4 * f) =
                                make_float4(a4[0], a4[1], a4[2], a4[3]);
                        }
                    } else {
#pragma unroll
                        for (int hf = 0; hf < 2; ++hf) {
                            float t8[8];
#pragma unroll
                            for (int r = 0; r < 8; ++r) t8[r] = (16 * J + 8 * hf + r <= i) ? hsc * x[8 * hf + r] : 0.f;
                            st16(Hs + kmaj(i, 16 * J + 8 * hf, kA2Lbo, kA2Sbo), t8);
                        }
                    }
                }
                if (g2 == 1) {
#pragma unroll
                    for (int J = 0; J < 4; ++J) {
                        if (J <= Iblk) continue;
                        if (!isH) {
#pragma unroll
                            for (int f = 0; f < 4; ++f)
                                *reinterpret_cast<float4 *>(As + i * kAS + 16 * J + 4 * f) =
                                    make_float4(0.f, 0.f, 0.f, 0.f);
                        } else {
                            const uint4 z = make_uint4(0, 0, 0, 0);
                            *reinterpret_cast<uint4 *>(Hs + kmaj(i, 16 * J, kA2Lbo, kA2Sbo)) = z;
                            *reinterpret_cast<uint4 *>(Hs + kmaj(i, 16 * J + 8, kA2Lbo, kA2Sbo)) = z;
                        }
                    }
                }
            }
            fence_before();
            bar_sync(kBarSv, kP1S);
            if (*err) break;
            if (st == 160) mbar_arrive(bar_rb);  // a warp that sits out the substitution

            // ================= T = (I - A)^{-1}, then T Diag(beta) as a bf16 operand.
            {
                // Block row I of the substitution (I - A_II) X = [A_I0 .. A_I,I-1 | I]
                // gives M_IK = T_II A_IK (K < I) and T_II = (I - A_II)^{-1} together:
                // 16 (I + 1) right-hand columns, 160 in all, four per group of four
                // threads (threads 0-159 of the side); each thread owns rows sub,
                // sub + 4, sub + 8, sub + 12 of its four columns. Once x_r is final
                // its owner broadcasts it (one shuffle per column) and every thread
                // pushes it into its later rows, so the dependent chain is one
                // shuffle and one FMA per row. T_II is written over A_II, so
                // every read of A precedes a barrier before the first write.
                const bool act = st < 160;  // whole warps
                const int g4 = st >> 2, sub = st & 3;
                const int I = g4 < 4 ? 0 : g4 < 12 ? 1 : g4 < 24 ? 2 : 3;
                const int cc = 4 * (g4 - (I == 0 ? 0 : I == 1 ? 4 : I == 2 ? 12 : 24));  // in [0, 16 (I + 1))
                const bool rhs_a = cc < 16 * I;  // columns of A_IK (K < I), or of the identity
                float a[4][16], xs[4][4];
                if (act) {
                    const float *Ab = As + 16 * I * kAS + 16 * I;
                    // This thread's rows of A_II (a[q][r] = A_II[4 q + sub][r],
                    // r < 4 q + sub; the rest unused).
#pragma unroll
                    for (int q = 0; q < 4; ++q)
#pragma unroll
                        for (int r4 = 0; r4 < 16; r4 += 4) {
                            if (r4 < 4 * q + 3) {
                                const float4 t = *reinterpret_cast<const float4 *>(Ab + (4 * q + sub) * kAS + r4);
                                a[q][r4] = t.x; a[q][r4 + 1] = t.y; a[q][r4 + 2] = t.z; a[q][r4 + 3] = t.w;
                            }
                        }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int row = 4 * q + sub;
                        if (rhs_a) {
                            const float4 t = *reinterpret_cast<const float4 *>(As + (16 * I + row) * kAS + cc);
                            xs[0][q] = t.x; xs[1][q] = t.y; xs[2][q] = t.z; xs[3][q] = t.w;
                        } else {
#pragma unroll
                            for (int k = 0; k < 4; ++k) xs[k][q] = row == cc + k - 16 * I ? 1.f : 0.f;
                        }
                    }
                }
                bar_sync(kBarSv, kP1S);
                if (act) {
#pragma unroll
                    for (int r = 0; r < 15; ++r) {
                        const int src = (lane & ~3) | (r & 3);
                        float xr[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) xr[k] = __shfl_sync(0xffffffffu, xs[k][r >> 2], src);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            if (4 * q + 3 > r && 4 * q + sub > r) {
#pragma unroll
                                for (int k = 0; k < 4; ++k) xs[k][q] += a[q][r] * xr[k];
                            }
                        }
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int row = 4 * q + sub;
                        float *dst = rhs_a ? Ms + (I * (I - 1) / 2 + (cc >> 4)) * 16 * kMS + row * kMS + (cc & 15)
                                           : Ts + (16 * I + row) * kAS + cc;
                        *reinterpret_cast<float4 *>(dst) = make_float4(xs[0][q], xs[1][q], xs[2][q], xs[3][q]);
                    }
                }
            }
            bar_sync(kBarSv, kP1S);
            {
                // Off-diagonal blocks: with M_IK = T_II A_IK (K < I), block row I of
                // (I - A) T = I gives T_IJ = sum_{K = J}^{I - 1} M_IK T_KJ. The
                // substitution above formed the six M blocks. Written out,
                //   T_10 = M_10 T_00,  T_21 = M_21 T_11,  T_32 = M_32 T_22,
                //   T_20 = M_20 T_00 + M_21 T_10,
                //   T_31 = (M_31 + M_32 M_21) T_11,
                //   T_30 = (M_30 + M_32 M_20) T_00 + (M_31 + M_32 M_21) T_10,
                // so two dependent levels suffice: level 1 forms T_10, T_21, T_32,
                // R = M_20 T_00, U = M_30 + M_32 M_20 and V = M_31 + M_32 M_21
                // (six warps, one 16 x 16 product each, a 1 x 8 strip per thread:
                // row r, columns 8 hf .. 8 hf + 7); level 2 forms T_20 = R + M_21
                // T_10, T_31 = V T_11 and T_30 = U T_00 + V T_10 (four warps; T_30's
                // two products split by columns over two warps, 1 x 4 strips).
                auto mi = [](int I, int K) { return I * (I - 1) / 2 + K; };  // M block index, K < I
                auto Tb = [&](int I, int J) { return Ts + 16 * I * kAS + 16 * J; };
                auto Mb = [&](int I, int K) { return Ms + mi(I, K) * 16 * kMS; };
                float *Rb = Rs, *Ub = Rs + 16 * kMS, *Vb = Rs + 2 * 16 * kMS;
                // acc[0 .. 4 nq) += P (16 x 16, row stride kMS) row r x Q (row
                // stride qs) columns c0 .. c0 + 4 nq - 1; every load before the FMAs.
                auto prod = [](float *acc, const float *P, const float *Q, int qs, int r, int c0, int nq) {
#pragma unroll
                    for (int h8 = 0; h8 < 16; h8 += 8) {
                        float pm[8];
                        float4 qv[8][2];
#pragma unroll
                        for (int m0 = 0; m0 < 8; m0 += 4) {
                            const float4 pv = *reinterpret_cast<const float4 *>(P + r * kMS + h8 + m0);
                            pm[m0] = pv.x; pm[m0 + 1] = pv.y; pm[m0 + 2] = pv.z; pm[m0 + 3] = pv.w;
                        }
#pragma unroll
                        for (int e = 0; e < 8; ++e)
#pragma unroll
                            for (int u = 0; u < 2; ++u)
                                if (u < nq) qv[e][u] = *reinterpret_cast<const float4 *>(Q + (h8 + e) * qs + c0 + 4 * u);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
#pragma unroll
                            for (int u = 0; u < 2; ++u)
                                if (u < nq) {
                                    acc[4 * u] += pm[e] * qv[e][u].x; acc[4 * u + 1] += pm[e] * qv[e][u].y;
                                    acc[4 * u + 2] += pm[e] * qv[e][u].z; acc[4 * u + 3] += pm[e] * qv[e][u].w;
                                }
                    }
                };
                const int r = lane >> 1, hf = lane & 1;
                {   // level 1: warps 0-5
                    const float *P = nullptr, *Q = nullptr, *init = nullptr;
                    float *dst = nullptr;
                    int qs = kAS, ds = kAS;
                    switch (sw) {
                        case 0: P = Mb(1, 0); Q = Tb(0, 0); dst = Tb(1, 0); break;
                        case 1: P = Mb(2, 1); Q = Tb(1, 1); dst = Tb(2, 1); break;
                        case 2: P = Mb(3, 2); Q = Tb(2, 2); dst = Tb(3, 2); break;
                        case 3: P = Mb(2, 0); Q = Tb(0, 0); dst = Rb; ds = kMS; break;
                        case 4: P = Mb(3, 2); Q = Mb(2, 0); qs = kMS; init = Mb(3, 0); dst = Ub; ds = kMS; break;
                        case 5: P = Mb(3, 2); Q = Mb(2, 1); qs = kMS; init = Mb(3, 1); dst = Vb; ds = kMS; break;
                        default: break;
                    }
                    if (sw < 6) {
                        float acc[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[j] = init ? init[r * kMS + 8 * hf + j] : 0.f;
                        prod(acc, P, Q, qs, r, 8 * hf, 2);
                        *reinterpret_cast<float4 *>(dst + r * ds + 8 * hf) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                        *reinterpret_cast<float4 *>(dst + r * ds + 8 * hf + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
                    }
                }
                bar_sync(kBarSv, kP1S);
                if (sw < 2) {  // level 2: T_20 (warp 0), T_31 (warp 1)
                    float acc[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) acc[j] = sw == 0 ? Rb[r * kMS + 8 * hf + j] : 0.f;
                    if (sw == 0) prod(acc, Mb(2, 1), Tb(1, 0), kAS, r, 8 * hf, 2);
                    else prod(acc, Vb, Tb(1, 1), kAS, r, 8 * hf, 2);
                    float *dst = sw == 0 ? Tb(2, 0) : Tb(3, 1);
                    *reinterpret_cast<float4 *>(dst + r * kAS + 8 * hf) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                    *reinterpret_cast<float4 *>(dst + r * kAS + 8 * hf + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
                } else if (sw < 4) {  // level 2: T_30 columns 8 (sw - 2) .. + 7, a 1 x 4 strip per thread
                    const int c0 = 8 * (sw - 2) + 4 * hf;
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
                    prod(acc, Ub, Tb(0, 0), kAS, r, c0, 1);
                    prod(acc, Vb, Tb(1, 0), kAS, r, c0, 1);
                    *reinterpret_cast<float4 *>(Tb(3, 0) + r * kAS + c0) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                }
                bar_sync(kBarSv, kP1S);
            }
            {
                // Row i, columns jb .. jb + 15 of T Diag(beta): two 16-byte runs per thread,
                const int i = st & 63, jb = 16 * (st >> 6);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float t8[8];
#pragma unroll
                    for (int f = 0; f < 2; ++f) {
                        const float4 t = *reinterpret_cast<const float4 *>(Ts + i * kAS + jb + 8 * h + 4 * f);
                        const float tv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = jb + 8 * h + 4 * f + e;
                            t8[4 * f + e] = j <= i ? tv[e] * beta_n[j] : 0.f;
                        }
                    }
                    st16(sm + P1::TBs + kmaj(i, jb + 8 * h, 1024, 128), t8);
                    // and rows 64-127 of the workspace's [H; T B], from which each
                    // state-pass CTA forms its slab of U = (T B) V
                    st16(reg + TcRegion::HT + kmaj(64 + i, jb + 8 * h, kA2Lbo, kA2Sbo), t8);
                }
            }
            fence_async_smem();
            fence_before();
            bar_sync(kBarSv, kP1S);
            // ================= W = (T B) L, into the first 64 columns of the item's TMEM half
            if (st == 0 && !*err) {
                fence_after();
                const uint32_t id = idesc_bf16(128, 64, 0, 0);
                const uint64_t lo = (uint64_t)par * (16384 >> 4);
#pragma unroll
                for (int s = 0; s < C / 16; ++s)
                    mma_bf16(tb, d_lt + lo + s * (2 * kA2Lbo >> 4), d_tb + s * (2 * 1024 >> 4), id, s > 0);
                commit(bar_w);
                ++w_issued;
            }
            if (!wait(bar_w, (uint32_t)n & 1)) break;
            fence_after();
            __syncwarp();
            {
                // W^T (lane = channel c, column = token) -> rows 64-127 of [s Qbar; W];
                // warp (quadrant, h) reads tokens 32 h .. 32 h + 31 of its channels.
                const int c = 32 * quad + lane, t0 = 32 * (sw >> 2);
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    float x[16];
                    tmem_ld16(tb + lane_base + t0 + 16 * m, x);
                    tmem_wait_ld();
                    st16(reg + TcRegion::A1 + mnmaj(64 + t0 + 16 * m, c, kA1Lbo, kA1Sbo), x);
                    st16(reg + TcRegion::A1 + mnmaj(64 + t0 + 16 * m + 8, c, kA1Lbo, kA1Sbo), x + 8);
                }
            }
            fence_before();
            bar_sync(kBarSv, kP1S);
            // Every thread of the side has written its part of the region (and
            // read its TMEM): the half, L^T and beta slots may take item n + 2.
            if (st == 0) mbar_arrive(bar_sf + par);
            ++n;
            advance(sl, hc);
        }
        if (st == 0 && w_issued > 0) mbar_wait(bar_w, (uint32_t)(w_issued - 1) & 1);

    }
    fence_before();
    bar_sync(0, kP1Threads);
    if (warp == 0) tmem_dealloc<512>(tmem);
}

template <int kVar>
__global__ void __launch_bounds__(kP1Threads, 1)
tc_intra_chunk(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_g, const float *__restrict__ g_head, Prologue pro,
               const float *__restrict__ beta, float scale, const ChunkEntry *__restrict__ table,
               const int *__restrict__ used_slots, long long nslots, int H,
               unsigned char *__restrict__ ws, int *__restrict__ status) {
    intra_chunk_body<kVar>(&tm_q, &tm_k, &tm_g, g_head, pro, beta, scale, table, used_slots, nslots, H,
                           ws, status, P1Walk{(int)blockIdx.x, (int)gridDim.x, nullptr, 1, 0});
}

// ---------------------------------------------------------------- phase 2
// One CTA per (sequence, head, TN-column slab of the state) and, with the
// segmented pass, per segment: TN = 32 (four CTAs of 608 threads per head) in
// the two-launch prefill, TN = 64 (two CTAs of 512 threads) in the fused one
// and in tc_state_pass64. Compute thread t of warp w = t / 32 owns TMEM lane /
// state row 32 (w % 4) + (t % 32) and a group of the slab's columns (the warp
// roles below).
// Per chunk, with S the state entering it:
//                  U  = (T B) V                 (formed a chunk ahead)
//   round trip 1:  D1 = [s Qbar; W] S          (rows 0-63: Qbar S, 64-127: W S)
//                  Z  = U - W S                 (lanes 64-127)
//   round trip 2:  D2 = Kbar^T Z,  D1[0:64] += H Z
//                  S <- Diag(exp G_n) S + D2,  O = D1[0:64] = s Qbar S + H Z
// ("Understanding Kimi Delta Attention", "The token outputs" and "One state
// crosses the chunk boundary"). S and Z enter the MMAs as bf16 hi + lo pairs.
// Warp roles, 32-column slabs: warps 0-15 compute. Warp 16's lane 0 issues
// the two products on the chain of dependent steps, and the warp keeps the
// named barriers with the compute warps. Warp 17's lane 0 issues the copies
// of the chunk tiles and warp 18's lane 0 the products off the chain (U a
// chunk ahead, H Z), both paced by mbarriers alone: an MMA's issue holds its
// thread while the tensor pipe is busy (about 60 cycles per M = 128, K = 16
// step), and a bulk copy's issue can too, which must not delay a named
// barrier. (Two roles in one warp would stall each other: a suspended wait
// holds the whole warp.)
// 64-column slabs (the fused prefill): 12 compute warps (three column groups
// of 24, 24 and 16 columns), warp 12 the chain and warp 13 the copies; the
// chain warp issues U and H Z as well (a warp of their own measured the same
// chunk period: the Z and state-update windows cover their issue). The fused
// kernel then fits in 16 warps: with more, one SM sub-partition holds five
// warps and the register file caps every thread at 96 registers, which slows
// phase 1.
constexpr int kP2Threads = 16 * 32 + 96;   // the 32-column state pass
constexpr int kFusedThreads = kP1Threads;  // the fused kernel (16 warps)
constexpr int kBarZ = 1, kBarS = 2;       // named barriers: Z written, state written
constexpr int kBarO = 3;                  // named barrier of the output warps (fused gate)
// A chunk's tiles sit in three rings, by lifetime:
//   X  [s Qbar; W], the first product's A operand: free once it completes; 2 deep.
//   K  Kbar^T and gamma: free once the second product completes; 2 deep.
//   H  [H; T B] and this CTA's TN columns of the chunk's value rows (bf16
//      MN-major, K = token, N = column: the B operand of U), wanted a chunk
//      early (U is formed a chunk ahead) and free once H Z (without outputs:
//      U) completes; 3 deep.
// A bulk copy fills an X or K slot; a bulk copy and a tensor-map copy an H slot.
constexpr int kXBufs = 2, kKBufs = 2, kHBufs = 3;
constexpr int kXBytes = (int)TcRegion::A2;                                 // 32 KiB
constexpr uint32_t kKCopy = (uint32_t)(TcRegion::HT - TcRegion::A2);      // Kbar^T, gamma
constexpr int kKGam = (int)(TcRegion::Gam - TcRegion::A2);
constexpr int kKBytes = ((int)kKCopy + 1023) / 1024 * 1024;              // 17 KiB
constexpr uint32_t kHTBytes = (uint32_t)(TcRegion::bytes - TcRegion::HT);  // 16 KiB
static_assert(kKCopy % 16 == 0 && kHTBytes % 16 == 0 && TcRegion::HT % 16 == 0,
              "bulk copies move 16-byte units from 16-byte boundaries");
constexpr uint32_t kBvLbo = 128, kBvSbo = 1024;  // value rows as an MN-major B operand
constexpr uint32_t kB1Lbo = 128, kB1Sbo = 2048;
constexpr uint32_t kB2Lbo = 128, kB2Sbo = 1024;
// mbarriers: X landed[2] and free[2], K landed[2] and free[2], H landed[3] and
// free[3]; first product, second product, H Z product, U product[2] (by chunk
// parity: U of the next chunk can complete before a compute thread waits for
// this chunk's), and the first product as the off-chain warp sees it (two
// arrivals: the product's commit and that lane's own, made once it has seen
// the phase before, so the barrier never runs a phase ahead of the lane).
constexpr int kP2NBar = 2 * (kXBufs + kKBufs + kHBufs) + 6;

// Shared memory and TMEM of the TN-column state pass (byte offsets; operand
// tiles 1 KiB aligned).
template <int TN>
struct P2L {
    static constexpr uint32_t kVBytes = C * TN * 2;
    static constexpr int kHBytes = (int)((kHTBytes + kVBytes + 1023) / 1024 * 1024);
    static constexpr int kK = kXBufs * kXBytes;
    static constexpr int kH = kK + kKBufs * kKBytes;
    static constexpr int kB1 = kH + kHBufs * kHBytes;  // S (hi | lo) bf16, MN-major [K = ch][N = 2 TN]
    static constexpr int kB2 = kB1 + D * 2 * TN * 2;   // [Z_hi | Z_lo] bf16, MN-major [K = token][N = 2 TN]
    static constexpr int kBar = kB2 + C * 2 * TN * 2;
    static constexpr int kTmem = kBar + 8 * kP2NBar;
    static constexpr int kErr = kTmem + 4;
    // Fused output gate (TN = 32 only, a 4-CTA cluster): three mbarriers (the
    // partial sums of a chunk's rows from the four CTAs have arrived, one per
    // chunk parity; the chunk's gate logits have landed), this CTA's per-row
    // partials of its four column groups, the four CTAs' per-row partials (two
    // chunk parities), and the gate logits of this CTA's columns for one chunk
    // (bf16 [64 tokens][TN], a tensor-map tile: global loads would hold the
    // output warps at their next named barrier until they return).
    static constexpr int kRedBar = (kErr + 4 + 7) / 8 * 8;
    static constexpr int kLoc = (kRedBar + 24 + 15) / 16 * 16;  // fp32 [4 column groups][64 rows]
    static constexpr int kRed = kLoc + 1024;                    // fp32 [2 parities][D / TN CTAs][64 rows]
    static constexpr int kZ = (kRed + 2 * (D / TN) * 64 * 4 + 127) / 128 * 128;
    static constexpr uint32_t kZBytes = C * TN * 2;
    static constexpr int kSmem = TN == 32 ? kZ + (int)kZBytes : kErr + 4;
    // TMEM columns: D1 alternates between [0, 2 TN) and [2 TN, 4 TN) from
    // chunk to chunk (the token outputs of chunk n are read while chunk n + 1's
    // first product runs); D2 = Kbar^T Z at [4 TN, 6 TN); U at [6 TN, 8 TN),
    // by chunk parity.
    static constexpr int kD2Col = 4 * TN, kUCol = 6 * TN, kCols = 8 * TN;
    static_assert(kB1 % 1024 == 0 && kB2 % 1024 == 0 && kHBytes % 1024 == 0, "operand tiles 1 KiB aligned");
    static_assert(kRedBar % 8 == 0 && kRed % 16 == 0 && kZ % 128 == 0, "gate buffers misaligned");
    static_assert(kSmem <= 232448, "phase-2 shared memory exceeds 227 KiB");
};
static_assert(kKBytes % 1024 == 0 && kXBytes % 1024 == 0, "operand tiles 1 KiB aligned");
constexpr uint32_t kRedBytes = (D / kTN) * 64 * 4;  // row partials a CTA receives per chunk (TN = 32)
constexpr int kGateCluster = D / kTN;                // CTAs of a head's state = the cluster

// Which chunks a state-pass launch walks. The serial pass is one segment of
// every chunk. The segmented pass (a chunk-level parallel prefix over the
// affine chunk maps S -> (Diag(gamma) - Kbar^T W) S + Kbar^T U) cuts each
// sequence into P segments of L chunks and runs two launches:
//  * transfer (segments 0 .. P-2): segment 0 runs from the true initial state
//    with outputs and stores its end state as the state entering segment 1;
//    segment p >= 1 runs its d_v tiles from a zero state (E_p) and d_k more
//    "identity" tiles from identity columns with U = 0 (M_p), without
//    outputs, into xfer;
//  * final (segments 1 .. P-1), after seg_combine: each segment runs from the
//    state entering it, with outputs; the last one writes the final state.
// sigmoid(z) = (1 + tanh(z / 2)) / 2 with the hardware tanh approximation
// (one transcendental instead of an exponential and a reciprocal; its error,
// below 1e-3 relative, is far inside the bf16 output's rounding).
__device__ __forceinline__ float sigmoid_fast(float z) {
    float th;
    asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(0.5f * z));
    return fmaf(0.5f, th, 0.5f);
}

// The output gate and RMS normalisation fused into the state pass's output
// write (z == NULL: plain outputs): out = w o / sqrt(mean(o^2) + eps) sigmoid(z)
// per (token, head) over the d_v channels ("Understanding Kimi Delta
// Attention", closing remarks: output gating and RMS normalisation).
struct OutGate {
    const __nv_bfloat16 *z;  // gate logits [tokens][H][D], or NULL (read through tm_z)
    const float *w;          // [D] per-channel weight, or NULL (ones)
    float eps;
};

struct SegPass {
    int L;         // chunks per segment
    int P;         // segments per sequence (1: the serial pass)
    int p_lo, np;  // segments of this launch: p_lo .. p_lo + np - 1
    int transfer;  // 1: transfer launch, 0: outputs launch
    float *xfer;   // [seq][H][P][D][2 D]: E_p in columns 0 .. D-1, M_p in D .. 2D-1
    float *enter;  // [seq][H][P][D][D]: the state entering segment p
};

// The state pass for one CTA: vblock is its index in the launch's grid order;
// `ready` (fused prefill) holds the flags phase 1 sets once a (slot, head)
// region is written, NULL when phase 1 has finished before the launch.
template <int TN>
__device__ __forceinline__ void state_pass_body(
    const unsigned char *__restrict__ ws, const int *__restrict__ seq_first_slot,
    const int *__restrict__ seq_order, const int32_t *__restrict__ cu_seqlens, int T_fixed,
    const float *init_state, __nv_bfloat16 *__restrict__ out, float *final_state, int H,
    int *__restrict__ status, const SegPass sp, const OutGate og_in, const CUtensorMap *tm_z,
    const CUtensorMap *tm_v, int vblock, const int *ready) {
    using L = P2L<TN>;
    // Compute warps: the four lane quadrants times CG column groups; a group
    // takes NP 8-column pieces of the slab (the last one may take fewer). With
    // 64-column slabs the Z rows (lanes 64-127, quadrants 2 and 3) take two more
    // warps (CW + 2, CW + 3) and four groups of 16 columns, which shortens the
    // Z step on the chain; rows 0-63 keep three groups (24, 24, 16).
    constexpr int CW = TN == kTN ? 16 : 12;
    constexpr int CG = CW / 4;
    constexpr int NP = (TN / 8 + CG - 1) / CG;
    constexpr int NJ = 8 * NP;                        // slab columns a compute thread holds, at most
    constexpr int kMma = CW, kCopy = CW + 1, kSideW = CW + 2;  // warp roles
    constexpr int kNComp = TN == kTN ? CW : CW + 2;   // compute warps
    constexpr int ZP = TN == kTN ? 1 : 2;             // pieces of a Z-row thread (lanes 64-127)
    constexpr int kSync = kNComp * 32 + 32;           // compute warps + MMA warp
    constexpr bool kSide = TN == kTN;     // U and H Z from their own warp
    extern __shared__ __align__(1024) unsigned char sm[];
    const OutGate og = TN == kTN ? og_in : OutGate{nullptr, nullptr, 0.f};
    const bool gated = og.z != nullptr;
    // A call whose chunk table was refused (or that already failed) does
    // nothing; the decision is taken once for the whole CTA. With the fused
    // output gate the CTA is one of a cluster and stays for the cluster
    // barriers, walking no chunk.
    const bool refused = __syncthreads_or(threadIdx.x == 0 && *status != 0) != 0;
    if (refused && !gated) return;
    // 1-D grid, sequences slowest in seq_order (longest first), then heads,
    // then segments, then the column tiles of one head and segment (adjacent:
    // they read the same tiles). A transfer launch has 2 D / TN tiles: the
    // d_v tiles, then the identity tiles.
    constexpr int kTiles = D / TN;
    const int tiles = sp.transfer ? 2 * kTiles : kTiles;
    const int per_h = sp.np * tiles, per_seq = H * per_h;
    const int rank = vblock / per_seq, rem = vblock - rank * per_seq;
    const int h = rem / per_h, rem2 = rem - h * per_h;
    const int p = sp.p_lo + rem2 / tiles, jt = rem2 - (rem2 / tiles) * tiles;
    const bool ident = jt >= kTiles;
    const int j0 = (ident ? jt - kTiles : jt) * TN;
    // Segment 0 of a transfer launch starts from the true initial state: it
    // needs no map, so its identity tiles have nothing to do.
    if (sp.transfer && p == 0 && ident) return;
    const bool outputs = !sp.transfer || p == 0;
    // The H ring is read by U (not in identity tiles) and by H Z (with outputs).
    const bool has_h = outputs || !ident;
    const int n = seq_order[rank];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int bos, len;
    if (cu_seqlens) {
        bos = cu_seqlens[n];
        len = cu_seqlens[n + 1] - bos;
    } else {
        bos = n * T_fixed;
        len = T_fixed;
    }
    const int all_chunks = (len + C - 1) / C;
    const int c0 = (int)min((long long)all_chunks, (long long)p * sp.L);
    const int nchunks = refused ? 0 : min(all_chunks - c0, sp.L);  // this segment's chunks
    const int slot0 = seq_first_slot[n] + c0;
    // Where the state comes from and where it goes, row r, columns j0 + js:
    const size_t nh = (size_t)n * H + h;
    const float *st_src = nullptr;  // NULL: zero (or identity columns)
    float *st_dst = nullptr;
    size_t dst_row = D;
    if (p == 0) {
        if (init_state) st_src = init_state + nh * D * D;
    } else if (!sp.transfer) {
        st_src = sp.enter + (nh * sp.P + p) * D * D;
    }
    if (sp.transfer) {
        if (p == 0) {
            st_dst = sp.enter + (nh * sp.P + 1) * D * D;
        } else {
            st_dst = sp.xfer + (nh * sp.P + p) * D * 2 * D + (ident ? D : 0);
            dst_row = 2 * D;
        }
    } else if (p == sp.P - 1 && final_state) {
        st_dst = final_state + nh * D * D;
    }
    unsigned char *B1 = sm + L::kB1;
    unsigned char *B2 = sm + L::kB2;
    uint64_t *bar_xl = reinterpret_cast<uint64_t *>(sm + L::kBar);  // [kXBufs] X tiles landed
    uint64_t *bar_xf = bar_xl + kXBufs;                              // [kXBufs] X tiles consumed
    uint64_t *bar_kl = bar_xf + kXBufs;                              // [kKBufs] K tiles landed
    uint64_t *bar_kf = bar_kl + kKBufs;                              // [kKBufs] K tiles consumed
    uint64_t *bar_hl = bar_kf + kKBufs;                              // [kHBufs] H tiles landed
    uint64_t *bar_hf = bar_hl + kHBufs;                              // [kHBufs] H tiles consumed
    uint64_t *bar_m1 = bar_hf + kHBufs;                              // first product done
    uint64_t *bar_m2 = bar_m1 + 1;                                   // second product done
    uint64_t *bar_m3 = bar_m2 + 1;                                   // H Z product done
    uint64_t *bar_u = bar_m3 + 1;                                    // [2] U product done
    uint64_t *bar_m1s = bar_u + 2;                                   // first product, off-chain warp
    uint64_t *red_full = reinterpret_cast<uint64_t *>(sm + L::kRedBar);  // [2] row partials arrived
    uint64_t *z_full = red_full + 2;                                     // gate logits landed
    float *loc = reinterpret_cast<float *>(sm + L::kLoc);
    float *red = reinterpret_cast<float *>(sm + L::kRed);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + L::kTmem);
    volatile int *err = reinterpret_cast<volatile int *>(sm + L::kErr);
    // Bounded waits. A phase that has completed returns at once; otherwise the
    // CTA's error flag is read first (a volatile shared read costs about as
    // much as a barrier test, so it stays off the path of waits that succeed
    // at once) and the wait is skipped once any warp has given up. A timeout
    // raises the flag and the call's status.
    auto wait = [&](uint64_t *bar, uint32_t parity) {  // false: gave up, or skipped after an error
        if (mbar_test(bar, parity)) return true;
        if (*err) return false;
        if (!mbar_wait(bar, parity)) {
            *err = 1;
            atomicExch(status, (int)KDA_ERR_TIMEOUT);
            return false;
        }
        return true;
    };
    auto spin = [&](uint64_t *bar, uint32_t parity) {  // the same, polling first
        if (mbar_poll(bar, parity) || *err) return;
        if (!mbar_wait(bar, parity)) {
            *err = 1;
            atomicExch(status, (int)KDA_ERR_TIMEOUT);
        }
    };

    // Compute-thread coordinates: TMEM lane / state row r, slab columns js .. js + NJ - 1.
    const bool compute = warp < CW || (TN != kTN && warp >= CW + 2);
    const bool zq = TN != kTN && (warp & 2) != 0;  // a Z-row warp of the 64-column pass
    const int r = 32 * (warp & 3) + lane, cgi = warp >> 2;
    const int js = TN == kTN ? 8 * NP * cgi : zq ? 16 * cgi : 24 * cgi;
    const int np = !compute ? 0 : TN == kTN ? min(NP, TN / 8 - NP * cgi) : zq ? 2 : (cgi < 2 ? 3 : 2);
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    float S[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) S[j] = ident && r == j0 + js + j ? 1.f : 0.f;
    auto put_state = [&]() {  // B1 rows js + j (hi) and TN + js + j (lo), K-row r
#pragma unroll
        for (int q = 0; q < NP; ++q) if (q < np) {
            uint4 hi, lo;
            split8(S + 8 * q, hi, lo);
            *reinterpret_cast<uint4 *>(B1 + mnmaj(js + 8 * q, r, kB1Lbo, kB1Sbo)) = hi;
            *reinterpret_cast<uint4 *>(B1 + mnmaj(TN + js + 8 * q, r, kB1Lbo, kB1Sbo)) = lo;
        }
    };
    if (compute) {
        if (st_src) {
            const float *src = st_src + (size_t)r * D + j0 + js;
#pragma unroll
            for (int q = 0; q < 2 * NP; ++q) if (q < 2 * np) {
                const float4 t4 = *reinterpret_cast<const float4 *>(src + 4 * q);
                S[4 * q] = t4.x; S[4 * q + 1] = t4.y; S[4 * q + 2] = t4.z; S[4 * q + 3] = t4.w;
            }
        }
        put_state();
    }
    if (warp == 0) tmem_alloc<L::kCols>(tslot);
    if (tid == 0) {
        // One arrival each, but two for the off-chain view of the first product.
        for (int i = 0; i < kP2NBar; ++i) mbar_init(bar_xl + i, bar_xl + i == bar_m1s ? 2 : 1);
        if (gated) {
            // Each chunk's phase: one local arrival (with the expected bytes,
            // 4 CTAs x 64 rows x 4 B) and the peers' asynchronous stores.
            for (int i = 0; i < 2; ++i) mbar_init(red_full + i, 1);
            mbar_init(z_full, 1);
        }
        *err = 0;
        mbar_fence_init();
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    // The first two chunks' phases expect their bytes, and the peers' barriers
    // are initialised, before anyone sends.
    if (gated && tid == 0)
        for (int i = 0; i < 2 && i < nchunks && !refused; ++i) mbar_expect_tx(red_full + i, kRedBytes);
    if (gated) cluster_sync();
    const uint32_t tmem = *tslot;

    // Chunk ch lives in slot ch % kXBufs of X (and likewise K, H) and is that
    // slot's (ch / kXBufs)-th use: its copies complete the phase of parity
    // (ch / kXBufs) & 1 of the slot's "landed" barrier, and its release the
    // phase of the same parity of the "free" one.
    if (warp == kCopy) {
        if (lane == 0) {
            // Chunk c's copies go out as their slots free, in the order the
            // slots free: H (chunk c - 3's last product), X (chunk c - 2's
            // first), K (chunk c - 2's second). In the fused prefill the
            // chunk's region is waited for first.
            int nx = 0, nk = 0, nhh = 0;  // copies issued per ring
            for (int ch = 0; ch < nchunks; ++ch) {
                const size_t slot = (size_t)(slot0 + ch);
                if (ready) {
                    const int *f = ready + slot * H + h;
                    bool got = false;
                    for (uint32_t it = 0; it < (1u << 22); ++it) {
                        if (ld_acquire_gpu(f) != 0) {
                            got = true;
                            break;
                        }
                        if ((it & 63) == 63 && (*err || *reinterpret_cast<volatile int *>(status) != 0))
                            break;
                        __nanosleep(256);
                    }
                    if (!got) {
                        *err = 1;
                        atomicCAS(status, 0, (int)KDA_ERR_TIMEOUT);
                        break;
                    }
                    fence_async_global();
                }
                const unsigned char *rg = ws + (slot * H + h) * TcRegion::bytes;
                if (has_h) {
                    if (ch >= kHBufs && !wait(bar_hf + ch % kHBufs, (uint32_t)(ch / kHBufs - 1) & 1)) break;
                    unsigned char *dst = sm + L::kH + (ch % kHBufs) * L::kHBytes;
                    uint64_t *bar = bar_hl + ch % kHBufs;
                    mbar_expect_tx(bar, kHTBytes + (ident ? 0u : L::kVBytes));
                    bulk_g2s(dst, rg + TcRegion::HT, kHTBytes, bar);
                    if (!ident) tma_load_3d(dst + kHTBytes, tm_v, 0, bos + (c0 + ch) * C, (h * D + j0) / 8, bar);
                    nhh = ch + 1;
                }
                if (ch >= kXBufs && !wait(bar_xf + ch % kXBufs, (uint32_t)(ch / kXBufs - 1) & 1)) break;
                mbar_expect_tx(bar_xl + ch % kXBufs, (uint32_t)kXBytes);
                bulk_g2s(sm + (ch % kXBufs) * kXBytes, rg, (uint32_t)kXBytes, bar_xl + ch % kXBufs);
                nx = ch + 1;
                if (ch >= kKBufs && !wait(bar_kf + ch % kKBufs, (uint32_t)(ch / kKBufs - 1) & 1)) break;
                mbar_expect_tx(bar_kl + ch % kKBufs, kKCopy);
                bulk_g2s(sm + L::kK + (ch % kKBufs) * kKBytes, rg + TcRegion::A2, kKCopy, bar_kl + ch % kKBufs);
                nk = ch + 1;
            }
            // Every copy lands before the CTA exits (bounded; a slot's last
            // use is the newest phase of its barrier).
            for (int cc = nx > kXBufs ? nx - kXBufs : 0; cc < nx; ++cc)
                mbar_wait(bar_xl + cc % kXBufs, (uint32_t)(cc / kXBufs) & 1);
            for (int cc = nk > kKBufs ? nk - kKBufs : 0; cc < nk; ++cc)
                mbar_wait(bar_kl + cc % kKBufs, (uint32_t)(cc / kKBufs) & 1);
            for (int cc = nhh > kHBufs ? nhh - kHBufs : 0; cc < nhh; ++cc)
                mbar_wait(bar_hl + cc % kHBufs, (uint32_t)(cc / kHBufs) & 1);
        }
        __syncwarp();
    } else if (kSide && warp == kSideW) {
        if (lane == 0 && has_h) {
            // U of chunk ch + 1 = [H; T B] times its value rows (rows 64-127 of
            // the product; the H rows give nothing used), into TMEM columns by
            // chunk parity, once chunk ch's first product has completed (the
            // pipe runs it while the compute warps form Z); chunk 0's first.
            // Then, with outputs, D1 += [H; T B] [Z_hi | Z_lo] once the second
            // product has completed, which adds H Z to the s Qbar S rows 0-63
            // (rows 64-127 take (T B) Z; W S there is consumed).
            // Phases stay in step: the first product's barrier here completes
            // a phase only with this warp's arrival; chunk ch + 1's second
            // product needs the outputs of chunk ch read, hence H Z of chunk ch
            // issued after this warp saw chunk ch's second product.
            const uint64_t d_ht = desc(smem_u32(sm + L::kH), kA2Lbo, kA2Sbo);
            const uint64_t d_v = desc(smem_u32(sm + L::kH + kHTBytes), kBvLbo, kBvSbo);
            const uint64_t d_b2 = desc(smem_u32(B2), kB2Lbo, kB2Sbo);
            const uint32_t id2 = idesc_bf16(128, 2 * TN, 0, 1), idu = idesc_bf16(128, TN, 0, 1);
            bool ok = true;
            auto issue_u = [&](int ch) {
                ok = ok && wait(bar_hl + ch % kHBufs, (uint32_t)(ch / kHBufs) & 1);
                if (!ok) return;
                const uint64_t ho = (uint64_t)(ch % kHBufs) * (L::kHBytes >> 4);
                fence_after();
#pragma unroll
                for (int s = 0; s < C / 16; ++s)
                    mma_bf16(tmem + L::kUCol + TN * (ch & 1), d_ht + ho + s * (2 * kA2Lbo >> 4),
                             d_v + ho + s * (2 * kBvLbo >> 4), idu, s > 0);
                commit(bar_u + (ch & 1));
            };
            if (!ident && nchunks > 0) issue_u(0);
            mbar_arrive(bar_m1s);  // chunk 0's phase
            for (int ch = 0; ch < nchunks && ok; ++ch) {
                if (!ident && ch + 1 < nchunks) {
                    spin(bar_m1s, (uint32_t)ch & 1);
                    mbar_arrive(bar_m1s);  // chunk ch + 1's phase
                    issue_u(ch + 1);
                }
                if (outputs && ok) {
                    spin(bar_m2, (uint32_t)ch & 1);
                    if (*err) break;
                    fence_after();
                    const uint64_t ho = (uint64_t)(ch % kHBufs) * (L::kHBytes >> 4);
#pragma unroll
                    for (int s = 0; s < C / 16; ++s)
                        mma_bf16(tmem + 2 * TN * (ch & 1), d_ht + ho + s * (2 * kA2Lbo >> 4),
                                 d_b2 + s * (2 * kB2Lbo >> 4), id2, 1);
                    commit(bar_m3);
                }
                // Everything this warp issued on chunk ch's H slot (its U, and
                // H Z) precedes this commit.
                commit(bar_hf + ch % kHBufs);
            }
        }
        __syncwarp();
    } else if (warp == kMma) {
        // One lane issues; the whole warp keeps the named-barrier protocol, so
        // the compute warps never wait on a barrier that cannot complete.
        // Descriptors of slot 0's tiles and of the state-side operands are
        // built once; a chunk adds its slot's offset and a K step a constant
        // (the address field is the byte address / 16).
        const uint64_t d_a1 = desc(smem_u32(sm), kA1Lbo, kA1Sbo);
        const uint64_t d_a2 = desc(smem_u32(sm + L::kK), kA2Lbo, kA2Sbo);
        const uint64_t d_b1 = desc(smem_u32(B1), kB1Lbo, kB1Sbo);
        const uint64_t d_b2 = desc(smem_u32(B2), kB2Lbo, kB2Sbo);
        const uint32_t id1 = idesc_bf16(128, 2 * TN, 1, 1), id2 = idesc_bf16(128, 2 * TN, 0, 1);
        bool ok = true;  // lane 0: every wait so far succeeded
        // Without the side warp: U of chunk ch + 1 right after chunk ch's first
        // product (the pipe runs it while the compute warps form Z), and H Z
        // right after the second product.
        const uint64_t d_ht = desc(smem_u32(sm + L::kH), kA2Lbo, kA2Sbo);
        const uint64_t d_v = desc(smem_u32(sm + L::kH + kHTBytes), kBvLbo, kBvSbo);
        const uint32_t idu = idesc_bf16(128, TN, 0, 1);
        auto issue_u = [&](int ch) {
            ok = ok && wait(bar_hl + ch % kHBufs, (uint32_t)(ch / kHBufs) & 1);
            if (!ok) return;
            const uint64_t ho = (uint64_t)(ch % kHBufs) * (L::kHBytes >> 4);
            fence_after();
#pragma unroll
            for (int s = 0; s < C / 16; ++s)
                mma_bf16(tmem + L::kUCol + TN * (ch & 1), d_ht + ho + s * (2 * kA2Lbo >> 4),
                         d_v + ho + s * (2 * kBvLbo >> 4), idu, s > 0);
            commit(bar_u + (ch & 1));
        };
        if (!kSide && lane == 0 && !ident && nchunks > 0) issue_u(0);
        for (int ch = 0; ch < nchunks; ++ch) {
            const uint64_t xo = (uint64_t)(ch % kXBufs) * (kXBytes >> 4);
            const uint64_t ko = (uint64_t)(ch % kKBufs) * (kKBytes >> 4);
            const uint32_t d1 = tmem + 2 * TN * (ch & 1);
            if (lane == 0) {
                // Chunk 0's tiles; a later chunk's were waited for before the
                // state barrier (off the chain of dependent steps).
                if (ch == 0) ok = ok && wait(bar_xl, 0);
                if (ok) {
                    // [s Qbar S; W S] with S = S_hi + S_lo: N = 2 TN (hi columns first).
                    fence_after();
#pragma unroll
                    for (int s = 0; s < D / 16; ++s)
                        mma_bf16(d1, d_a1 + xo + s * (2 * kA1Lbo >> 4), d_b1 + s * (2 * kB1Lbo >> 4),
                                 id1, s > 0);
                    commit(bar_m1);
                    if (kSide) commit(bar_m1s);
                }
                // The X slot is free once everything issued so far has completed.
                commit(bar_xf + ch % kXBufs);
                if (!kSide && !ident && ch + 1 < nchunks) issue_u(ch + 1);
                // The second product reads the K tiles.
                ok = ok && wait(bar_kl + ch % kKBufs, (uint32_t)(ch / kKBufs) & 1);
            }
            __syncwarp();
            bar_sync(kBarZ, kSync);  // Z of this chunk is in B2
            fence_after();
            if (lane == 0) {
                if (ok) {
                    // D2 = Kbar^T [Z_hi | Z_lo] (N = 2 TN).
#pragma unroll
                    for (int s = 0; s < C / 16; ++s)
                        mma_bf16(tmem + L::kD2Col, d_a2 + ko + s * (2 * kA2Lbo >> 4),
                                 d_b2 + s * (2 * kB2Lbo >> 4), id2, s > 0);
                    commit(bar_m2);
                    if (!kSide && outputs) {
                        // D1 += [H; T B] [Z_hi | Z_lo]: H Z into the s Qbar S rows.
                        const uint64_t ho = (uint64_t)(ch % kHBufs) * (L::kHBytes >> 4);
#pragma unroll
                        for (int s = 0; s < C / 16; ++s)
                            mma_bf16(d1, d_ht + ho + s * (2 * kA2Lbo >> 4), d_b2 + s * (2 * kB2Lbo >> 4),
                                     id2, 1);
                        commit(bar_m3);
                    }
                }
                commit(bar_kf + ch % kKBufs);
                // Chunk ch's U (issued a chunk ago) and H Z were the H slot's readers.
                if (!kSide && has_h) commit(bar_hf + ch % kHBufs);
                if (ch + 1 < nchunks)
                    ok = ok && wait(bar_xl + (ch + 1) % kXBufs, (uint32_t)((ch + 1) / kXBufs) & 1);
            }
            __syncwarp();
            bar_sync(kBarS, kSync);  // the new state is in B1
            fence_after();
        }
        __syncwarp();
    } else if (compute) {
        uint32_t p1 = 0, p2 = 0, p3 = 0;  // phases of the three product barriers
        uint32_t rph = 0;                 // phases of the two row-partial barriers (bit per parity)
        const bool zrow = r >= 64;
        float wv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) wv[j] = gated && og.w ? og.w[j0 + js + j] : 1.f;
        const uint32_t crank = gated ? cluster_rank() : 0u;
        // Token outputs of chunk `ch` (rows 0-63 of its D1): s Qbar S + H Z,
        // or with the fused gate (TN = 32: eight columns a thread) w o / rms(o)
        // sigmoid(z), the mean of squares over all D columns: this CTA's 32
        // are summed through shared memory, then every CTA of the cluster
        // sends its row sums to all four.
        // The gate logits of chunk ch: one tensor-map tile (TN columns x 64
        // tokens) into the slot, issued by thread 0 once every output thread
        // has read the previous chunk's.
        const __nv_bfloat16 *zslot = reinterpret_cast<const __nv_bfloat16 *>(sm + L::kZ);
        auto issue_z = [&](int ch) {
            if (tid != 0 || ch >= nchunks) return;
            mbar_expect_tx(z_full, L::kZBytes);
            tma_load_3d(sm + L::kZ, tm_z, j0, h, bos + (c0 + ch) * C, z_full);
        };
        uint32_t zph = 0;
        int z_issued = 0;  // tiles issued (tid 0)
        if (gated && outputs) {
            issue_z(0);
            z_issued = nchunks > 0 ? 1 : 0;
        }
        // Plain outputs are stored as soon as they are read. With the gate, part
        // one (before this chunk's Z barrier) reads the outputs and sends their
        // row sums of squares to the cluster; part two (while the second
        // product runs) forms w sigmoid(z), takes the four CTAs' sums,
        // normalises and stores.
        float o8[8];
        uint4 zr = make_uint4(0u, 0u, 0u, 0u);
        auto put_outputs_a = [&](int ch) {  // ch counts this segment's chunks
            const uint32_t d1 = tmem + lane_base + 2 * TN * (ch & 1);
            if (!gated) {
                const int clen = min(C, len - (c0 + ch) * C);
#pragma unroll
                for (int q = 0; q < NP; ++q) if (q < np) {
                    float hi[8], lo[8], o[8];
                    tmem_ld8(d1 + js + 8 * q, hi);
                    tmem_ld8(d1 + TN + js + 8 * q, lo);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 8; ++j) o[j] = hi[j] + lo[j];
                    if (r < clen)
                        *reinterpret_cast<uint4 *>(out + ((size_t)(bos + (c0 + ch) * C + r) * H + h) * D +
                                                   j0 + js + 8 * q) = pack8(o);
                }
                return;
            }
            if (!mbar_test(z_full, zph) && !*err && !mbar_wait(z_full, zph)) {
                *err = 1;
                atomicExch(status, (int)KDA_ERR_TIMEOUT);
            }
            zph ^= 1;
            zr = *reinterpret_cast<const uint4 *>(zslot + r * TN + js);
            __syncwarp();
            float hi[8], lo[8];
            tmem_ld8(d1 + js, hi);
            tmem_ld8(d1 + TN + js, lo);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 8; ++j) o8[j] = hi[j] + lo[j];
            const int par = ch & 1;
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) ss += o8[j] * o8[j];
            loc[(js >> 3) * 64 + r] = ss;
            // The z reads (generic proxy) are ordered before the tensor-map
            // copy that refills the slot (async proxy) after the barrier.
            fence_async_smem();
            // Every output thread has read its z (the slot is free) and has
            // finished the previous chunk, whose row sums it read: that
            // barrier's next phase (chunk ch + 1) may now expect its bytes,
            // before this CTA sends anything a peer could answer with them.
            bar_sync(kBarO, 256);
            if (ch + 1 < nchunks) {
                issue_z(ch + 1);
                z_issued = ch + 2;
            }
            if (tid == 0 && ch >= 1 && ch + 1 < nchunks) mbar_expect_tx(red_full + (par ^ 1), kRedBytes);
            if (tid < 16) {
                // Rows 4 tid .. 4 tid + 3: this CTA's sums, 16 bytes to each CTA.
                float4 pr;
                float *pp = reinterpret_cast<float *>(&pr);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int row = 4 * tid + i;
                    pp[i] = loc[row] + loc[64 + row] + loc[128 + row] + loc[192 + row];
                }
                float *slot = red + (par * kGateCluster + (int)crank) * 64 + 4 * tid;
#pragma unroll
                for (uint32_t dst = 0; dst < (uint32_t)kGateCluster; ++dst)
                    st_async_cluster_v4(cluster_addr(slot, dst), pr, cluster_addr(red_full + par, dst));
            }
        };
        auto put_outputs_b = [&](int ch) {
            if (!gated) return;  // stored by part one
            const int clen = min(C, len - (c0 + ch) * C);
            const size_t orow = ((size_t)(bos + (c0 + ch) * C + r) * H + h) * D + j0 + js;
            {
                const int par = ch & 1;
                float gz[8];
                const uint32_t zu[4] = {zr.x, zr.y, zr.z, zr.w};
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float zj = __uint_as_float((j & 1) ? (zu[j >> 1] & 0xFFFF0000u) : (zu[j >> 1] << 16));
                    gz[j] = wv[j] * sigmoid_fast(zj);
                }
                if (!mbar_test_cluster(red_full + par, (rph >> par) & 1u) && !*err &&
                    !mbar_wait_cluster(red_full + par, (rph >> par) & 1u)) {
                    *err = 1;
                    atomicExch(status, (int)KDA_ERR_TIMEOUT);
                }
                rph ^= 1u << par;
                const float *rp = red + par * kGateCluster * 64 + r;
                float tot = 0.f;
#pragma unroll
                for (int q = 0; q < kGateCluster; ++q) tot += rp[q * 64];
                const float rs = rsqrtf(tot * (1.f / D) + og.eps);
#pragma unroll
                for (int j = 0; j < 8; ++j) o8[j] *= gz[j] * rs;
            }
            if (r < clen) *reinterpret_cast<uint4 *>(out + orow) = pack8(o8);
        };
        for (int ch = 0; ch < nchunks; ++ch) {
            const uint32_t d1 = tmem + 2 * TN * (ch & 1);
            // The K tiles landed before this chunk's second product was
            // issued; this thread's own wait makes the copied decay visible.
            wait(bar_kl + ch % kKBufs, (uint32_t)(ch / kKBufs) & 1);
            const float gam = reinterpret_cast<const float *>(sm + L::kK + (ch % kKBufs) * kKBytes + kKGam)[r];
            if (zrow && outputs && ch > 0) {
                // The previous chunk's H Z product reads B2, which this chunk's
                // Z overwrites (it is issued by another thread than the first
                // product, whose completion therefore does not imply its own).
                wait(bar_m3, p3);
                p3 ^= 1;
            }
            // This chunk's U row (formed while the previous state was updated).
            float uv[NJ];
#pragma unroll
            for (int j = 0; j < NJ; ++j) uv[j] = 0.f;
            if (zrow && !ident) {
                spin(bar_u + (ch & 1), (uint32_t)(ch >> 1) & 1);
                fence_after();
                __syncwarp();  // tcgen05.ld is warp-collective: reconverge after the per-lane wait
                // Z-row threads hold exactly ZP pieces; their loads are issued
                // before one wait, so that the latencies overlap.
                float u8[ZP][8];
#pragma unroll
                for (int q = 0; q < ZP; ++q) tmem_ld8(tmem + lane_base + L::kUCol + TN * (ch & 1) + js + 8 * q, u8[q]);
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < ZP; ++q)
#pragma unroll
                    for (int j = 0; j < 8; ++j) uv[8 * q + j] = u8[q][j];
            }
            if (!zrow && outputs && ch > 0) {
                // The previous chunk's outputs, complete once its H Z product is:
                // read while this chunk's first product runs.
                wait(bar_m3, p3);
                p3 ^= 1;
                fence_after();
                __syncwarp();  // tcgen05.ld is warp-collective: reconverge after the per-lane wait
                put_outputs_a(ch - 1);
            }
            spin(bar_m1, p1);
            p1 ^= 1;
            fence_after();
            __syncwarp();  // tcgen05.ld is warp-collective: reconverge after the per-lane wait
            if (zrow) {
                // Z = U - W S for token row i, slab columns js .. js + NJ - 1.
                const int i = r - 64;
                float hi[ZP][8], lo[ZP][8];
#pragma unroll
                for (int q = 0; q < ZP; ++q) {
                    tmem_ld8(d1 + lane_base + js + 8 * q, hi[q]);
                    tmem_ld8(d1 + lane_base + TN + js + 8 * q, lo[q]);
                }
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < ZP; ++q) {
                    float z[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) z[j] = uv[8 * q + j] - (hi[q][j] + lo[q][j]);
                    uint4 zh, zl;
                    split8(z, zh, zl);
                    *reinterpret_cast<uint4 *>(B2 + mnmaj(js + 8 * q, i, kB2Lbo, kB2Sbo)) = zh;
                    *reinterpret_cast<uint4 *>(B2 + mnmaj(TN + js + 8 * q, i, kB2Lbo, kB2Sbo)) = zl;
                }
            }
            fence_async_smem();
            fence_before();
            bar_arrive(kBarZ, kSync);
            if (!zrow && outputs && ch > 0) put_outputs_b(ch - 1);  // while the second product runs
            spin(bar_m2, p2);
            p2 ^= 1;
            fence_after();
            __syncwarp();  // tcgen05.ld is warp-collective: reconverge after the per-lane wait
            // Pieces in pairs: both loads of a pair before one wait.
#pragma unroll
            for (int q0 = 0; q0 < NP; q0 += 2) {
                float hi[2][8], lo[2][8];
#pragma unroll
                for (int u = 0; u < 2; ++u) if (q0 + u < NP && q0 + u < np) {
                    tmem_ld8(tmem + lane_base + L::kD2Col + js + 8 * (q0 + u), hi[u]);
                    tmem_ld8(tmem + lane_base + L::kD2Col + TN + js + 8 * (q0 + u), lo[u]);
                }
                tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < 2; ++u) if (q0 + u < NP && q0 + u < np) {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        S[8 * (q0 + u) + j] = gam * S[8 * (q0 + u) + j] + (hi[u][j] + lo[u][j]);
                }
            }
            put_state();
            fence_async_smem();
            fence_before();
            // A full barrier here (an arrive would do on the normal path, where
            // the product barriers pace the compute warps) keeps every warp
            // within one phase of the named barriers even when a timeout has
            // made the product waits fall through.
            bar_sync(kBarS, kSync);
        }
        if (nchunks > 0 && !zrow && outputs) {
            wait(bar_m3, p3);
            fence_after();
            __syncwarp();  // tcgen05.ld is warp-collective: reconverge after the per-lane wait
            put_outputs_a(nchunks - 1);
            put_outputs_b(nchunks - 1);
        }
        // Every z tile lands before the CTA exits (bounded; the output threads
        // waited for each one unless an error made them skip).
        if (gated && tid == 0 && z_issued > 0) mbar_wait(z_full, (uint32_t)(z_issued - 1) & 1u);
        if (st_dst && !refused && !*err) {
            float *dst = st_dst + (size_t)r * dst_row + j0 + js;
#pragma unroll
            for (int q = 0; q < 2 * NP; ++q)
                if (q < 2 * np) *reinterpret_cast<float4 *>(dst + 4 * q) = make_float4(S[4 * q], S[4 * q + 1], S[4 * q + 2], S[4 * q + 3]);
        }
    }
    fence_before();
    __syncthreads();
    // No CTA leaves while a peer may still write into its shared memory.
    if (gated) cluster_sync();
    if (warp == 0) tmem_dealloc<L::kCols>(tmem);
}

__global__ void __launch_bounds__(kP2Threads, 1)
tc_state_pass(const unsigned char *__restrict__ ws, const int *__restrict__ seq_first_slot,
              const int *__restrict__ seq_order, const int32_t *__restrict__ cu_seqlens,
              int T_fixed, const float *init_state, __nv_bfloat16 *__restrict__ out,
              float *final_state, int H, int *__restrict__ status, const SegPass sp,
              const OutGate og, const __grid_constant__ CUtensorMap tm_z,
              const __grid_constant__ CUtensorMap tm_v) {
    state_pass_body<kTN>(ws, seq_first_slot, seq_order, cu_seqlens, T_fixed, init_state, out,
                         final_state, H, status, sp, og, &tm_z, &tm_v, (int)blockIdx.x, nullptr);
}

// The serial state pass with 64-column slabs as a launch of its own (two CTAs
// per sequence and head; the fused kernel's state-pass role without the ready
// flags). Per column it costs less than the 32-column pass (about 3.7k cycles
// per chunk for 64 columns against 2 x 2.9k), the 32-column pass has the shorter
// chain: this one serves many chains, where the CTAs run in several waves.
__global__ void __launch_bounds__(kFusedThreads, 1)
tc_state_pass64(const unsigned char *__restrict__ ws, const int *__restrict__ seq_first_slot,
                const int *__restrict__ seq_order, const int32_t *__restrict__ cu_seqlens, int T_fixed,
                const float *init_state, __nv_bfloat16 *__restrict__ out, float *final_state, int H,
                int *__restrict__ status, const __grid_constant__ CUtensorMap tm_v) {
    const SegPass sp{1 << 30, 1, 0, 1, 0, nullptr, nullptr};
    state_pass_body<64>(ws, seq_first_slot, seq_order, cu_seqlens, T_fixed, init_state, out, final_state,
                        H, status, sp, OutGate{nullptr, nullptr, 0.f}, &tm_v, &tm_v, (int)blockIdx.x,
                        nullptr);
}

// The fused prefill: one cooperative launch whose first n_state CTAs run the
// state pass with 64-column slabs while the rest run phase 1, chunk-major,
// handing each (slot, head) region over through its ready flag. Phase 1
// never waits for the state pass, and the launch is cooperative (all CTAs
// resident at once), so every flag a state-pass CTA waits for gets set.
template <int kVar>
__global__ void __launch_bounds__(kFusedThreads, 1)
tc_prefill_fused(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_v,
                 const float *__restrict__ g_head, Prologue pro, const float *__restrict__ beta,
                 float scale, const ChunkEntry *__restrict__ table, const int *__restrict__ used_slots,
                 long long nslots, int H, unsigned char *__restrict__ ws, int *__restrict__ status,
                 const int *__restrict__ seq_first_slot, const int *__restrict__ seq_order,
                 const int32_t *__restrict__ cu_seqlens, int T_fixed, const float *init_state,
                 __nv_bfloat16 *__restrict__ out, float *final_state, int n_state, int *ready, int ilv,
                 int nch) {
    if ((int)blockIdx.x < n_state) {
        const SegPass sp{1 << 30, 1, 0, 1, 0, nullptr, nullptr};
        state_pass_body<64>(ws, seq_first_slot, seq_order, cu_seqlens, T_fixed, init_state, out,
                            final_state, H, status, sp, OutGate{nullptr, nullptr, 0.f}, &tm_v, &tm_v,
                            (int)blockIdx.x, ready);
    } else {
        intra_chunk_body<kVar>(&tm_q, &tm_k, &tm_g, g_head, pro, beta, scale, table, used_slots, nslots,
                               H, ws, status,
                               P1Walk{(int)blockIdx.x - n_state, (int)gridDim.x - n_state, ready, ilv, nch});
    }
}

// Composition of the segment maps, in order: enter[p + 1] = M_p enter[p] + E_p
// for p = 1 .. P - 2 (enter[1] is segment 0's end state). One CTA per
// (sequence, head, 32-column tile of the state); fp32 throughout. Thread t
// owns row t / 2 and 16 columns; the state tile stays in shared memory from
// one segment to the next.
constexpr int kCombThreads = 256;
constexpr int kCombCols = 32;
constexpr int kCombMs = D + 1;  // padded row stride of M_p: rows t / 2 fall in distinct banks
constexpr size_t kCombSmem = sizeof(float) * ((size_t)D * kCombMs + (size_t)D * kCombCols);

__global__ void __launch_bounds__(kCombThreads)
seg_combine(const float *__restrict__ xfer, float *__restrict__ enter, int P) {
    extern __shared__ float csm[];
    float *Ms = csm;                   // [D][kCombMs]
    float *Ss = csm + D * kCombMs;     // [D][kCombCols]
    const int nh = blockIdx.x / (D / kCombCols), j0 = (blockIdx.x % (D / kCombCols)) * kCombCols;
    const int tid = threadIdx.x, i = tid >> 1, jh = (tid & 1) * 16;
    const float *x0 = xfer + (size_t)nh * P * D * 2 * D;
    float *e0 = enter + (size_t)nh * P * D * D;
    for (int idx = tid; idx < D * kCombCols; idx += kCombThreads) {
        const int k = idx / kCombCols, j = idx % kCombCols;
        Ss[k * kCombCols + j] = e0[((size_t)1 * D + k) * D + j0 + j];
    }
    for (int p = 1; p + 1 < P; ++p) {
        const float *xp = x0 + (size_t)p * D * 2 * D;
        for (int idx = tid; idx < D * D / 4; idx += kCombThreads) {
            const int row = idx / (D / 4), c4 = idx % (D / 4);
            const float4 m = *reinterpret_cast<const float4 *>(xp + (size_t)row * 2 * D + D + 4 * c4);
            float *dst = Ms + row * kCombMs + 4 * c4;
            dst[0] = m.x; dst[1] = m.y; dst[2] = m.z; dst[3] = m.w;
        }
        __syncthreads();
        float acc[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] = xp[(size_t)i * 2 * D + j0 + jh + j];
#pragma unroll 4
        for (int k = 0; k < D; ++k) {
            const float m = Ms[i * kCombMs + k];
            const float4 *sr = reinterpret_cast<const float4 *>(Ss + k * kCombCols + jh);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 sv = sr[q];
                acc[4 * q] += m * sv.x; acc[4 * q + 1] += m * sv.y;
                acc[4 * q + 2] += m * sv.z; acc[4 * q + 3] += m * sv.w;
            }
        }
        __syncthreads();  // every thread is done with Ss and Ms
        float *ep = e0 + ((size_t)(p + 1) * D + i) * D + j0 + jh;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 v = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
            *reinterpret_cast<float4 *>(ep + 4 * q) = v;
            *reinterpret_cast<float4 *>(Ss + i * kCombCols + jh + 4 * q) = v;
        }
    }
}

}  // namespace

// Workspace bytes per (slot, head): its region and, after all regions, its
// ready flag (the fused prefill's hand-over from phase 1 to the state pass).
size_t tc_region_bytes() { return TcRegion::bytes + sizeof(int); }

namespace {

// cuTensorMapEncodeTiled, fetched from the driver at run time so that the
// library does not link libcuda.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// A [tokens][H][128] tensor seen as 3-D (channel, head, token) with boxes of
// 128 channels x 1 head x 64 tokens; out-of-range tokens read as zeros.
cudaError_t token_rows_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize, int H,
                           long long tokens) {
    EncodeTiledFn enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)D * esize, (cuuint64_t)H * D * esize};
    const cuuint32_t box[3] = {(cuuint32_t)D, 1u, (cuuint32_t)C};
    const cuuint32_t unit[3] = {1u, 1u, 1u};
    const CUresult r = enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, unit,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The gate logits [tokens][H][128] bf16 seen as 3-D (channel, head, token)
// with boxes of one state-pass CTA's 32 columns x 1 head x 64 tokens.
cudaError_t gate_rows_map(CUtensorMap *m, const void *base, int H, long long tokens) {
    EncodeTiledFn enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kTN, 1u, (cuuint32_t)C};
    const cuuint32_t unit[3] = {1u, 1u, 1u};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                           strides, box, unit, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The value rows [tokens][H][128] bf16 seen as 3-D (8 channels, token, group
// of 8 channels across the heads) with boxes of 8 channels x 64 tokens x
// tn / 8 groups: a box lands as [group][token][8 channels], the MN-major
// operand layout (K = token, N = channel) with 128-byte K steps and 1 KiB
// channel-group strides. Tokens past the tensor read as zeros.
cudaError_t value_rows_map(CUtensorMap *m, const void *base, int H, long long tokens, int tn) {
    EncodeTiledFn enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {8u, (cuuint64_t)tokens, (cuuint64_t)H * D / 8};
    const cuuint64_t strides[2] = {(cuuint64_t)H * D * 2, 16u};
    const cuuint32_t box[3] = {8u, (cuuint32_t)C, (cuuint32_t)(tn / 8)};
    const cuuint32_t unit[3] = {1u, 1u, 1u};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                           strides, box, unit, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Whether the fused single launch is expected to beat the two launches, from
// a cost model of the measured rates on this part: phase 1 about 9.4k
// cycles per (chunk, head) item and SM; the state pass about 2.9k cycles per
// chunk with 32-column slabs and 3.76k with 64-column ones. Two launches take
// phase 1 on every SM, then the chain; the fused one runs phase 1 on the SMs
// the 64-column state pass leaves and the chain beside it.
bool fuse_pays(long long items, int chain_chunks, long long n_state, int sm_count) {
    if (n_state < 1 || n_state > sm_count - 8) return false;
    const double p1_all = 9.4 * (double)items / (double)(items < sm_count ? items : sm_count);
    const double p1_rest = 9.4 * (double)items / (double)(sm_count - n_state);
    const double two = p1_all + 2.9 * chain_chunks;
    const double fused = (p1_rest > 3.76 * chain_chunks ? p1_rest : 3.76 * chain_chunks) + 9.4;
    return fused < 0.95 * two;
}

// Segments of the state pass for the `segments` option (0: automatic, 1: the
// serial chain, k: k segments), at most seg_max (the workspace's bound) and
// one per chunk. Automatic: as many as keep the transfer launch within one
// wave (chains x (D/kTN + 2 D/kTN (P - 2)) CTAs <= SMs), with at least 8
// chunks per segment, and only when that makes 3 or more (with two, as many
// chunks run in series as with one) and T >= 32 chunks.
int state_segments(int segments, int seg_max, int nch, long long chains, int sm_count) {
    constexpr int kTiles = D / kTN;
    if (seg_max < 2 || segments == 1 || nch < 2 || chains <= 0) return 1;
    if (segments >= 2) return min(segments, min(seg_max, nch));
    if (nch < 32) return 1;
    const long long per = sm_count / chains;  // CTAs per chain in one wave
    long long p = per >= kTiles ? (per - kTiles) / (2 * kTiles) + 2 : 1;
    if (p > seg_max) p = seg_max;
    if (p > nch / 8) p = nch / 8;
    return p >= 3 ? (int)p : 1;
}

}  // namespace

cudaError_t launch_prefill_tc(const void *q, const void *k, const void *v, const float *g,
                              const float *beta, float scale, const float *init_state,
                              const int32_t *cu_seqlens, void *out, float *final_state,
                              int T_fixed, long long tokens, int H, int num_seqs, long long slots,
                              const ChunkEntry *table, const int *seq_first_slot,
                              unsigned char *region, int *status, const Prologue &pro,
                              int segments, int seg_max, float *seg_ws, const GateParams &gate,
                              int fused, cudaStream_t stream, cudaEvent_t *events) {
    // Per device, once: the SM count (phase 1 runs one persistent CTA per SM),
    // the dynamic shared-memory opt-ins and cooperative-launch support.
    // Repeating this is idempotent.
    static int sm_counts[64];
    static bool coop_ok[64];
    constexpr int kFusedSmem = P1::bytes > P2L<64>::kSmem ? P1::bytes : P2L<64>::kSmem;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (sm_counts[dev] == 0) {
        int n = 0, coop = 0;
        if ((err = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (err = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess)
            return err;
#define KDA_SMEM(F, B)                                                                             \
    if ((err = cudaFuncSetAttribute(F, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(B))) != \
        cudaSuccess)                                                                               \
        return err;
        KDA_SMEM(tc_intra_chunk<kVarChannel>, P1::bytes)
        KDA_SMEM(tc_intra_chunk<kVarRuntime>, P1::bytes)
        KDA_SMEM(tc_intra_chunk<kVarScalar>, P1::bytes)
        KDA_SMEM(tc_intra_chunk<kVarNone>, P1::bytes)
        KDA_SMEM(tc_intra_chunk<kVarGated>, P1::bytes)
        KDA_SMEM(tc_prefill_fused<kVarChannel>, kFusedSmem)
        KDA_SMEM(tc_prefill_fused<kVarRuntime>, kFusedSmem)
        KDA_SMEM(tc_prefill_fused<kVarScalar>, kFusedSmem)
        KDA_SMEM(tc_prefill_fused<kVarNone>, kFusedSmem)
        KDA_SMEM(tc_prefill_fused<kVarGated>, kFusedSmem)
        KDA_SMEM(tc_state_pass, P2L<kTN>::kSmem)
        KDA_SMEM(tc_state_pass64, P2L<64>::kSmem)
        KDA_SMEM(seg_combine, kCombSmem)
#undef KDA_SMEM
        coop_ok[dev] = coop != 0;
        sm_counts[dev] = n;
    }
    const int sm_count = sm_counts[dev];
    const int *used = seq_first_slot + num_seqs;
    const int *order = seq_first_slot + num_seqs + 1;
    const int nch = (T_fixed + C - 1) / C;
    const long long items = slots * H;
    // The fused output gate runs on the serial chain (its clusters are the
    // four column tiles of one sequence and head).
    const OutGate og{static_cast<const __nv_bfloat16 *>(gate.z), gate.w, gate.eps};
    const int P = og.z ? 1 : state_segments(segments, seg_max, nch, (long long)num_seqs * H, sm_count);
    // The fused launch: on the serial chain, with chunk c of every sequence at
    // the same place in phase 1's order (fixed-length batches, or one packed
    // sequence), and when the cost model favours it. With the output gate it
    // writes plain outputs and the gate pass follows (one read of o and z, one
    // write: cheaper than the two launches with the gate in the state pass,
    // whose output warps then lengthen every chunk).
    const long long n_state = (long long)num_seqs * H * (D / 64);
    const int chain_chunks = cu_seqlens ? (int)(slots / (num_seqs > 0 ? num_seqs : 1)) : nch;
    const bool use_fused = fused >= 0 && coop_ok[dev] && P <= 1 && slots > 0 && tokens > 0 &&
                           (!cu_seqlens || num_seqs == 1) && n_state <= sm_count - 8 &&
                           (fused == 1 || fuse_pays(items, chain_chunks, n_state, sm_count));
    int var = kVarRuntime;
    if (!pro.l2norm) {
        if (pro.decay == KDA_DECAY_NONE)  // the gate is never applied
            var = kVarNone;
        else if (pro.gate == KDA_GATE_LOG)
            var = pro.decay == KDA_DECAY_CHANNEL ? kVarChannel : kVarScalar;
    } else if (pro.decay == KDA_DECAY_CHANNEL && pro.gate == KDA_GATE_LOGSIGMOID) {
        var = kVarGated;
    }
    if ((err = mark(events, 1, stream)) != cudaSuccess) return err;
    CUtensorMap tq, tk, tg;
    memset(&tg, 0, sizeof(tg));  // read only with a per-channel g
    if (slots > 0 && tokens > 0) {
        if ((err = token_rows_map(&tq, q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, tokens)) != cudaSuccess ||
            (err = token_rows_map(&tk, k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, tokens)) != cudaSuccess)
            return err;
        if (pro.decay == KDA_DECAY_CHANNEL &&
            (err = token_rows_map(&tg, g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, H, tokens)) != cudaSuccess)
            return err;
    }
    if (use_fused) {
        // Ready flags after the regions: one int per (slot, head), cleared here.
        int *ready = reinterpret_cast<int *>(region + (size_t)slots * H * TcRegion::bytes);
        CUtensorMap tv;
        if ((err = value_rows_map(&tv, v, H, tokens, 64)) != cudaSuccess) return err;
        if ((err = cudaMemsetAsync(ready, 0, (size_t)slots * H * sizeof(int), stream)) != cudaSuccess)
            return err;
        const int ilv = cu_seqlens ? 1 : num_seqs;
        const int nstate = (int)n_state;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)sm_count);
        cfg.blockDim = dim3(kFusedThreads);
        cfg.dynamicSmemBytes = kFusedSmem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(out);
        unsigned char *ws = region;
#define KDA_FUSED(V)                                                                               \
    err = cudaLaunchKernelEx(&cfg, tc_prefill_fused<V>, tq, tk, tg, tv, g, pro, beta, scale, table, \
                             used, slots, H, ws, status, seq_first_slot, order, cu_seqlens, T_fixed, \
                             init_state, o, final_state, nstate, ready, ilv, nch)
        switch (var) {
            case kVarChannel: KDA_FUSED(kVarChannel); break;
            case kVarScalar: KDA_FUSED(kVarScalar); break;
            case kVarNone: KDA_FUSED(kVarNone); break;
            case kVarGated: KDA_FUSED(kVarGated); break;
            default: KDA_FUSED(kVarRuntime); break;
        }
#undef KDA_FUSED
        if (err == cudaSuccess) {
            // Phase 1 and the state pass are one launch: both phase marks follow it.
            if ((err = mark(events, 2, stream)) != cudaSuccess) return err;
            if (og.z && (err = launch_output_gate_rmsnorm(out, og.z, og.w, og.eps, out, tokens * H, D,
                                                          KDA_DTYPE_BF16, stream)) != cudaSuccess)
                return err;
            return mark(events, 3, stream);
        }
        // Not resident all at once on this device (or not supported): the
        // two launches below do the same work.
        if (err != cudaErrorCooperativeLaunchTooLarge && err != cudaErrorNotSupported) return err;
        (void)cudaGetLastError();
    }
    if (slots > 0 && tokens > 0) {
        const unsigned grid = (unsigned)(items < sm_count ? items : sm_count);
#define KDA_P1_LAUNCH(V)                                                                        \
    tc_intra_chunk<V><<<grid, kP1Threads, P1::bytes, stream>>>(tq, tk, tg, g, pro, beta, scale,     \
                                                               table, used, slots, H, region, status)
        switch (var) {
            case kVarChannel: KDA_P1_LAUNCH(kVarChannel); break;
            case kVarScalar: KDA_P1_LAUNCH(kVarScalar); break;
            case kVarNone: KDA_P1_LAUNCH(kVarNone); break;
            case kVarGated: KDA_P1_LAUNCH(kVarGated); break;
            default: KDA_P1_LAUNCH(kVarRuntime); break;
        }
#undef KDA_P1_LAUNCH
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    if ((err = mark(events, 2, stream)) != cudaSuccess) return err;
    if (num_seqs > 0) {
        static_assert(2 * (D / kTN) <= kMaxStateTiles, "grid bound checked with kMaxStateTiles");
        constexpr int kTiles = D / kTN;
        constexpr int kSmem = P2L<kTN>::kSmem;
        CUtensorMap tz, tv;
        memset(&tz, 0, sizeof(tz));  // read only by the fused gate
        memset(&tv, 0, sizeof(tv));  // read only when there are tokens
        if (og.z && (err = gate_rows_map(&tz, og.z, H, tokens)) != cudaSuccess) return err;
        if (tokens > 0 && (err = value_rows_map(&tv, v, H, tokens, kTN)) != cudaSuccess) return err;
        if (P <= 1 && og.z) {
            static_assert(kGateCluster == kTiles, "a cluster holds the column tiles of one head");
            const SegPass sp{1 << 30, 1, 0, 1, 0, nullptr, nullptr};
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)num_seqs * H * kTiles);
            cfg.blockDim = dim3(kP2Threads);
            cfg.dynamicSmemBytes = kSmem;
            cfg.stream = stream;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = kGateCluster;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            if ((err = cudaLaunchKernelEx(&cfg, tc_state_pass, (const unsigned char *)region,
                                          seq_first_slot, order, cu_seqlens, T_fixed, init_state,
                                          static_cast<__nv_bfloat16 *>(out), final_state, H, status,
                                          sp, og, tz, tv)) != cudaSuccess)
                return err;
        } else if (P <= 1 && (long long)num_seqs * H * kTiles > 2LL * sm_count) {
            // Many chains: the 32-column pass would run in more than two waves,
            // so the 64-column pass, cheaper per column, finishes first.
            CUtensorMap tv64;
            memset(&tv64, 0, sizeof(tv64));
            if (tokens > 0 && (err = value_rows_map(&tv64, v, H, tokens, 64)) != cudaSuccess) return err;
            tc_state_pass64<<<(unsigned)num_seqs * H * (D / 64), kFusedThreads, P2L<64>::kSmem, stream>>>(
                region, seq_first_slot, order, cu_seqlens, T_fixed, init_state,
                static_cast<__nv_bfloat16 *>(out), final_state, H, status, tv64);
            if ((err = cudaGetLastError()) != cudaSuccess) return err;
        } else if (P <= 1) {
            const SegPass sp{1 << 30, 1, 0, 1, 0, nullptr, nullptr};
            tc_state_pass<<<(unsigned)num_seqs * H * kTiles, kP2Threads, kSmem, stream>>>(
                region, seq_first_slot, order, cu_seqlens, T_fixed, init_state,
                static_cast<__nv_bfloat16 *>(out), final_state, H, status, sp, og, tz, tv);
            if ((err = cudaGetLastError()) != cudaSuccess) return err;
        } else {
            const int L = (nch + P - 1) / P;
            const int Pn = (nch + L - 1) / L;  // no empty segment
            float *xfer = seg_ws;
            float *enter = seg_ws + (size_t)num_seqs * H * Pn * D * 2 * D;
            const SegPass sa{L, Pn, 0, Pn - 1, 1, xfer, enter};
            tc_state_pass<<<(unsigned)num_seqs * H * (Pn - 1) * 2 * kTiles, kP2Threads, kSmem,
                            stream>>>(region, seq_first_slot, order, cu_seqlens, T_fixed,
                                      init_state, static_cast<__nv_bfloat16 *>(out), final_state,
                                      H, status, sa, og, tz, tv);
            if ((err = cudaGetLastError()) != cudaSuccess) return err;
            if (Pn > 2) {
                seg_combine<<<(unsigned)num_seqs * H * (D / kCombCols), kCombThreads, kCombSmem,
                              stream>>>(xfer, enter, Pn);
                if ((err = cudaGetLastError()) != cudaSuccess) return err;
            }
            const SegPass sc{L, Pn, 1, Pn - 1, 0, xfer, enter};
            tc_state_pass<<<(unsigned)num_seqs * H * (Pn - 1) * kTiles, kP2Threads, kSmem,
                            stream>>>(region, seq_first_slot, order, cu_seqlens, T_fixed,
                                      init_state, static_cast<__nv_bfloat16 *>(out), final_state,
                                      H, status, sc, og, tz, tv);
            if ((err = cudaGetLastError()) != cudaSuccess) return err;
        }
    }
    return mark(events, 3, stream);
}

}  // namespace kda
