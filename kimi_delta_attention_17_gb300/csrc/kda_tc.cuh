// Inline-PTX helpers for the tensor-core (tcgen05 / TMEM / bulk-copy)
// kernels of the prefill. sm_100-family only.
//
// Shared-memory operand tiles use the no-swizzle canonical layouts of
// tcgen05.mma: 8 x 16-byte "core matrices" of 128 contiguous bytes. In a
// K-major tile a core holds 8 rows (M or N index) x 8 consecutive K elements;
// in an MN-major tile a core holds 8 consecutive K rows x 8 consecutive M/N
// elements. The descriptor's leading byte offset (LBO) is the distance between
// cores adjacent along K, its stride byte offset (SBO) the distance between
// cores adjacent along M/N.
#pragma once

#include <stdint.h>

namespace kda {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Byte offset of element (mn, k) of a 16-bit K-major tile.
__host__ __device__ constexpr uint32_t kmaj(int mn, int k, uint32_t lbo, uint32_t sbo) {
    return (uint32_t)(mn >> 3) * sbo + (uint32_t)(k >> 3) * lbo + (uint32_t)(mn & 7) * 16u +
           (uint32_t)(k & 7) * 2u;
}
// Byte offset of element (mn, k) of a 16-bit MN-major tile.
__host__ __device__ constexpr uint32_t mnmaj(int mn, int k, uint32_t lbo, uint32_t sbo) {
    return (uint32_t)(mn >> 3) * sbo + (uint32_t)(k >> 3) * lbo + (uint32_t)(k & 7) * 16u +
           (uint32_t)(mn & 7) * 2u;
}

// Shared-memory matrix descriptor, no swizzle.
__device__ __forceinline__ uint64_t desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor: kind::f16 with bf16 A and B, fp32 accumulator.
// a_mn / b_mn select MN-major (1) or K-major (0) operands.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A * B^T over one K=16 step.
__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{.reg .pred p; setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;}" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void commit(uint64_t *mbar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(mbar))
        : "memory");
}

__device__ __forceinline__ void fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Makes this thread's generic-proxy shared-memory writes visible to the
// async proxy (tensor core, bulk copies).
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Allocates `ncols` TMEM columns (power of two >= 32); one whole warp calls.
template <int ncols>
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "n"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
template <int ncols>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "n"(ncols));
}

// 16 consecutive fp32 columns of this thread's TMEM lane (warp-collective;
// the address must name the warp's own 32-lane slice).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%"
        "15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// 8 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t *mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(mbar)), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(mbar)),
                 "r"(bytes)
                 : "memory");
}
// Arrives once on mbar (no transaction bytes).
__device__ __forceinline__ void mbar_arrive(uint64_t *mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(mbar)) : "memory");
}
// Named barrier `id` of `nthreads` threads (whole warps): arrive without
// waiting, or arrive and wait for the others.
__device__ __forceinline__ void bar_arrive(int id, int nthreads) {
    asm volatile("barrier.cta.arrive.aligned %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void bar_sync(int id, int nthreads) {
    asm volatile("barrier.cta.sync.aligned %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Barrier `id` over `nthreads` threads (whole warps) that also returns whether
// `pred` holds in every one of them (bar_and) or in any (bar_or).
__device__ __forceinline__ bool bar_and(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{.reg .pred p, q; setp.ne.u32 p, %1, 0; barrier.cta.red.and.aligned.pred q, %2, %3, p; "
        "selp.u32 %0, 1, 0, q;}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ bool bar_or(int id, int nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{.reg .pred p, q; setp.ne.u32 p, %1, 0; barrier.cta.red.or.aligned.pred q, %2, %3, p; "
        "selp.u32 %0, 1, 0, q;}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}
// A flag in global memory handed from one CTA to another: the writer's
// release orders every earlier write it has seen (a barrier before it makes
// its CTA's writes seen) before the flag; the reader's acquire orders its
// later reads after it.
__device__ __forceinline__ void st_release_gpu(int *p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Orders this thread's earlier generic-proxy accesses of global memory (such
// as an acquire of data another CTA wrote) before its later async-proxy ones
// (bulk and tensor copies).
__device__ __forceinline__ void fence_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Barrier `id` over `nthreads` threads of the CTA (whole warps),
// returning whether `pred` held in every one of them.
__device__ __forceinline__ bool bar_and(bool pred, int id, int nthreads) {
    uint32_t r;
    asm volatile(
        "{.reg .pred p, q; setp.ne.u32 p, %1, 0; barrier.cta.red.and.aligned.pred q, %2, %3, p; "
        "selp.u32 %0, 1, 0, q;}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}
// Bounded wait for the phase with the given parity to complete. Returns false
// if it gave up (after roughly a second or more of polling). A phase that has
// already completed is seen by the first, non-blocking test.
__device__ __forceinline__ bool mbar_wait(uint64_t *mbar, uint32_t parity, uint32_t limit = 1u << 22);
__device__ __forceinline__ bool mbar_wait(uint64_t *mbar, uint32_t parity, uint32_t limit) {
    const uint32_t a = smem_u32(mbar);
    {
        uint32_t done;
        asm volatile(
            "{.reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, "
            "0, p;}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
    }
    for (uint32_t it = 0; it < limit; ++it) {
        uint32_t ok;
        asm volatile(
            "{.reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, "
            "0, p;}"
            : "=r"(ok)
            : "r"(a), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    return false;
}

// One non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test(uint64_t *mbar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{.reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, "
        "p;}"
        : "=r"(done)
        : "r"(smem_u32(mbar)), "r"(parity)
        : "memory");
    return done != 0;
}
// Up to 4096 non-blocking tests; returns whether the phase completed.
__device__ __forceinline__ bool mbar_poll(uint64_t *mbar, uint32_t parity) {
    for (int it = 0; it < 4096; ++it)
        if (mbar_test(mbar, parity)) return true;
    return false;
}

// Bounded wait that polls with the non-blocking test (no suspend and wake-up
// in between): for waits on the critical path whose phase completes within a
// few hundred cycles. Falls back to the blocking wait after 4096 polls.
__device__ __forceinline__ bool mbar_spin(uint64_t *mbar, uint32_t parity) {
    const uint32_t a = smem_u32(mbar);
    for (int it = 0; it < 4096; ++it) {
        uint32_t done;
        asm volatile(
            "{.reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, "
            "0, p;}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return mbar_wait(mbar, parity);
}

// ---- thread-block clusters (distributed shared memory; no multicast)

// This CTA's rank within its cluster.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The shared::cluster address of the variable at `p` (this CTA's shared
// memory) in the CTA of rank `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_addr(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// Asynchronous 4-byte store into the shared memory of a CTA of the cluster
// (cluster addresses), completing 4 transaction bytes on that CTA's mbarrier;
// no fence: the mbarrier's phase completion publishes the value.
__device__ __forceinline__ void st_async_cluster_f32(uint32_t addr, float v, uint32_t mbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(
                     addr),
                 "f"(v), "r"(mbar)
                 : "memory");
}
// The same for 16 bytes (four consecutive floats; addr 16-byte aligned).
__device__ __forceinline__ void st_async_cluster_v4(uint32_t addr, float4 v, uint32_t mbar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
            addr),
        "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(mbar)
        : "memory");
}
// Arrives once on the mbarrier at cluster address `addr`, releasing this
// thread's earlier writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr)
                 : "memory");
}
// Bounded wait on a local mbarrier whose arrivals come from other CTAs of the
// cluster (acquire at cluster scope). Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *mbar, uint32_t parity,
                                                  uint32_t limit = 1u << 22) {
    const uint32_t a = smem_u32(mbar);
    for (uint32_t it = 0; it < limit; ++it) {
        uint32_t ok;
        asm volatile(
            "{.reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; "
            "selp.u32 %0, 1, 0, p;}"
            : "=r"(ok)
            : "r"(a), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    return false;
}
// One non-blocking test of such a barrier (acquire at cluster scope).
__device__ __forceinline__ bool mbar_test_cluster(uint64_t *mbar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{.reg .pred p; mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; "
        "selp.u32 %0, 1, 0, p;}"
        : "=r"(done)
        : "r"(smem_u32(mbar)), "r"(parity)
        : "memory");
    return done != 0;
}
// Barrier over every thread of every CTA of the cluster (release / acquire).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// 16-byte asynchronous copy global -> shared (cp.async); with src_bytes < 16
// the rest of the 16 bytes is filled with zeros (src_bytes = 0: zeros only).
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
// An arrival on mbar once every earlier cp.async of this thread has landed
// (the arrival is one of the barrier's expected count).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t *mbar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(mbar))
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// 1-D bulk copy global -> shared, completing `bytes` transactions on mbar.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *mbar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(mbar))
        : "memory");
}

// 3-D tiled TMA load of one box of `map` at element coordinates (x, y, z)
// into shared memory, completing its bytes on mbar. `map` is the address of a
// __grid_constant__ CUtensorMap kernel parameter.
__device__ __forceinline__ void tma_load_3d(void *dst, const void *map, int x, int y, int z,
                                            uint64_t *mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
        "{%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(mbar))
        : "memory");
}

// Packs 8 floats as 8 bf16 (round to nearest even), two per instruction,
// into one 16-byte vector (element 0 in the lowest half-word).
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint4 pack8(const float *x) {
    return make_uint4(pack2(x[0], x[1]), pack2(x[2], x[3]), pack2(x[4], x[5]), pack2(x[6], x[7]));
}
// Splits x0, x1 into bf16 pairs with x ~ hi + lo: hi keeps the upper 16 bits
// of each float (truncation, one byte permute for the pair), lo = x - hi is
// exact in fp32 and rounds once to bf16, so hi + lo carries 16 significant
// bits (|x - hi - lo| <= 2^-16 |x|).
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const uint32_t u0 = __float_as_uint(x0), u1 = __float_as_uint(x1);
    hi = __byte_perm(u0, u1, 0x7632);
    lo = pack2(x0 - __uint_as_float(u0 & 0xFFFF0000u), x1 - __uint_as_float(u1 & 0xFFFF0000u));
}
// split2 over 8 values: two 16-byte vectors (hi, lo).
__device__ __forceinline__ void split8(const float *x, uint4 &hi, uint4 &lo) {
    split2(x[0], x[1], hi.x, lo.x);
    split2(x[2], x[3], hi.y, lo.y);
    split2(x[4], x[5], hi.z, lo.z);
    split2(x[6], x[7], hi.w, lo.w);
}

}  // namespace tc
}  // namespace kda
