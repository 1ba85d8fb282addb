// Blackwell (sm_100 family) tensor-core plumbing in inline PTX: tensor-memory
// allocation, shared-memory matrix descriptors, tcgen05.mma (bf16 in, fp32 accumulate),
// commit to an mbarrier, bounded mbarrier waits and tensor-memory loads.
//
// Shared-memory operand layout used throughout ("no swizzle" canonical layout): the
// operand is cut into core matrices of 8 rows x 16 bytes (8 x 8 bf16), each stored as
// 128 contiguous bytes, one 16-byte row after the other.
//   K-major operand (K contiguous): core-matrix row = 8 consecutive k of one m/n row.
//     LBO = byte distance between core matrices adjacent along K,
//     SBO = byte distance between core matrices adjacent along M/N.
//   MN-major operand (M or N contiguous): core-matrix row = 8 consecutive m/n of one k.
//     LBO = byte distance between core matrices adjacent along K,
//     SBO = byte distance between core matrices adjacent along M/N.
//   (Both assignments were checked on B300 against a CPU GEMM for M = 128,
//   N in {64, 256}, K in {64, 128} and every combination of operand majors.)
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ssm {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Shared-memory matrix descriptor, no swizzle (layout type 0), descriptor version 1.
__device__ __forceinline__ uint64_t make_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Instruction descriptor for kind::f16 with bf16 A and B, fp32 D.
// a_mn / b_mn: operand stored MN-major (1) or K-major (0).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4)      // D format: f32
           | (1u << 7)    // A format: bf16
           | (1u << 10)   // B format: bf16
           | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Byte offset of element (row r, k) in a K-major operand tile with K columns.
__device__ __forceinline__ uint32_t off_kmajor(int r, int k, int K) {
    return (uint32_t)((r >> 3) * ((K >> 3) * 128) + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2);
}
// Byte offset of element (mn, k) in an MN-major operand tile with MN rows along M/N.
__device__ __forceinline__ uint32_t off_mnmajor(int mn, int k, int MN) {
    return (uint32_t)((k >> 3) * ((MN >> 3) * 128) + (mn >> 3) * 128 + (k & 7) * 16 + (mn & 7) * 2);
}

// Descriptor of k-step `ks` (16 elements of K) for the layouts above.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, int K, int ks) {
    return make_desc(base + (uint32_t)ks * 256u, 128u, (uint32_t)(K >> 3) * 128u);
}
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, int MN, int ks) {
    const uint32_t kstride = (uint32_t)(MN >> 3) * 128u;  // between core matrices along K
    return make_desc(base + (uint32_t)ks * 2u * kstride, kstride, 128u);
}

// Descriptor advance per k-step (16 elements of K), in units of the 16-byte address
// field: K-major tiles move 256 bytes, MN-major tiles two core matrices along K.
__host__ __device__ constexpr uint64_t kstep_kmajor() { return 256u >> 4; }
__host__ __device__ constexpr uint64_t kstep_mnmajor(int MN) { return (uint64_t)(2 * (MN >> 3) * 128) >> 4; }

// ---- tensor memory (one full warp executes these)
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
                 "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;"); }
// Make generic-proxy shared-memory writes visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;"); }

// D(tmem) (+)= A(smem) * B(smem); issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// Arrive once on `mbar` when every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
        smem_u32(mbar)));
}

__device__ __forceinline__ void mbar_init(uint64_t* mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(mbar)), "r"(count));
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;"); }

__device__ __forceinline__ bool mbar_try_wait(uint64_t* mbar, uint32_t phase) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(mbar)), "r"(phase));
    return done != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for `phase` of `mbar`: try_wait suspends the waiting thread in hardware
// between checks (so waiting warps take no issue slots from the working ones), and the
// wait gives up (returns false) after about one second of wall time or 2^24 checks,
// whichever comes first.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* mbar, uint32_t phase, uint32_t max_checks) {
    if (mbar_try_wait(mbar, phase)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; it < max_checks; ++it) {
        if (mbar_try_wait(mbar, phase)) return true;
        if ((it & 255u) == 0 && globaltimer_ns() - t0 > 1000000000ull) return false;
    }
    return false;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* mbar, uint32_t phase) {
    return mbar_wait_bounded(mbar, phase, 1u << 24);
}

// Load 16 consecutive fp32 columns of this warp's 32 TMEM lanes (lane = row).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Issue a load of 16 columns without waiting; complete with tmem_wait_ld().
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
// Issue a load of 8 columns without waiting; complete with tmem_wait_ld().
__device__ __forceinline__ void tmem_ld8_async(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_async(uint32_t taddr, uint32_t (&r)[16]) { tmem_ld16_async(taddr, r); }
__device__ __forceinline__ void tmem_ld_async(uint32_t taddr, uint32_t (&r)[8]) { tmem_ld8_async(taddr, r); }
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---- TMA (bulk asynchronous copies into shared memory, completion on an mbarrier)

// Expect `bytes` more transaction bytes on `mbar` and arrive once (one thread).
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(mbar)), "r"(bytes)
                 : "memory");
}

// Tiled 3-D tensor copy global -> shared: the box of the tensor map at coordinates
// (c0 innermost, c1, c2); elements outside the tensor are filled with zeros.  c0 times
// the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int c0, int c1, int c2, uint64_t* mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(mbar))
        : "memory");
}

// Contiguous bulk copy global -> shared of `bytes` (16-byte aligned addresses, a
// multiple of 16 bytes).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(mbar))
                 : "memory");
}

// Tiled 3-D tensor copy shared -> global of the tensor map's box at (c0, c1, c2), in the
// calling thread's bulk group; rows outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const void* tmap, const void* src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(src))
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until this thread's bulk groups have finished reading shared memory / completed.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Descriptor of a no-swizzle operand with explicit strides: lbo = bytes between core
// matrices adjacent along K, sbo = along M/N (the layouts written by TMA boxes that are
// 8 elements wide, one 16-byte core-matrix row per box row).
__device__ __forceinline__ uint64_t desc_strided(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return make_desc(saddr, lbo, sbo);
}

// Descriptor of an operand in the 128-byte swizzle layout that TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B (rows of 128 bytes, the 16-byte chunks of row r stored at
// chunk ^ (r % 8), groups of 8 rows 1024 bytes apart; the region 1024-byte aligned).
// K-major: 64 K-elements per row, K steps of 16 advance the start by 32 bytes inside a
// row; sbo = 1024.  MN-major with 64 MN-elements per row: K steps of 16 rows advance
// the start by 2048 bytes; the 8-row groups are 1024 bytes apart (lbo and sbo both 1024
// here, since one 64-element row covers the whole MN extent).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return make_desc(saddr, lbo, sbo) | ((uint64_t)2 << 61);
}

// TMEM address of (lane, column).
__device__ __forceinline__ uint32_t taddr(uint32_t base, uint32_t lane, uint32_t col) {
    return base + (lane << 16) + col;
}

}  // namespace tc
}  // namespace ssm
