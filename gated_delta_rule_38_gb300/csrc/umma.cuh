// Blackwell (sm_103a) tensor-core helpers: tcgen05 MMA with TMEM accumulators,
// shared-memory operand descriptors, mbarrier waits with an iteration bound.
//
// Operand tiles use the 128-byte swizzle: a tile is a set of 64-element-wide
// (128-byte) column blocks; inside a block, row r's 16-byte chunk c sits at
// chunk position c ^ (r & 7); blocks start on 1024-byte boundaries.  The same
// bytes serve as a K-major operand (rows = M/N index, columns = K) and as an
// MN-major operand (rows = K index, columns = M/N index).
#pragma once

#include <stdint.h>

namespace gdr {
namespace umma {

// Byte offset of (row, col) in a swizzled tile whose 64-column blocks are `block_bytes` apart.
__device__ __forceinline__ uint32_t off(int row, int col, uint32_t block_bytes) {
    return (uint32_t)(col >> 6) * block_bytes + (uint32_t)row * 128u +
           ((uint32_t)(((col & 63) >> 3) ^ (row & 7)) << 4) + (uint32_t)(col & 7) * 2u;
}

// Shared-memory matrix descriptor, 128-byte swizzle.
//   K-major operand : lbo unused (16), sbo = byte stride between 8-row groups (1024).
//   MN-major operand: lbo = byte stride between 64-wide M/N blocks, sbo = stride between 8 K-row groups (1024).
__device__ __forceinline__ uint64_t desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version
    d |= (uint64_t)2 << 61;  // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16, fp32 accumulation.  bf16 selects bf16 (else fp16) operands.
__device__ __forceinline__ uint32_t idesc(int M, int N, bool bf16, bool a_mn, bool b_mn) {
    uint32_t d = 1u << 4;  // D = f32
    if (bf16) d |= (1u << 7) | (1u << 10);
    d |= (uint32_t)a_mn << 15;
    d |= (uint32_t)b_mn << 16;
    d |= (uint32_t)(N >> 3) << 17;
    d |= (uint32_t)(M >> 4) << 24;
    return d;
}

__device__ __forceinline__ void mma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t id, bool accumulate) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(id), "r"((uint32_t)accumulate));
}

__device__ __forceinline__ void commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(mbar));
}

__device__ __forceinline__ void mbar_init(uint32_t mbar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(mbar), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::); }

// Wait for the phase with the given parity; gives up after `limit` polls and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity, long limit = 200000000L) {
    uint32_t done = 0;
    for (long it = 0; it < limit; ++it) {
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(mbar), "r"(parity));
        if (done) return true;
    }
    return false;
}

// The same wait by spinning on a non-suspending test: a thread that has waited a long time in try_wait was
// seen to resume several hundred cycles after the phase completed, so waits on a critical path spin.
__device__ __forceinline__ bool mbar_spin(uint32_t mbar, uint32_t parity, long limit = 200000000L) {
    uint32_t done = 0;
    for (long it = 0; it < limit; ++it) {
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(mbar), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::); }
// Generic-proxy shared stores -> visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::); }

// Warp-collective TMEM allocation (ncols a power of two >= 32); the address lands in *slot.
__device__ __forceinline__ void alloc(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(slot_smem), "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::);
}
__device__ __forceinline__ void dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols));
}

// 32 lanes x 16 consecutive fp32 columns (warp w reads lanes 32*(w%4)..).
__device__ __forceinline__ void ld16(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::); }

// TMEM address of (lane, column) relative to a base returned by alloc.
__device__ __forceinline__ uint32_t taddr(uint32_t base, int lane, int col) {
    return base + ((uint32_t)lane << 16) + (uint32_t)col;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d));
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 u;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n" : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w) : "r"(addr));
    return u;
}

}  // namespace umma
}  // namespace gdr

namespace gdr {
namespace tma {

// 3-D tiled bulk tensor load into shared memory; completion is counted in bytes on `mbar`.
// `map` must live in kernel-parameter (grid-constant) memory.
__device__ __forceinline__ void load3d(uint32_t dst, const void *map, int c0, int c1, int c2, uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];\n" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(mbar)
        : "memory");
}

// A hint that brings a box into L2 ahead of its load (no shared memory, no completion to wait for).
__device__ __forceinline__ void prefetch3d(const void *map, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];\n" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

// 3-D tiled bulk tensor store from shared memory (same box and swizzle as the loads), as one bulk group of the
// issuing thread; `commit_group` closes the group, `wait_read` waits until the thread's groups have finished
// reading shared memory, `wait_all` until they are complete.
__device__ __forceinline__ void store3d(const void *map, int c0, int c1, int c2, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];\n" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void commit_group() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory"); }
// ... until all but the most recent group have finished reading shared memory
__device__ __forceinline__ void wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;\n" ::: "memory"); }
__device__ __forceinline__ void wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }

// Plain (untiled) bulk copy of `bytes` contiguous bytes from global into shared memory, completion counted in
// bytes on `mbar`.  Both addresses 16-byte aligned, `bytes` a multiple of 16.
__device__ __forceinline__ void load1d(uint32_t dst, const void *src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(mbar)
                 : "memory");
}

// One arrival that also announces `bytes` of transactions on the barrier's current phase.
__device__ __forceinline__ void expect_tx(uint32_t mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(mbar), "r"(bytes) : "memory");
}

}  // namespace tma
}  // namespace gdr
