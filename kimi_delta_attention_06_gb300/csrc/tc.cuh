// tc.cuh -- thin inline-PTX wrappers for the sm_100-family tensor-core path
// (tcgen05 MMA with TMEM accumulators, mbarriers, shared-memory descriptors).
//
// Layout conventions (shared-memory operand tiles written by threads):
//   * K-major, 128-byte swizzle: rows of 128 bytes (32 fp32/tf32 or 64 bf16
//     elements along K); 8-row groups of 1024 bytes are contiguous; the
//     16-byte chunk index inside a row is XOR-ed with (row % 8).  A tile with
//     more than one 128-byte K slab stores the slabs one after another, each
//     slab holding all rows.  Tile bases are 1024-byte aligned.
//   * MN-major, 128-byte swizzle: the same physical arrangement with the roles
//     swapped: each 128-byte row runs along M (or N) and rows are K indices.
// These two coincide physically, so one tile can serve as a K-major operand
// of one MMA and as an MN-major operand of another.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace kda {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- shared-memory matrix descriptor -----------------------------------------------
// bits  0-13 start address >> 4, 16-29 leading byte offset >> 4,
// bits 32-45 stride byte offset >> 4, 46-47 version (1), 61-63 layout/swizzle.
enum : uint32_t { kSwizzleNone = 0, kSwizzle128B = 2, kSwizzle64B = 4, kSwizzle32B = 6 };

__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(swz & 0x7u) << 61;
    return d;
}

// ---- instruction descriptor (kind::f16 / kind::tf32) -------------------------------
// bits 4-5 D format (1 = f32), 7-9 A format, 10-12 B format
// (kind::f16: 0 = f16, 1 = bf16; kind::tf32: 2 = tf32), bit 15 A major,
// bit 16 B major (0 = K-major, 1 = MN-major), 17-22 N >> 3, 24-28 M >> 4.
enum : uint32_t { kFmtF16 = 0, kFmtBF16 = 1, kFmtTF32 = 2 };

__host__ __device__ constexpr uint32_t idesc(int M, int N, uint32_t fmt, bool a_mn, bool b_mn) {
    return (1u << 4) | (fmt << 7) | (fmt << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// ---- MMA issue (one thread) --------------------------------------------------------------
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n"
        :: "r"(d_tmem), "l"(a), "l"(b), "r"(id), "r"(acc));
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n"
        :: "r"(d_tmem), "l"(a), "l"(b), "r"(id), "r"(acc));
}

// Arrive on an mbarrier once all previously issued MMAs of this thread complete.
__device__ __forceinline__ void mma_commit(void* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}

// ---- TMEM allocation (whole warp) ---------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Make generic-proxy shared-memory writes visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_smem_to_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- TMEM -> registers: 32 lanes x 32 bit, 16 consecutive columns ------------------------
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&r)[16]) {
    uint32_t* u = reinterpret_cast<uint32_t*>(r);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
          "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]),
          "=r"(u[13]), "=r"(u[14]), "=r"(u[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- mbarrier -----------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(void* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ uint32_t mbar_try_wait(void* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for phase `parity` of an mbarrier, giving up after `limit_ns`.
// Returns 1 when the phase completed, 0 on timeout.
__device__ __forceinline__ uint32_t mbar_wait_bounded(void* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return 1;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return 1;
        if (globaltimer_ns() - t0 > limit_ns) return 0;
    }
}

// ---- swizzled tile addressing ----------------------------------------------------------------
// Byte offset of 32-bit element (row, col) in a 128B-swizzled tile of `rows` rows whose
// 128-byte slabs (32 elements of `col`) are stored one after another.
__host__ __device__ __forceinline__ uint32_t sw128_off32(uint32_t row, uint32_t col, uint32_t rows) {
    const uint32_t slab = col >> 5, cb = (col & 31u) * 4u;
    return slab * rows * 128u + row * 128u + ((((cb >> 4) ^ (row & 7u)) << 4) | (cb & 15u));
}
// Same for 16-bit elements (64 per 128-byte row).
__host__ __device__ __forceinline__ uint32_t sw128_off16(uint32_t row, uint32_t col, uint32_t rows) {
    const uint32_t slab = col >> 6, cb = (col & 63u) * 2u;
    return slab * rows * 128u + row * 128u + ((((cb >> 4) ^ (row & 7u)) << 4) | (cb & 15u));
}

}  // namespace tc
}  // namespace kda

namespace kda {
namespace tc {

// Named CTA barrier over `nthreads` threads (a multiple of 32) with id 1..15.
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ANDs a predicate across the participating threads.
__device__ __forceinline__ uint32_t named_sync_and(uint32_t id, uint32_t nthreads, uint32_t pred) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %3, 0;\n\t"
        "bar.red.and.pred q, %1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(out) : "r"(id), "r"(nthreads), "r"(pred) : "memory");
    return out;
}

__device__ __forceinline__ void mbar_arrive(void* bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}\n"
                 :: "r"(smem_u32(bar)) : "memory");
}

}  // namespace tc
}  // namespace kda

namespace kda {
namespace tc {

// ---- thread-block clusters / distributed shared memory -------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Shared::cluster address of the same variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t local_saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive (release at cluster scope) on an mbarrier of another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(cluster_addr) : "memory");
}
// try_wait with cluster-scope acquire (for phases completed by remote arrivals).
__device__ __forceinline__ uint32_t mbar_try_wait_cluster(void* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok;
}
__device__ __forceinline__ uint32_t mbar_wait_cluster_bounded(void* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait_cluster(bar, parity)) return 1;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return 1;
        if (globaltimer_ns() - t0 > limit_ns) return 0;
    }
}

}  // namespace tc
}  // namespace kda

namespace kda {
namespace tc {

// ---- TMA (tensor bulk copies) ------------------------------------------------------------
__device__ __forceinline__ void mbar_arrive_expect_tx(void* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
// 2-D tiled TMA store of a shared-memory box to coordinates (x, y), tracked in the issuing
// thread's current bulk group.  x * element size must be a multiple of 16 bytes, x, y >= 0.
__device__ __forceinline__ void tma_store_2d(const void* tmap, uint32_t src_smem, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                 :: "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(src_smem) : "memory");
}
// Prefetch the box at coordinates (x, y) of a tensor map into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_2d(const void* tmap, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];"
                 :: "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y) : "memory");
}
// 2-D tiled TMA load of the box at coordinates (x, y) into this CTA's shared memory;
// completion is reported as transaction bytes on `bar`.  x * element size must be a
// multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst_smem, const void* tmap, int x, int y, void* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst_smem), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar)) : "memory");
}

}  // namespace tc
}  // namespace kda

namespace kda {
namespace tc {

// Relaxed remote arrival: a pure signal, ordering no memory accesses of this thread.
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" :: "r"(cluster_addr) : "memory");
}
// Non-blocking probe of an mbarrier phase.
__device__ __forceinline__ uint32_t mbar_test_wait(void* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok;
}

}  // namespace tc
}  // namespace kda

namespace kda {
namespace tc {

// ---- bulk copies between shared and global memory ----------------------------------------
// Store `bytes` (multiple of 16) of this CTA's shared memory to global memory, tracked in
// the issuing thread's current bulk group.
__device__ __forceinline__ void bulk_store_s2g(void* gdst, uint32_t src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :: "l"(gdst), "r"(src_smem), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every bulk group of this thread has completed (its writes are performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Wait until every bulk group of this thread has finished reading its source.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Load `bytes` (multiple of 16) from global memory into this CTA's shared memory;
// completion is counted as transaction bytes on `bar`.
__device__ __forceinline__ void bulk_load_g2s(uint32_t dst_smem, const void* gsrc, uint32_t bytes, void* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst_smem), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
// Order this thread's global accesses between the generic and the async proxy.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Non-blocking probe with cluster-scope acquire (phases completed by remote arrivals).
__device__ __forceinline__ uint32_t mbar_test_wait_cluster(void* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok;
}

}  // namespace tc
}  // namespace kda
