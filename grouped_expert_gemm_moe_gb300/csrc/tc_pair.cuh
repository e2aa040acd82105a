// tc_pair.cuh -- CTA-pair (cluster of 2, tcgen05 cta_group::2) pieces shared
// by the pair grouped GEMMs: cluster ids, cross-CTA barrier signals, TMA
// loads that complete on the pair's CTA 0 barrier, pair MMAs and commits.
#pragma once

#include "tc_common.cuh"

namespace moe {

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// Shared::cluster address of the object at shared address `addr` in the
// cluster's CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// All threads of both CTAs; orders each CTA's earlier shared-memory work
// (barrier initialisation, remote arrivals) before the other's later work.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive on a barrier of either CTA of the pair (a shared::cluster address)
// with the default, CTA-scope release.  The pair's thread-to-thread hand-offs
// are of tensor memory, whose order comes from the tcgen05 waits and fences
// around the barrier (tcgen05.wait::st or ::ld, then
// fence::before_thread_sync, before the arrive; fence::after_thread_sync
// after the wait), and the waiter only needs the arrival itself; TMA bytes
// are counted on the barriers by the copies.  A cluster-scope release (or
// acquire) on these barriers cost 0.3-0.9 us per hand-off under load: it
// waits for the SM's outstanding memory traffic.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// 2-D tiled TMA load into this CTA's shared memory whose completion is
// counted on `bar_cluster` (a shared::cluster address: this CTA's barrier or
// the pair's CTA 0 barrier).
__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *map,
                                                 uint32_t bar_cluster, int x, int y,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster), "l"(policy)
        : "memory");
}

// The same for a 3-D box (x = k, y = row, z = plane).
__device__ __forceinline__ void tma_load_3d_pair(void *dst, const CUtensorMap *map,
                                                 uint32_t bar_cluster, int x, int y, int z,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar_cluster),
        "l"(policy)
        : "memory");
}

// The same for a 4-D box (x = k, then y, z, w).
__device__ __forceinline__ void tma_load_4d_pair(void *dst, const CUtensorMap *map,
                                                 uint32_t bar_cluster, int x, int y, int z, int w,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar_cluster),
        "l"(policy)
        : "memory");
}

// The same for a 5-D box (x = k, then y, z, w, v).
__device__ __forceinline__ void tma_load_5d_pair(void *dst, const CUtensorMap *map,
                                                 uint32_t bar_cluster, int x, int y, int z, int w,
                                                 int v, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(v),
        "r"(bar_cluster), "l"(policy)
        : "memory");
}

template <uint32_t NCOLS>
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *slot) {   // one warp in each CTA
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(slot)),
                 "n"(NCOLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

template <uint32_t NCOLS>
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr) {   // one warp in each CTA
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "n"(NCOLS)
                 : "memory");
}

__device__ __forceinline__ void tc_mma_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the barrier at `bar`'s offset in both CTAs of the pair when
// every MMA this thread issued so far has completed.
__device__ __forceinline__ void tc_commit_pair_both(uint64_t *bar) {
    const uint16_t mask = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(mask)
        : "memory");
}

// The same, on this CTA's barrier only.
__device__ __forceinline__ void tc_commit_pair_local(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ int abox_rows(int rows) {
    return rows <= 0 ? 0 : rows <= 16 ? 16 : rows <= 32 ? 32 : rows <= 64 ? 64 : 128;
}

}  // namespace moe
