// Thread-block cluster helpers (sm_90+): the CTA's rank and the cluster
// counts, the cluster-wide barrier, and a load from a peer CTA's shared
// memory (distributed shared memory).
#pragma once

#include <stdint.h>

namespace rn {

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t n;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(n));
    return n;
}
__device__ __forceinline__ uint32_t cluster_index_x() {
    uint32_t i;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(i));
    return i;
}
__device__ __forceinline__ uint32_t cluster_size_x() {
    uint32_t n;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return n;
}
// Every thread of every CTA of the cluster arrives; shared-memory writes
// before it are visible to the cluster after it. The aligned cluster barrier
// needs each warp converged when it gets there (see named_barrier_sync in
// common.cuh): __syncwarp() first.
__device__ __forceinline__ void cluster_sync_all() {
    __syncwarp();
    asm volatile(
        "barrier.cluster.arrive.release.aligned;\n\t"
        "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ float ld_peer_f32(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    float v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

}  // namespace rn
