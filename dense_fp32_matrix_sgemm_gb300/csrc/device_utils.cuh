// Small device-side helpers shared by the SGEMM kernels: asynchronous
// global->shared copies (cp.async, sm_80+), shared-memory addresses, and
// thread-block-cluster primitives (rank, barrier, distributed shared memory).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sgemm {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous copy that reads `src_bytes` (0..16) bytes and zero-fills
// the rest of the destination; with src_bytes == 0 nothing is read.
// Bypasses L1 (.cg): each tile element is staged in shared memory exactly once.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n"
                 :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// 4-byte asynchronous copy with the same zero-fill rule (src_bytes 0 or 4).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void *src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n"
                 :: "r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" :: "n"(N) : "memory");
}

__device__ __forceinline__ float4 ldg_f4(const float *p) {
    return __ldg(reinterpret_cast<const float4 *>(p));
}

// Rank of this CTA within its cluster, and the number of CTAs in the cluster.
// Programmatic dependent launch.  pdl_wait: the calling thread waits until
// the grids this launch depends on have completed and their memory is
// visible (returns at once when the launch has no such dependency).
// pdl_trigger: this CTA allows the next launch in the stream, if it was
// launched as a programmatic dependent, to start being scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t n;
    asm volatile("mov.u32 %0, %%cluster_nctarank;\n" : "=r"(n));
    return n;
}

// Cluster-wide barrier: every thread of every CTA in the cluster arrives; the
// release/acquire pair makes shared-memory writes made before it visible to
// distributed-shared-memory reads after it.  Not the .aligned form, so
// threads need not be converged when they reach it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n"
                 "barrier.cluster.wait.acquire;\n" ::: "memory");
}

// Cluster-wide barrier that orders nothing: a CTA passes it once every CTA
// of the cluster has arrived.  For the barrier that keeps a CTA's shared
// memory alive until its peers have read it: each reading thread has used
// the values it loaded before it arrives, so no release is needed.
__device__ __forceinline__ void cluster_sync_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed;\n"
                 "barrier.cluster.wait;\n" ::: "memory");
}

// 16-byte load from the shared memory of CTA `rank` of this cluster, at the
// offset that `local` (a shared::cta address) has in this CTA.
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(remote) : "r"(local), "r"(rank));
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(remote) : "memory");
    return v;
}

// Sum over ranks 0..n-1 (n <= 16) of the float4 at the offset `local` has in
// each CTA of the cluster, added in rank order.  All n loads are issued before
// the first add, so their latencies overlap instead of adding up.
__device__ __forceinline__ float4 cluster_sum_f4(uint32_t local, uint32_t n) {
    float4 v[16];
#pragma unroll
    for (uint32_t q = 0; q < 16; ++q)
        if (q < n) v[q] = ld_cluster_f4(local, q);
    float4 sum = v[0];
#pragma unroll
    for (uint32_t q = 1; q < 16; ++q) {
        if (q < n) {
            sum.x += v[q].x;
            sum.y += v[q].y;
            sum.z += v[q].z;
            sum.w += v[q].w;
        }
    }
    return sum;
}

// 4-byte load from the shared memory of CTA `rank` of this cluster.
__device__ __forceinline__ float ld_cluster_f32(uint32_t local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(remote) : "r"(local), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];\n" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// cluster_sum_f4 for one float.
__device__ __forceinline__ float cluster_sum_f32(uint32_t local, uint32_t n) {
    float v[16];
#pragma unroll
    for (uint32_t q = 0; q < 16; ++q)
        if (q < n) v[q] = ld_cluster_f32(local, q);
    float sum = v[0];
#pragma unroll
    for (uint32_t q = 1; q < 16; ++q)
        if (q < n) sum += v[q];
    return sum;
}

}  // namespace sgemm
