// Small device-side helpers shared by the SGEMM kernels: asynchronous
// global->shared copies (cp.async, sm_80+) and shared-memory addresses.
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

}  // namespace sgemm
