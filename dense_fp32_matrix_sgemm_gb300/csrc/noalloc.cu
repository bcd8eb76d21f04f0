// sgemm_f32_tf32x3_noalloc: the 3xTF32 tensor-core product with its scratch
// taken from memory the library reserves for itself, so the call allocates
// nothing and needs no workspace argument.
//
// The scratch is the file-scope array below.  Host code cannot use the
// array's name as a device address (in host code it names a host-side
// stand-in), so the device address is looked up with cudaGetSymbolAddress,
// once per context with that context current, and handed to the kernels.
#include <cstdio>
#include <mutex>

#include <cuda_runtime.h>

#include "gemm_args.h"
#include "sgemm_gb300.h"

namespace sgemm {

int record_error(int code, const char *msg);

namespace {

// 64 MiB of device scratch, held by every GPU that loads this library until
// the process exits.
constexpr unsigned long long kNoallocScratchBytes = 64ull << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of the scratch in the current context, looked up with
// cudaGetSymbolAddress the first time a call runs in that context (which also
// makes the runtime set up the device's context if it is not yet current).
// The cache is keyed on the context's unique id, not on the device number:
// after cudaDeviceReset, or with another context made current, the address is
// looked up again instead of reusing one that belongs to a dead or different
// context.
int scratch_for_current_context(void **out) {
    static PerContext<void *> cached;
    void *p = nullptr;
    if (cached.get(current_context_id(), p)) {
        *out = p;
        return SGEMM_OK;
    }
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
        char msg[256];
        snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the built-in scratch failed: %s",
                 cudaGetErrorString(e));
        return record_error(SGEMM_EDEVICE, msg);
    }
    cached.put(current_context_id(), p);
    *out = p;
    return SGEMM_OK;
}

}  // namespace
}  // namespace sgemm

extern "C" uint64_t sgemm_f32_tf32x3_noalloc_max_bytes(void) {
    return sgemm::kNoallocScratchBytes;
}

extern "C" int sgemm_f32_tf32x3_noalloc(int64_t M, int64_t N, int64_t K, const float *A,
                                        int64_t lda, const float *B, int64_t ldb, float *C,
                                        int64_t ldc, int transA, int transB, void *stream) {
    // Sizes beyond the built-in scratch are rejected before anything runs.
    // The planes must fit; the stream-K schedule's partial tiles are used
    // when they fit too, exactly as sgemm_f32_tf32x3 does with a workspace of
    // this size.
    const uint64_t need =
        (M <= 0 || N <= 0 || K <= 0) ? 0 : sgemm::tf32x3_workspace_min_bytes(M, N, K, 1);
    if (need > sgemm::kNoallocScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "M=%lld N=%lld K=%lld needs %llu bytes of scratch; the built-in scratch of "
                 "sgemm_f32_tf32x3_noalloc holds %llu bytes (2*(M+N)*round_up(K,32)*4 must fit)",
                 (long long)M, (long long)N, (long long)K, (unsigned long long)need,
                 sgemm::kNoallocScratchBytes);
        return sgemm::record_error(SGEMM_EWORKSPACE, msg);
    }
    void *scratch = nullptr;
    if (need > 0) {
        const int st = sgemm::scratch_for_current_context(&scratch);
        if (st != SGEMM_OK) return st;
    }
    // The split kernels write every scratch element the GEMM kernel reads, so
    // nothing has to be cleared between calls.
    return sgemm_f32_tf32x3(M, N, K, A, lda, B, ldb, C, ldc, transA, transB, scratch,
                            sgemm::kNoallocScratchBytes, stream);
}
