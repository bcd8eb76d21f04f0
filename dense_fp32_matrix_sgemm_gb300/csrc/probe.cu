// Peak probes: FP32 FMA throughput (the measured denominator of "% of FP32
// peak") and the TF32 tensor-pipe throughput of tcgen05.mma; the raster-group
// and chunk-length knobs that measurements of the block order's L2 reuse and
// of the K-chunked kernel's accuracy use.
#include <atomic>
#include <cstdint>

#include <cuda_runtime.h>

#include "sgemm_gb300.h"
#include "gemm_args.h"
#include "sgemm_gb300_probe.h"

namespace sgemm {
namespace {

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 8;
constexpr int kChains = 16;   // independent float2 chains per thread

template <bool PACKED>
__global__ void __launch_bounds__(kThreads) fp32_probe_kernel(float *out, long long iters) {
    // x <- x * m + c converges to c / (1 - m) = 1; values stay normal.
    const float m = 0.9990234375f, c = 1.0f - m;
    float2 x[kChains];
#pragma unroll
    for (int j = 0; j < kChains; ++j)
        x[j] = make_float2(0.5f + 0.01f * j + 1e-6f * threadIdx.x, 0.25f + 0.01f * j);
    const float2 m2 = make_float2(m, m), c2 = make_float2(c, c);
    for (long long i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < kChains; ++j) {
            if constexpr (PACKED) {
                x[j] = __ffma2_rn(x[j], m2, c2);
            } else {
                x[j].x = fmaf(x[j].x, m, c);
                x[j].y = fmaf(x[j].y, m, c);
            }
        }
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kChains; ++j) s += x[j].x + x[j].y;
    out[blockIdx.x * (int64_t)blockDim.x + threadIdx.x] = s / (2 * kChains);
}

int64_t probe_ctas() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return (int64_t)sms * kCtasPerSm;
}

std::atomic<int> g_raster_group{8};

}  // namespace

int raster_group() { return g_raster_group.load(std::memory_order_relaxed); }

}  // namespace sgemm

extern "C" int sgemm_set_raster_group(int group_m) {
    if (group_m < 0 || group_m > 65536) return -1;
    return sgemm::g_raster_group.exchange(group_m == 0 ? 8 : group_m);
}

extern "C" int sgemm_set_tf32x3_chunk_k(int chunk_k) { return sgemm::set_tf32x3_chunk_k(chunk_k); }

extern "C" int64_t sgemm_probe_out_elems(void) { return sgemm::probe_ctas() * sgemm::kThreads; }

extern "C" int sgemm_probe_fp32_fma(int packed, int64_t iterations, float *out, double *flops_out,
                                    void *stream) {
    if ((packed != 0 && packed != 1) || iterations <= 0) return SGEMM_EINVAL_DIM;
    if (out == nullptr || flops_out == nullptr) return SGEMM_EINVAL_PTR;
    const int64_t ctas = sgemm::probe_ctas();
    if (ctas <= 0) return SGEMM_EDEVICE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (packed)
        sgemm::fp32_probe_kernel<true><<<(unsigned)ctas, sgemm::kThreads, 0, s>>>(out, iterations);
    else
        sgemm::fp32_probe_kernel<false><<<(unsigned)ctas, sgemm::kThreads, 0, s>>>(out, iterations);
    if (cudaGetLastError() != cudaSuccess) return SGEMM_ELAUNCH;
    *flops_out = 2.0 * 2.0 * sgemm::kChains * (double)iterations * (double)ctas * sgemm::kThreads;
    return SGEMM_OK;
}

extern "C" int sgemm_probe_tf32_mma(int64_t iterations, float *out, double *flops_out,
                                    void *stream) {
    if (iterations <= 0 || iterations > (1 << 20)) return SGEMM_EINVAL_DIM;
    if (out == nullptr || flops_out == nullptr) return SGEMM_EINVAL_PTR;
    int dev = 0, sms = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        sms <= 0 || major * 10 + minor != 103)
        return SGEMM_EDEVICE;
    if (sgemm::launch_tf32_mma_probe(iterations, out, sms, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return SGEMM_ELAUNCH;
    *flops_out = sgemm::tf32_mma_probe_flops_per_iteration() * (double)iterations * (double)sms;
    return SGEMM_OK;
}

extern "C" int sgemm_selftest_wait_timeout(int64_t limit_cycles, void *stream) {
    if (limit_cycles < 1000 || limit_cycles > 4000000000LL) return SGEMM_EINVAL_DIM;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_EDEVICE;
    if (sgemm::launch_wait_timeout_selftest(limit_cycles, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return SGEMM_ELAUNCH;
    return SGEMM_OK;
}
