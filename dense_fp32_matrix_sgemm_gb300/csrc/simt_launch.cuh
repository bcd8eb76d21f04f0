// Launch helper for one (transA, transB) pair of the SIMT kernel family.
// Each pair is instantiated in its own translation unit so the variants
// compile in parallel.
#pragma once

#include <atomic>

#include "simt_sgemm.cuh"

namespace sgemm {
namespace simt {

// Tuned configuration for GB300: K slice, pipeline depth, packed FMA.
constexpr int kBK = 32;
constexpr int kStages = 3;
constexpr bool kFfma2 = true;
constexpr int kBN = 128;
constexpr int kMinBlocks = 1;   // one 96 KB CTA per SM, up to 255 registers per thread

template <bool TA, bool TB, bool VEC>
cudaError_t launch_variant(const GemmArgs &a, cudaStream_t s) {
    auto kern = sgemm_simt_kernel<kBK, kStages, kBN, TA, TB, VEC, kFfma2, kMinBlocks>;
    constexpr int smem = smem_bytes<kBK, kStages, kBN>();
    if (smem > 48 * 1024) {
        // The opt-in shared-memory limit is a per-device function attribute.
        static std::atomic<unsigned long long> configured{0};
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        const unsigned long long bit = 1ull << (dev & 63);
        if (!(configured.load() & bit)) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
            if (e != cudaSuccess) return e;
            configured.fetch_or(bit);
        }
    }
    GemmArgs g = a;
    g.tiles_m = (a.M + BM - 1) / BM;
    g.tiles_n = (a.N + kBN - 1) / kBN;
    const long long blocks = (long long)g.batch * g.tiles_m * g.tiles_n;
    kern<<<(unsigned)blocks, THREADS, smem, s>>>(g);
    return cudaGetLastError();
}

template <bool TA, bool TB>
cudaError_t launch_pair(const GemmArgs &a, bool vec, cudaStream_t s) {
    return vec ? launch_variant<TA, TB, true>(a, s) : launch_variant<TA, TB, false>(a, s);
}

}  // namespace simt
}  // namespace sgemm
