// Launch helper for one (transA, transB) pair of the SIMT kernel family.
// Each pair is instantiated in its own translation unit so the variants
// compile in parallel.
#pragma once

#include <atomic>

#include "simt_sgemm.cuh"

namespace sgemm {
namespace simt {

// Two tuned configurations for GB300, both one 96 KB CTA of 256 threads per
// SM with packed FMA: 128 x 128 tiles (K slice 32, 3 stages) and 128 x 256
// tiles (K slice 32, 2 stages).  The wider tile does 1.95x the work of the
// narrow one in a little less than 1.95x its time, but comes in half as
// many pieces, so which one finishes first depends on how the tiles fall
// into waves of one CTA per SM (see pick_wide_tile).
constexpr int kBK = 32;
constexpr bool kFfma2 = true;
constexpr int kMinBlocks = 1;
constexpr int kStagesNarrow = 3;
constexpr int kStagesWide = 2;
constexpr double kWideTileCost = 1.95;   // time of a 128x256 tile / a 128x128 tile
// k step at which corner-turned slices are written to shared memory: spreading
// the stores away from the tile's closing barrier gains about 1 %.
constexpr int kCommitNarrow = 16;
constexpr int kCommitWide = 8;
// Short reductions (K <= kShortK, at most 8 K slices per tile): two CTAs per
// SM (128 registers, 2 stages) so one CTA's fill and stores overlap the other's
// FMAs; 32 % faster on 96 x 512 x 512 x 64 although the register cap spills a
// little.
constexpr int kShortK = 256;

inline int sm_count() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
    const int d = dev & 63;
    int v = cached[d].load();
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 1;
        cached[d].store(v);
    }
    return v;
}

// Estimated time in units of one 128x128 tile: full waves times tile cost.
inline bool pick_wide_tile(const GemmArgs &a) {
    const long long sms = sm_count();
    const long long tm = (a.M + BM - 1) / BM;
    const long long narrow = (long long)a.batch * tm * ((a.N + 127) / 128);
    const long long wide = (long long)a.batch * tm * ((a.N + 255) / 256);
    const double cost_narrow = (double)((narrow + sms - 1) / sms);
    const double cost_wide = kWideTileCost * (double)((wide + sms - 1) / sms);
    return cost_wide < cost_narrow;
}

template <int STAGES, int BN_, bool TA, bool TB, bool VEC, int MINB = kMinBlocks>
cudaError_t launch_config(const GemmArgs &a, cudaStream_t s) {
    constexpr int commit = BN_ == 256 ? kCommitWide : (STAGES == 2 ? kBK : kCommitNarrow);
    auto kern = sgemm_simt_kernel<kBK, STAGES, BN_, TA, TB, VEC, kFfma2, MINB, commit>;
    constexpr int smem = smem_bytes<kBK, STAGES, BN_>();
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
    g.tiles_n = (a.N + BN_ - 1) / BN_;
    const long long blocks = (long long)g.batch * g.tiles_m * g.tiles_n;
    kern<<<(unsigned)blocks, THREADS, smem, s>>>(g);
    return cudaGetLastError();
}

// The wide tile is used only where B arrives by cp.async (row-major B) and
// with 16-byte access: corner-turning a 256-wide B slice needs 32 more
// staging registers than the 255-register budget leaves.
template <bool TA, bool TB, bool VEC>
cudaError_t launch_variant(const GemmArgs &a, cudaStream_t s) {
    if constexpr (VEC) {
        if (a.K <= kShortK) return launch_config<2, 128, TA, TB, VEC, 2>(a, s);
    }
    if constexpr (VEC && !TB) {
        if (pick_wide_tile(a)) return launch_config<kStagesWide, 256, TA, TB, VEC>(a, s);
    }
    return launch_config<kStagesNarrow, 128, TA, TB, VEC>(a, s);
}

template <bool TA, bool TB>
cudaError_t launch_pair(const GemmArgs &a, bool vec, cudaStream_t s) {
    return vec ? launch_variant<TA, TB, true>(a, s) : launch_variant<TA, TB, false>(a, s);
}

}  // namespace simt
}  // namespace sgemm
