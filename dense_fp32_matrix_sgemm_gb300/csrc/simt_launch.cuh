// Launch helper for one (transA, transB) pair of the SIMT kernel family.
// Each pair is instantiated in its own translation unit so the variants
// compile in parallel.
#pragma once

#include <atomic>
#include <utility>

#include "simt_sgemm.cuh"
#include "simt_small.cuh"

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
// little.  Row-major A with B stored transposed (both corner-turned) takes the
// same configuration at every K: 3072^3 53.8 -> 55.9 TFLOP/s, 8192 x 8192 x
// 4096 56.8 -> 60.5 against one 3-stage CTA per SM.
constexpr int kShortK = 256;
// Cluster split-K: problems whose 128 x 128 tiles (all batches) cover at most
// half the SMs split K over the S CTAs of a cluster, S in {2, 4, 8, 16} (16
// with the non-portable cluster-size opt-in), each CTA taking whole 32-deep
// slices.
constexpr int kMaxClusterSplit = 16;

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

// Launches `kern` as a programmatic dependent of the previous work in the
// stream: its CTAs may be scheduled once every CTA of the previous launch has
// called pdl_trigger (or exited), and must call pdl_wait before touching
// memory that launch writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Sets the opt-in dynamic shared-memory size of `kern` once per context.
template <typename Kern>
cudaError_t ensure_smem_attribute(Kern kern, int smem, PerContext<bool> &configured) {
    if (smem <= 48 * 1024) return cudaSuccess;
    bool done = false;
    if (configured.get(current_context_id(), done)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured.put(current_context_id(), true);
    return cudaSuccess;
}

template <int STAGES, int BN_, bool TA, bool TB, bool VEC, int MINB = kMinBlocks>
cudaError_t launch_config(const GemmArgs &a, cudaStream_t s) {
    constexpr int commit = BN_ == 256 ? kCommitWide : (STAGES == 2 ? kBK : kCommitNarrow);
    auto kern = sgemm_simt_kernel<kBK, STAGES, BN_, TA, TB, VEC, kFfma2, MINB, commit>;
    constexpr int smem = smem_bytes<kBK, STAGES, BN_>();
    static PerContext<bool> configured;
    cudaError_t e = ensure_smem_attribute(kern, smem, configured);
    if (e != cudaSuccess) return e;
    GemmArgs g = a;
    g.tiles_m = (a.M + BM - 1) / BM;
    g.tiles_n = (a.N + BN_ - 1) / BN_;
    const long long blocks = (long long)g.batch * g.tiles_m * g.tiles_n;
    kern<<<(unsigned)blocks, THREADS, smem, s>>>(g);
    return cudaGetLastError();
}

// The cluster split for one (transA, transB, vec) variant.  Returns false
// (launching nothing) when the problem has enough tiles to fill the GPU, K is
// too short to split, or no cluster size lets every cluster be resident at
// once; else launches and stores the launch status in `err`.
template <bool TA, bool TB, bool VEC>
bool launch_cluster_split(const GemmArgs &a, cudaStream_t s, cudaError_t &err) {
    constexpr int kStages = kStagesNarrow;
    auto kern = sgemm_simt_kernel<kBK, kStages, 128, TA, TB, VEC, kFfma2, kMinBlocks, kCommitNarrow,
                                  true>;
    constexpr int smem = smem_bytes<kBK, kStages, 128, true>();
    const long long sms = sm_count();
    const long long tm = (a.M + BM - 1) / BM, tn = (a.N + 127) / 128;
    const long long tiles = (long long)a.batch * tm * tn;
    if (a.kchunk != 0 || tiles * 2 > sms) return false;
    const long long slices = (a.K + kBK - 1) / kBK;
    if (slices < 2) return false;

    static PerContext<bool> configured;
    err = ensure_smem_attribute(kern, smem, configured);
    if (err != cudaSuccess) return true;
    int dev = 0;
    err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return true;
    // clusters of 16 need the non-portable size opt-in (a function attribute,
    // set once per context)
    static PerContext<bool> nonportable;
    bool opted = false;
    if (!nonportable.get(current_context_id(), opted)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess)
            (void)cudaGetLastError();   // then clusters of 16 report no residency below
        nonportable.put(current_context_id(), true);
    }

    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;

    // Clusters of each size that fit on the device at once (0: not asked yet,
    // -1: that size cannot run); a split that needs a second wave loses.
    static std::atomic<int> resident[64][4];
    auto fits = [&](int c) {
        std::atomic<int> &slot = resident[dev & 63][c == 2 ? 0 : (c == 4 ? 1 : (c == 8 ? 2 : 3))];
        int n = slot.load();
        if (n == 0) {
            attr[0].val.clusterDim.x = (unsigned)c;
            cfg.gridDim = dim3((unsigned)c);
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
                (void)cudaGetLastError();   // the unsplit kernels still serve the call
                n = -1;
            }
            slot.store(n);
        }
        return n >= tiles;
    };
    // the fewest 32-deep slices per CTA; the smallest cluster among equals
    int S = 1;
    long long best = slices;
    for (int c = 2; c <= kMaxClusterSplit; c *= 2) {
        if (tiles * c > sms || c > slices) break;
        const long long per = (slices + c - 1) / c;
        if (per < best && fits(c)) {
            best = per;
            S = c;
        }
    }
    if (S < 2) return false;

    GemmArgs g = a;
    g.tiles_m = (int)tm;
    g.tiles_n = (int)tn;
    g.kchunk = (int)(best * kBK);
    attr[0].val.clusterDim.x = (unsigned)S;
    cfg.gridDim = dim3((unsigned)(tiles * S));
    err = cudaLaunchKernelEx(&cfg, kern, g);
    return true;
}

// 32-deep K slices per CTA when `tiles` tiles split K over clusters of the
// largest power of two up to 16 with tiles * S <= sms (residency not checked):
// the work on each CTA's critical path.
inline long long split_slices_per_cta(long long tiles, long long slices, long long sms) {
    long long best = slices;
    for (long long c = 2; c <= kMaxClusterSplit; c *= 2) {
        if (tiles * c > sms || c > slices) break;
        best = (slices + c - 1) / c;
    }
    return best;
}

// A 64 x 64 slice (4 x 4 outputs per thread, two 16-byte shared loads per 8
// packed FMAs) costs about 0.65 of a 128 x 128 one on its CTA's critical path
// (measured: 128 x 128 x 32768 on 64 CTAs of 64 x 64 against 16 of 128 x 128,
// 64 slices each, 114 against 180 us).  So the small tiles pay where they cut
// the slices per CTA: 256^3 (1 slice each way, 8.2 -> 6.6 us), 384^3 (2 -> 3,
// 11.1 -> 8.6 us), but not 512^3 (2 -> 8, 16.2 against 17.0 us) or
// 256 x 256 x 4096 (8 -> 16, 28.6 against 43.6 us).
constexpr double kSmallSliceCost = 0.65;

// The 64 x 64 cluster split (simt_small.cuh) for problems whose 64 x 64
// tiles cover at most half the SMs (256^3: 16 tiles) and whose slices per CTA
// it cuts enough against the 128 x 128 split (kSmallSliceCost).  S CTAs per
// cluster, S in {1, 2, 4, 8, 16}: the fewest 32-deep slices per CTA subject to
// tiles * S <= SMs and every cluster being resident at once.  Returns false
// (launching nothing) when the problem is not such a case; else launches and
// stores the launch status in `err`.
template <bool TA, bool TB, bool VEC>
bool launch_small_split(const GemmArgs &a, cudaStream_t s, cudaError_t &err) {
    auto kern = sgemm_simt_small_kernel<TA, TB, VEC>;
    const long long sms = sm_count();
    const long long tm = (a.M + kSmallTile - 1) / kSmallTile;
    const long long tn = (a.N + kSmallTile - 1) / kSmallTile;
    const long long tiles = (long long)a.batch * tm * tn;
    if (a.kchunk != 0 || tiles * 2 > sms) return false;
    const long long slices = (a.K + kSmallBK - 1) / kSmallBK;
    {
        const long long big_tiles = (long long)a.batch * ((a.M + BM - 1) / BM) * ((a.N + 127) / 128);
        const double small = kSmallSliceCost * (double)split_slices_per_cta(tiles, slices, sms);
        const double big = (double)split_slices_per_cta(big_tiles, (a.K + kBK - 1) / kBK, sms);
        if (!(small < big)) return false;
    }

    int dev = 0;
    err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return true;
    static PerContext<bool> nonportable;
    bool opted = false;
    if (!nonportable.get(current_context_id(), opted)) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess)
            (void)cudaGetLastError();   // then clusters of 16 report no residency below
        nonportable.put(current_context_id(), true);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static std::atomic<int> resident[64][4];
    auto fits = [&](int c) {
        std::atomic<int> &slot = resident[dev & 63][c == 2 ? 0 : (c == 4 ? 1 : (c == 8 ? 2 : 3))];
        int n = slot.load();
        if (n == 0) {
            attr[0].val.clusterDim.x = (unsigned)c;
            cfg.gridDim = dim3((unsigned)c);
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
                (void)cudaGetLastError();
                n = -1;
            }
            slot.store(n);
        }
        return n >= tiles;
    };
    int S = 1;
    long long best = slices;
    for (int c = 2; c <= kMaxClusterSplit; c *= 2) {
        if (tiles * c > sms || c > slices) break;
        const long long per = (slices + c - 1) / c;
        if (per < best && fits(c)) {
            best = per;
            S = c;
        }
    }
    GemmArgs g = a;
    g.tiles_m = (int)tm;
    g.tiles_n = (int)tn;
    g.kchunk = (int)(best * kSmallBK);
    attr[0].val.clusterDim.x = (unsigned)S;
    cfg.gridDim = dim3((unsigned)(tiles * S));
    err = cudaLaunchKernelEx(&cfg, kern, g);
    return true;
}

// The wide tile is used only where B arrives by cp.async (row-major B) and
// with 16-byte access: corner-turning a 256-wide B slice needs 32 more
// staging registers than the 255-register budget leaves.
template <bool TA, bool TB, bool VEC>
cudaError_t launch_variant(const GemmArgs &a, cudaStream_t s) {
    cudaError_t err = cudaSuccess;
    if (launch_small_split<TA, TB, VEC>(a, s, err)) return err;
    if (launch_cluster_split<TA, TB, VEC>(a, s, err)) return err;
    // 16-byte access: the TMA-fed kernel (two CTAs per SM), unless the
    // operands cannot be described as tensor maps
    if constexpr (VEC) {
        if (simt_tma_eligible(a, TA, TB, VEC) && launch_simt_tma(a, TA, TB, s, err)) return err;
    }
    if constexpr (VEC) {
        if (a.K <= kShortK || (TB && !TA)) return launch_config<2, 128, TA, TB, VEC, 2>(a, s);
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

// Stream-K launch: the tile kernel on one CTA per SM, then the fix-up pass.
template <int STAGES, int BN_, bool TA, bool TB, bool VEC, int CK>
cudaError_t launch_streamk_config(const GemmArgs &a, const StreamKPlan &pl, void *ws,
                                  cudaStream_t s) {
    auto kern = sgemm_simt_streamk_kernel<kBK, STAGES, BN_, TA, TB, VEC, kFfma2, kMinBlocks, CK>;
    constexpr int smem = smem_bytes<kBK, STAGES, BN_>();
    static PerContext<bool> configured;
    cudaError_t e = ensure_smem_attribute(kern, smem, configured);
    if (e != cudaSuccess) return e;
    GemmArgs g = a;
    g.tiles_m = (a.M + BM - 1) / BM;
    g.tiles_n = (a.N + BN_ - 1) / BN_;
    StreamK sk;
    sk.tiles_dp = pl.tiles_dp;
    sk.tiles_sk = pl.tiles_sk;
    sk.kslices = pl.kslices;
    sk.G = pl.G;
    sk.units = pl.units;
    sk.ws = static_cast<float *>(ws);
    kern<<<(unsigned)pl.G, THREADS, smem, s>>>(g, sk);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_pdl(streamk_fixup_kernel<BN_, VEC>, streamk_fixup_grid<BN_>(pl.tiles_sk),
                      dim3(256), 0, s, g, sk);
}

template <bool TA, bool TB, bool VEC>
cudaError_t launch_streamk_variant(const GemmArgs &a, const StreamKPlan &pl, void *ws,
                                   cudaStream_t s) {
    if constexpr (VEC && !TB) {
        if (pl.wide) return launch_streamk_config<kStagesWide, 256, TA, TB, VEC, kCommitWide>(a, pl, ws, s);
    }
    return launch_streamk_config<kStagesNarrow, 128, TA, TB, VEC, kCommitNarrow>(a, pl, ws, s);
}

template <bool TA, bool TB>
cudaError_t launch_streamk_pair(const GemmArgs &a, bool vec, const StreamKPlan &pl, void *ws,
                                cudaStream_t s) {
    return vec ? launch_streamk_variant<TA, TB, true>(a, pl, ws, s)
               : launch_streamk_variant<TA, TB, false>(a, pl, ws, s);
}

}  // namespace simt
}  // namespace sgemm
