// SIMT FP32 SGEMM for small problems: 64 x 64 output tiles with K split over
// the CTAs of a thread-block cluster.
//
// A product whose 128 x 128 tiles cover at most a quarter of the SMs (256^3:
// four tiles) leaves most of the GPU idle, and the cluster split of the
// 128 x 128 kernel (simt_sgemm.cuh, CSPLIT) still puts a whole 128 x 128 x 32
// slice on each CTA's critical path: about 2 us of FMAs for one SM.  Here the
// tile is 64 x 64, so 256^3 becomes 16 tiles, and K is split over clusters of
// S CTAs (up to 16), each taking whole 32-deep slices: 128 CTAs of one slice
// each at 256^3.  This is the split-K of the ChetanC28/cuda-kernels page
// ("splitting the K dimension across blocks for small problems") with the
// reduction kept on chip, as in the 128 x 128 cluster split:
//   * 256 threads, each owning a 4 x 4 block of the tile (rows 4 ty .. 4 ty+3,
//     columns 4 tx .. 4 tx+3), accumulated with packed fp32 FMAs in ascending
//     k: each output's terms of a chunk are summed by one thread in order;
//   * both operand slices are stored K-major ([32][64] floats) with the same
//     float4-granular XOR swizzle and loaders as the 128 x 128 kernel
//     (TileLoader): 16-byte cp.async for M/N-contiguous operands, 128-bit
//     register-staged loads and a corner turn for K-contiguous ones; edges are
//     zero-filled;
//   * two stages, one CTA barrier per slice;
//   * CTA q of a cluster parks its 64 x 64 partial in its own shared memory;
//     after a cluster barrier it sums rows [64 q / S, 64 (q+1) / S) over ranks
//     0..S-1 in that order through distributed shared memory, applies the
//     epilogue and stores; a second cluster barrier keeps every CTA's shared
//     memory alive until its peers have read it.
// The chunk sums are added in chunk order: deterministic, and exact on small
// integers, like every SIMT path.
#pragma once

#include "simt_sgemm.cuh"

namespace sgemm {
namespace simt {

constexpr int kSmallTile = 64;
constexpr int kSmallBK = 32;
constexpr int kSmallPartialLd = kSmallTile + 4;   // partial-tile row stride (floats)

constexpr int small_smem_bytes() {
    constexpr int pipe = 2 * kSmallBK * 2 * kSmallTile * (int)sizeof(float);
    constexpr int part = kSmallTile * kSmallPartialLd * (int)sizeof(float);
    return pipe > part ? pipe : part;
}

// Launched in 1-D clusters of S CTAs; CTA q of a cluster covers k in
// [q * kchunk, min(K, (q + 1) * kchunk)) of tile blockIdx.x / S (tiles_m and
// tiles_n of `p` count 64 x 64 tiles).
template <bool TA, bool TB, bool VEC>
__global__ void __launch_bounds__(THREADS) sgemm_simt_small_kernel(const GemmArgs p) {
    constexpr int T = kSmallTile, BK = kSmallBK;
    constexpr int STILE = BK * T;   // floats of one operand slice
    __shared__ __align__(16) float smem[small_smem_bytes() / sizeof(float)];
    float *As = smem;               // [2][BK][T]
    float *Bs = smem + 2 * STILE;   // [2][BK][T]

    int z, tm, tn;
    raster(p, (int)(blockIdx.x / cluster_size()), z, tm, tn);
    const int m0 = tm * T, n0 = tn * T;
    const int kq = (int)cluster_rank();
    const int Kz = min(p.kchunk, p.K - kq * p.kchunk);   // <= 0: this rank has no chunk

    TileLoader<BK, T, !TA, VEC> la;
    la.base = p.A + (int64_t)z * p.strideA;
    la.ld = p.lda;
    la.mn0 = m0;
    la.mn_ext = p.M;
    la.K = Kz;
    TileLoader<BK, T, TB, VEC> lb;
    lb.base = p.B + (int64_t)z * p.strideB;
    lb.ld = p.ldb;
    lb.mn0 = n0;
    lb.mn_ext = p.N;
    lb.K = Kz;
    const int64_t kbeg = (int64_t)kq * p.kchunk;
    la.base += TA ? kbeg * p.lda : kbeg;
    lb.base += TB ? kbeg : kbeg * p.ldb;

    const int tid = threadIdx.x;
    const int ty = tid >> 4, tx = tid & 15;
    const int a_col = 4 * ty, b_col = 4 * tx;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    const int nk = Kz > 0 ? (Kz + BK - 1) / BK : 0;
    if (nk > 0) {
        la.fetch(0, As);
        lb.fetch(0, Bs);
        cp_async_commit();
        la.commit(As);
        lb.commit(Bs);
    }
    for (int t = 0; t < nk; ++t) {
        const int cur = t & 1, nxt = cur ^ 1;
        // slice t has landed (its copies and its corner-turned stores), and
        // every thread is done with slice t - 1, whose stage is refilled next
        cp_async_wait<0>();
        __syncthreads();
        if (t + 1 < nk) {
            la.fetch((t + 1) * BK, As + nxt * STILE);
            lb.fetch((t + 1) * BK, Bs + nxt * STILE);
            cp_async_commit();
        }
        const float *at = As + cur * STILE, *bt = Bs + cur * STILE;
#pragma unroll 8
        for (int kk = 0; kk < BK; ++kk) {
            const float4 a = *reinterpret_cast<const float4 *>(at + kk * T + (a_col ^ swz<BK>(kk)));
            const float4 b = *reinterpret_cast<const float4 *>(bt + kk * T + (b_col ^ swz<BK>(kk)));
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 ai = make_float2(av[i], av[i]);
                float2 c0 = make_float2(acc[i][0], acc[i][1]);
                float2 c1 = make_float2(acc[i][2], acc[i][3]);
                c0 = __ffma2_rn(ai, make_float2(b.x, b.y), c0);
                c1 = __ffma2_rn(ai, make_float2(b.z, b.w), c1);
                acc[i][0] = c0.x;
                acc[i][1] = c0.y;
                acc[i][2] = c1.x;
                acc[i][3] = c1.y;
            }
        }
        // the corner-turned operand of slice t + 1 (its loads overlapped the FMAs)
        if (t + 1 < nk) {
            la.commit(As + nxt * STILE);
            lb.commit(Bs + nxt * STILE);
        }
    }

    float *Cz = p.C + (int64_t)z * p.strideC;
    const bool plain = plain_epilogue(p);
    const uint32_t csize = cluster_size();
    if (csize == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = m0 + a_col + i;
            if (row < p.M)
                store_c4(p, Cz + (int64_t)row * p.ldc, n0 + b_col,
                         make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]), VEC, plain);
        }
        return;
    }
    // park the partial tile over the pipeline buffers once every thread is
    // done reading them
    __syncthreads();
    float *part = smem;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4 *>(part + (a_col + i) * kSmallPartialLd + b_col) =
            make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    cluster_sync();
    const int r0 = (int)((uint32_t)kq * T / csize), r1 = (int)(((uint32_t)kq + 1) * T / csize);
    constexpr int G = T / 4;   // float4 groups per row
    for (int g = tid; g < (r1 - r0) * G; g += THREADS) {
        const int r = r0 + g / G, c = 4 * (g % G);
        const uint32_t at = smem_u32(part + r * kSmallPartialLd + c);
        const float4 sum = cluster_sum_f4(at, csize);
        const int row = m0 + r;
        if (row < p.M) store_c4(p, Cz + (int64_t)row * p.ldc, n0 + c, sum, VEC, plain);
    }
    // no CTA may leave (releasing its shared memory) while a peer still reads it
    cluster_sync_relaxed();
}

}  // namespace simt
}  // namespace sgemm
