// SIMT FP32 SGEMM for sm_103a: C = op(A) op(B) on the CUDA cores.
//
// Design, after "CUDA GEMM operator performance optimization" (sections 4-10)
// and re-tuned for Blackwell:
//   * block tile 128 x BN (BN = 128 or 256), K sliced in steps of BK (section 4);
//   * 256 threads, each owning an 8 x 8 register tile split into four 4 x 4
//     sub-blocks 64 rows/columns apart (section 8.5, option 3), so every
//     fragment read is one 16-byte shared-memory load;
//   * warps of 4 x 8 threads laid out in Z order (section 8.5, option 4) so a
//     quarter-warp touches two A and four B float4s: broadcast, no conflicts;
//   * both operand tiles are stored K-major in shared memory ([BK][128],
//     "A transposed", section 7.3).  Operands that are contiguous along M/N
//     (A^T storage, row-major B) are copied with 16-byte cp.async; operands
//     contiguous along K (row-major A, B^T storage) are corner-turned: 128-bit
//     global loads into registers, then four scalar stores (section 7.3; the
//     corner turning of the PMPP tiled kernel);
//   * float4 groups of tile row kk are XOR-swizzled by a function of kk>>2
//     (section 8.5, option 2, at float4 granularity) which makes the
//     corner-turn stores conflict-free while reads stay 16-byte aligned;
//   * STAGES-deep pipeline: cp.async groups for the asynchronous operand, the
//     register-staged operand loaded one tile ahead, one barrier per K tile
//     (sections 9-10);
//   * packed two-wide FP32 FMA (fma.rn.f32x2, sm_100+) halves the issue slots
//     of the outer product, leaving room for the shared-memory loads;
//   * tiles are rasterised in groups of `group_m` tile rows so that a wave of
//     CTAs shares A and B panels in L2 (section 2.3);
//   * edge tiles are zero-padded on load and stores are guarded (DD2360
//     workbook, section 14.3);
//   * problems with too few tiles to fill the GPU split K across the CTAs of
//     a thread-block cluster (CSPLIT): each CTA accumulates one K chunk of the
//     same tile, parks its partial tile in its own shared memory, and after a
//     cluster barrier every CTA sums a band of rows over all the cluster's
//     partials, read through distributed shared memory in rank order.  This
//     is the split-K of the ChetanC28/cuda-kernels page (splitting K across
//     blocks for small problems) with the reduction kept on chip.
// Each output's K terms are accumulated by one thread, in ascending k, with
// fp32 FMAs (under CSPLIT: per chunk, and the chunk sums are then added in
// chunk order): the result is deterministic.
#pragma once

#include "device_utils.cuh"
#include "gemm_args.h"

namespace sgemm {
namespace simt {

constexpr int BM = 128;
constexpr int THREADS = 256;

// Element offset of float4 group 0 of tile row kk after swizzling: the group
// index is XORed with a multiple of (128/BK)/4 chosen so that the rows a warp
// writes during a corner turn land in 32 distinct banks.  Always a multiple of
// 4 and below 32, so a float4 stays whole and within its 32-float segment.
template <int BK>
__device__ __forceinline__ int swz(int kk) {
    return (128 / BK) * (kk >> 2);
}

// Loads one BK x ROWS slice of an operand into a K-major shared tile
// ([BK][ROWS] floats).  Element (mn, k) of the operand lives at
// base[mn*ld + k] when KCONTIG, else at base[k*ld + mn].  Out-of-range
// elements are stored as zero.
template <int BK, int ROWS, bool KCONTIG, bool VEC>
struct TileLoader {
    static constexpr int ELEMS = BK * ROWS / THREADS;  // per thread per slice
    static constexpr int VECS = ELEMS / 4;
    static constexpr int KQ = BK / 4;                  // float4 groups along k per row
    static constexpr int GROUPS = ROWS / 4;            // float4 groups along mn per k row

    const float *base;
    int64_t ld;
    int mn0, mn_ext, K;
    float4 rv[(KCONTIG && VEC) ? VECS : 1];
    float rs[(KCONTIG && !VEC) ? ELEMS : 1];

    // Start moving slice k0.  Asynchronous operands go straight to `tile`
    // (cp.async, committed by the caller); staged operands land in registers.
    __device__ __forceinline__ void fetch(int k0, float *tile) {
        const int tid = threadIdx.x;
        if constexpr (!KCONTIG && VEC) {
#pragma unroll
            for (int r = 0; r < VECS; ++r) {
                const int g = tid + r * THREADS;
                const int kk = g / GROUPS, mq = g % GROUPS;
                const int mn = mn0 + 4 * mq, k = k0 + kk;
                int nv = mn_ext - mn;
                nv = nv < 0 ? 0 : (nv > 4 ? 4 : nv);
                if (k >= K) nv = 0;
                const float *src = nv ? base + (int64_t)k * ld + mn : base;
                cp_async_16(smem_u32(tile + kk * ROWS + ((4 * mq) ^ swz<BK>(kk))), src, nv * 4);
            }
        } else if constexpr (!KCONTIG && !VEC) {
#pragma unroll
            for (int r = 0; r < ELEMS; ++r) {
                const int e = tid + r * THREADS;
                const int kk = e / ROWS, mm = e % ROWS;
                const int mn = mn0 + mm, k = k0 + kk;
                const bool ok = (mn < mn_ext) && (k < K);
                const float *src = ok ? base + (int64_t)k * ld + mn : base;
                cp_async_4(smem_u32(tile + kk * ROWS + (mm ^ swz<BK>(kk))), src, ok ? 4 : 0);
            }
        } else if constexpr (KCONTIG && VEC) {
#pragma unroll
            for (int r = 0; r < VECS; ++r) {
                const int g = tid + r * THREADS;
                const int row = g / KQ, kq = g % KQ;
                const int mn = mn0 + row, k = k0 + 4 * kq;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (mn < mn_ext) {
                    const float *p = base + (int64_t)mn * ld + k;
                    if (k + 3 < K) {
                        v = ldg_f4(p);
                    } else {
                        if (k + 0 < K) v.x = __ldg(p + 0);
                        if (k + 1 < K) v.y = __ldg(p + 1);
                        if (k + 2 < K) v.z = __ldg(p + 2);
                    }
                }
                rv[r] = v;
            }
        } else {
#pragma unroll
            for (int r = 0; r < ELEMS; ++r) {
                const int e = tid + r * THREADS;
                const int row = e / BK, kk = e % BK;
                const int mn = mn0 + row, k = k0 + kk;
                rs[r] = (mn < mn_ext && k < K) ? __ldg(base + (int64_t)mn * ld + k) : 0.f;
            }
        }
    }

    // Write a staged slice (corner turn) into `tile`; no-op for cp.async operands.
    __device__ __forceinline__ void commit(float *tile) {
        const int tid = threadIdx.x;
        if constexpr (KCONTIG && VEC) {
#pragma unroll
            for (int r = 0; r < VECS; ++r) {
                const int g = tid + r * THREADS;
                const int row = g / KQ, kq = g % KQ;
                const int kk = 4 * kq;
                const int col = row ^ swz<BK>(kk);   // same swizzle for kk..kk+3
                tile[(kk + 0) * ROWS + col] = rv[r].x;
                tile[(kk + 1) * ROWS + col] = rv[r].y;
                tile[(kk + 2) * ROWS + col] = rv[r].z;
                tile[(kk + 3) * ROWS + col] = rv[r].w;
            }
        } else if constexpr (KCONTIG && !VEC) {
#pragma unroll
            for (int r = 0; r < ELEMS; ++r) {
                const int e = tid + r * THREADS;
                const int row = e / BK, kk = e % BK;
                tile[kk * ROWS + (row ^ swz<BK>(kk))] = rs[r];
            }
        }
    }
};

// Row stride (floats) of the partial tile a CSPLIT CTA parks in shared
// memory: 4 floats of padding put the two rows a quarter-warp writes in
// different banks.
constexpr int kPartialLd = 128 + 4;

template <int BK, int STAGES, int BN_, bool CSPLIT = false>
constexpr int smem_bytes() {
    constexpr int pipe = STAGES * BK * (BM + BN_) * (int)sizeof(float);
    constexpr int part = CSPLIT ? BM * kPartialLd * (int)sizeof(float) : 0;
    return pipe > part ? pipe : part;
}

// Maps a linear tile index to (batch, tile row, tile column), walking
// `group_m` tile rows down a column before moving right.
__device__ __forceinline__ void raster(const GemmArgs &p, int bid, int &z, int &tm, int &tn) {
    const int per_batch = p.tiles_m * p.tiles_n;
    z = bid / per_batch;
    const int t = bid - z * per_batch;
    const int group = p.group_m * p.tiles_n;
    const int g = t / group;
    const int first = g * p.group_m;
    const int rows = min(p.tiles_m - first, p.group_m);
    const int r = t - g * group;
    tm = first + r % rows;
    tn = r / rows;
}

// Stores four consecutive outputs of a row, applying the epilogue
// C = alpha * acc + beta * C + bias[col] unless it is the plain one.  Columns
// at or past N are neither read nor written; 16-byte accesses when `vec`
// allows and the four columns are all in range.
__device__ __forceinline__ void store_c4(const GemmArgs &p, float *crow, int col, float4 v,
                                         bool vec, bool plain) {
    const bool full = vec && col + 3 < p.N;
    if (!plain) {
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p.beta != 0.f) {
            if (full) {
                o = *reinterpret_cast<const float4 *>(crow + col);
            } else {
                if (col + 0 < p.N) o.x = crow[col + 0];
                if (col + 1 < p.N) o.y = crow[col + 1];
                if (col + 2 < p.N) o.z = crow[col + 2];
                if (col + 3 < p.N) o.w = crow[col + 3];
            }
        }
        float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p.bias != nullptr) {
            if (col + 0 < p.N) b.x = p.bias[col + 0];
            if (col + 1 < p.N) b.y = p.bias[col + 1];
            if (col + 2 < p.N) b.z = p.bias[col + 2];
            if (col + 3 < p.N) b.w = p.bias[col + 3];
        }
        v.x = fmaf(p.beta, o.x, p.alpha * v.x) + b.x;
        v.y = fmaf(p.beta, o.y, p.alpha * v.y) + b.y;
        v.z = fmaf(p.beta, o.z, p.alpha * v.z) + b.z;
        v.w = fmaf(p.beta, o.w, p.alpha * v.w) + b.w;
    }
    if (full) {
        *reinterpret_cast<float4 *>(crow + col) = v;
    } else {
        if (col + 0 < p.N) crow[col + 0] = v.x;
        if (col + 1 < p.N) crow[col + 1] = v.y;
        if (col + 2 < p.N) crow[col + 2] = v.z;
        if (col + 3 < p.N) crow[col + 3] = v.w;
    }
}

// The K-slice pipeline of one tile: zeroes acc, then accumulates the
// loaders' K range (ktiles slices of BK; <= 0 loads nothing) into the
// thread's 8 x (BN_/16) register tile.  Ends with no copy in flight.
template <int BK, int STAGES, int BN_, bool TA, bool TB, bool VEC, bool FFMA2, int CK>
__device__ __forceinline__ void tile_mainloop(TileLoader<BK, BM, !TA, VEC> &la,
                                              TileLoader<BK, BN_, TB, VEC> &lb, float *As,
                                              float *Bs, int ktiles, int a_col, int b_col,
                                              float (&acc)[8][BN_ / 16]) {
    constexpr int TN = BN_ / 16;
    constexpr int NSB = BN_ / 64;
    constexpr int ATILE = BK * BM;
    constexpr int BTILE = BK * BN_;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < ktiles) {
            la.fetch(s * BK, As + s * ATILE);
            lb.fetch(s * BK, Bs + s * BTILE);
            la.commit(As + s * ATILE);
            lb.commit(Bs + s * BTILE);
        }
        cp_async_commit();
    }

    int rstage = 0;            // stage holding tile kt
    int wstage = STAGES - 1;   // stage receiving tile kt + STAGES - 1
    for (int kt = 0; kt < ktiles; ++kt) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();

        const int nt = kt + STAGES - 1;
        if (nt < ktiles) {
            la.fetch(nt * BK, As + wstage * ATILE);
            lb.fetch(nt * BK, Bs + wstage * BTILE);
        }
        cp_async_commit();

        const float *at = As + rstage * ATILE;
        const float *bt = Bs + rstage * BTILE;
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            const int sw = swz<BK>(kk);
            const float *br = bt + kk * BN_;
            if constexpr (CK < BK) {
                if (kk == CK && nt < ktiles) {
                    la.commit(As + wstage * ATILE);
                    lb.commit(Bs + wstage * BTILE);
                }
            }
            const float *ar = at + kk * BM;
            const float4 a0 = *reinterpret_cast<const float4 *>(ar + (a_col ^ sw));
            const float4 a1 = *reinterpret_cast<const float4 *>(ar + 64 + (a_col ^ sw));
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            float b[TN];
#pragma unroll
            for (int h = 0; h < NSB; ++h) {
                const float4 bv = *reinterpret_cast<const float4 *>(br + 64 * h + (b_col ^ sw));
                b[4 * h + 0] = bv.x;
                b[4 * h + 1] = bv.y;
                b[4 * h + 2] = bv.z;
                b[4 * h + 3] = bv.w;
            }
            if constexpr (FFMA2) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 ai = make_float2(a[i], a[i]);
#pragma unroll
                    for (int j = 0; j < TN; j += 2) {
                        float2 c = make_float2(acc[i][j], acc[i][j + 1]);
                        c = __ffma2_rn(ai, make_float2(b[j], b[j + 1]), c);
                        acc[i][j] = c.x;
                        acc[i][j + 1] = c.y;
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
        }

        if (CK >= BK && nt < ktiles) {
            la.commit(As + wstage * ATILE);
            lb.commit(Bs + wstage * BTILE);
        }
        rstage = (rstage + 1 == STAGES) ? 0 : rstage + 1;
        wstage = (wstage + 1 == STAGES) ? 0 : wstage + 1;
    }
    cp_async_wait<0>();
}

// Block tile 128 x BN_ (BN_ = 128 or 256); each thread owns an 8 x (BN_/16)
// register tile made of 4 x 4 sub-blocks spaced 64 rows / 64 columns apart.
// CK: the k step of the tile loop at which register-staged (corner-turned)
// slices are written to shared memory; BK means after the last step.
// CSPLIT: launched in 1-D clusters of S CTAs (S divides 128); CTA q of the
// cluster covers k in [q*kchunk, min(K, (q+1)*kchunk)) of tile blockIdx.x / S.
template <int BK, int STAGES, int BN_, bool TA, bool TB, bool VEC, bool FFMA2, int MINB,
          int CK = BK, bool CSPLIT = false>
__global__ void __launch_bounds__(THREADS, MINB) sgemm_simt_kernel(const GemmArgs p) {
    static_assert(CK >= 0 && CK <= BK, "commit step out of range");
    static_assert(!CSPLIT || BN_ == 128, "the cluster split uses 128 x 128 tiles");
    static_assert(BK == 8 || BK == 16 || BK == 32, "BK must be 8, 16 or 32");
    static_assert(BN_ == 128 || BN_ == 256, "BN must be 128 or 256");
    static_assert(STAGES >= 2, "need at least two stages");
    constexpr int TN = BN_ / 16;         // columns per thread
    constexpr int NSB = BN_ / 64;        // 4-wide column sub-blocks per thread
    constexpr int ATILE = BK * BM;
    extern __shared__ __align__(16) float smem[];
    float *As = smem;
    float *Bs = smem + STAGES * ATILE;

    int z, tm, tn;
    raster(p, CSPLIT ? (int)(blockIdx.x / cluster_size()) : (int)blockIdx.x, z, tm, tn);
    const int m0 = tm * BM, n0 = tn * BN_;
    // split-K: the K-chunk [kq*kchunk, min(K, (kq+1)*kchunk)), where kq is the
    // problem index z (partial planes; the strides step by one chunk) or,
    // under CSPLIT, the rank in the cluster.  Ranks past the last chunk get
    // Kz <= 0 and load nothing.
    const int kq = CSPLIT ? (int)cluster_rank() : z;
    const int Kz = (CSPLIT || p.kchunk > 0) ? min(p.kchunk, p.K - kq * p.kchunk) : p.K;

    // A is contiguous along K unless stored transposed; B the other way round.
    TileLoader<BK, BM, !TA, VEC> la;
    la.base = p.A + (int64_t)z * p.strideA;
    la.ld = p.lda;
    la.mn0 = m0;
    la.mn_ext = p.M;
    la.K = Kz;
    TileLoader<BK, BN_, TB, VEC> lb;
    lb.base = p.B + (int64_t)z * p.strideB;
    lb.ld = p.ldb;
    lb.mn0 = n0;
    lb.mn_ext = p.N;
    lb.K = Kz;
    if constexpr (CSPLIT) {
        const int64_t kbeg = (int64_t)kq * p.kchunk;
        la.base += TA ? kbeg * p.lda : kbeg;
        lb.base += TB ? kbeg : kbeg * p.ldb;
    }

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int lane_row = (lane & 1) | ((lane >> 4) << 1);   // Z-order 4 x 8
    const int lane_col = (lane >> 1) & 7;
    const int ty = (warp >> 1) * 4 + lane_row;               // 0..15
    const int tx = (warp & 1) * 8 + lane_col;                // 0..15
    const int a_col = 4 * ty;
    const int b_col = 4 * tx;

    float acc[8][TN];
    tile_mainloop<BK, STAGES, BN_, TA, TB, VEC, FFMA2, CK>(la, lb, As, Bs, (Kz + BK - 1) / BK, a_col,
                                                         b_col, acc);

    float *Cz = p.C + (int64_t)z * p.strideC;
    const bool plain = plain_epilogue(p);
    if constexpr (CSPLIT) {
        // Park the partial tile (row-major, kPartialLd floats per row) over the
        // pipeline buffers once every warp is done reading them.
        __syncthreads();
        float *part = smem;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = i < 4 ? a_col + i : 64 + a_col + (i - 4);
#pragma unroll
            for (int h = 0; h < NSB; ++h)
                *reinterpret_cast<float4 *>(part + r * kPartialLd + h * 64 + b_col) =
                    make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2],
                                acc[i][4 * h + 3]);
        }
        cluster_sync();
        // CTA q finishes rows [q*128/S, (q+1)*128/S) of the tile: the sum over
        // ranks 0..S-1 of the partials, in that order, then the epilogue.
        const uint32_t crank = (uint32_t)kq, csize = cluster_size();
        const int r0 = (int)(crank * BM / csize), r1 = (int)((crank + 1) * BM / csize);
        constexpr int G = BN_ / 4;   // float4 groups per row
        for (int g = tid; g < (r1 - r0) * G; g += THREADS) {
            const int r = r0 + g / G, c = 4 * (g % G);
            const uint32_t at = smem_u32(part + r * kPartialLd + c);
            const float4 sum = cluster_sum_f4(at, csize);
            const int row = m0 + r;
            if (row < p.M) store_c4(p, Cz + (int64_t)row * p.ldc, n0 + c, sum, VEC, plain);
        }
        // No CTA may leave (releasing its shared memory) while a peer still reads it.
        cluster_sync_relaxed();
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int row = m0 + (i < 4 ? a_col + i : 64 + a_col + (i - 4));
            if (row >= p.M) continue;
            float *crow = Cz + (int64_t)row * p.ldc;
#pragma unroll
            for (int h = 0; h < NSB; ++h) {
                const int col = n0 + h * 64 + b_col;
                const float4 v = make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2],
                                             acc[i][4 * h + 3]);
                store_c4(p, crow, col, v, VEC, plain);
            }
        }
    }
}

// ------------------------------------------------------------------ stream-K

// Stream-K schedule of the tile kernel over G CTAs (one per SM), for problems
// whose tiles fill the SMs a non-whole number of times (3072^3: 288 tiles of
// 128 x 256 on 152 SMs, so a second wave of 136).  The first tiles_dp tiles
// (whole waves) are computed whole, tile c + i*G on CTA c.  The K slices of
// the remaining tiles_sk tiles are dealt out evenly: CTA c takes units
// [c*U/G, (c+1)*U/G) of U = tiles_sk * kslices, in tile order, slices
// ascending.  A tile whose slices all fall to one CTA is stored to C.  A tile
// shared between CTAs is a piece of each: the CTA's first piece goes to
// workspace slot [c][0], its last to [c][1], and streamk_fixup_kernel adds a
// tile's pieces in K order.  No CTA waits for another.
struct StreamK {
    int tiles_dp, tiles_sk, kslices, G;
    int64_t units;
    float *ws;   // [G][2][BM * BN] partial tiles, row-major
};

// Units [0, u) of CTA c start at floor(c*U/G); the CTA owning unit u.
__host__ __device__ inline int streamk_owner(int64_t u, int64_t U, int G) {
    return (int)(((u + 1) * G - 1) / U);
}

template <int BK, int STAGES, int BN_, bool TA, bool TB, bool VEC, bool FFMA2, int MINB, int CK>
__global__ void __launch_bounds__(THREADS, MINB)
sgemm_simt_streamk_kernel(const GemmArgs p, const StreamK sk) {
    constexpr int TN = BN_ / 16;
    constexpr int NSB = BN_ / 64;
    constexpr int ATILE = BK * BM;
    extern __shared__ __align__(16) float smem[];
    float *As = smem;
    float *Bs = smem + STAGES * ATILE;

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int lane_row = (lane & 1) | ((lane >> 4) << 1);   // Z-order 4 x 8
    const int lane_col = (lane >> 1) & 7;
    const int a_col = 4 * ((warp >> 1) * 4 + lane_row);
    const int b_col = 4 * ((warp & 1) * 8 + lane_col);

    // Everything about piece i is recomputed from (blockIdx.x, i): no schedule
    // state lives across the main loop.  tiles_sk < G, so a CTA's stream-K
    // range is at most kslices units long: at most two pieces.
    const int c = blockIdx.x;
    const int ndp = c < sk.tiles_dp ? (sk.tiles_dp - 1 - c) / sk.G + 1 : 0;
    int nsk;
    {
        const int64_t u0 = (int64_t)c * sk.units / sk.G, u1 = ((int64_t)c + 1) * sk.units / sk.G;
        nsk = u0 == u1 ? 0 : (u0 / sk.kslices == (u1 - 1) / sk.kslices ? 1 : 2);
    }
#pragma unroll 1
    for (int i = 0; i < ndp + nsk; ++i) {
        int t, s0, s1;
        float *part = nullptr;   // null: store the finished tile to C
        if (i < ndp) {
            t = c + i * sk.G;
            s0 = 0;
            s1 = sk.kslices;
        } else {
            const int k = i - ndp;   // 0: the range's first piece, 1: its last
            const int64_t u0 = (int64_t)c * sk.units / sk.G;
            const int64_t u1 = ((int64_t)c + 1) * sk.units / sk.G;
            const int64_t ub = k == 0 ? u0 : (u0 / sk.kslices + 1) * sk.kslices;
            const int tl = (int)(ub / sk.kslices);
            s0 = (int)(ub - (int64_t)tl * sk.kslices);
            s1 = (int)min((int64_t)sk.kslices, s0 + (u1 - ub));
            t = sk.tiles_dp + tl;
            if (!(s0 == 0 && s1 == sk.kslices))
                part = sk.ws + ((int64_t)c * 2 + k) * (BM * BN_);
        }
        int z, tm, tn;
        raster(p, t, z, tm, tn);
        const int m0 = tm * BM, n0 = tn * BN_;
        const int64_t kbeg = (int64_t)s0 * BK;
        const int Kz = min(p.K, s1 * BK) - s0 * BK;
        TileLoader<BK, BM, !TA, VEC> la;
        la.base = p.A + (int64_t)z * p.strideA + (TA ? kbeg * p.lda : kbeg);
        la.ld = p.lda;
        la.mn0 = m0;
        la.mn_ext = p.M;
        la.K = Kz;
        TileLoader<BK, BN_, TB, VEC> lb;
        lb.base = p.B + (int64_t)z * p.strideB + (TB ? kbeg : kbeg * p.ldb);
        lb.ld = p.ldb;
        lb.mn0 = n0;
        lb.mn_ext = p.N;
        lb.K = Kz;
        float acc[8][TN];
        tile_mainloop<BK, STAGES, BN_, TA, TB, VEC, FFMA2, CK>(la, lb, As, Bs, (Kz + BK - 1) / BK,
                                                             a_col, b_col, acc);
        if (part != nullptr) {
            // the whole 128 x BN_ block, unmasked: the workspace holds full tiles
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int row = r < 4 ? a_col + r : 64 + a_col + (r - 4);
#pragma unroll
                for (int h = 0; h < NSB; ++h)
                    *reinterpret_cast<float4 *>(part + row * BN_ + h * 64 + b_col) =
                        make_float4(acc[r][4 * h], acc[r][4 * h + 1], acc[r][4 * h + 2],
                                    acc[r][4 * h + 3]);
            }
        } else {
            float *Cz = p.C + (int64_t)z * p.strideC;
            const bool plain = plain_epilogue(p);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int row = m0 + (r < 4 ? a_col + r : 64 + a_col + (r - 4));
                if (row >= p.M) continue;
                float *crow = Cz + (int64_t)row * p.ldc;
#pragma unroll
                for (int h = 0; h < NSB; ++h) {
                    const int col = n0 + h * 64 + b_col;
                    store_c4(p, crow, col,
                             make_float4(acc[r][4 * h], acc[r][4 * h + 1], acc[r][4 * h + 2],
                                         acc[r][4 * h + 3]),
                             VEC, plain);
                }
            }
        }
        __syncthreads();   // every warp is done with the ring before the next prologue refills it
    }
}

// Adds the pieces of the shared stream-K tiles: grid streamk_fixup_grid<BN_>,
// kFixupVecs float4 per thread (256 float4 apart, so each load instruction is
// coalesced across the CTA), the loads of a tile's first three pieces issued
// before any add; pieces added in K order (CTA order), then stored to C with
// the epilogue.
// Tiles that fell whole to one CTA are skipped.
constexpr int kFixupVecs = 4;

template <int BN_>
inline dim3 streamk_fixup_grid(int tiles_sk) {
    return dim3((unsigned)(BM * BN_ / (1024 * kFixupVecs)), (unsigned)tiles_sk);
}

template <int BN_, bool VEC>
__global__ void __launch_bounds__(256) streamk_fixup_kernel(const GemmArgs p, const StreamK sk) {
    constexpr int V = kFixupVecs;
    static_assert((BM * BN_) % (1024 * V) == 0, "whole float4 groups per CTA");
    pdl_wait();   // launched as a dependent of the tile kernel: its pieces first
    const int tl = blockIdx.y;
    const int64_t U = sk.units, f = (int64_t)tl * sk.kslices, l = f + sk.kslices - 1;
    const int c0 = streamk_owner(f, U, sk.G), c1 = streamk_owner(l, U, sk.G);
    if (c0 == c1) return;
    // element of the 128 x BN_ tile of this thread's vector r: e0 + 1024 r
    const int e0 = (blockIdx.x * 256 * V + threadIdx.x) * 4;
    float4 acc[V];
#pragma unroll
    for (int r = 0; r < V; ++r) acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    // the piece of CTA c in this tile, or null when c has no units
    auto piece_of = [&](int c) -> const float * {
        const int64_t start = (int64_t)c * U / sk.G;
        if (((int64_t)c + 1) * U / sk.G == start) return nullptr;
        const int slot = start >= f ? 0 : 1;   // the tile is c's first piece or its last
        return sk.ws + ((int64_t)c * 2 + slot) * (BM * BN_) + e0;
    };
    // the first three pieces (a shared tile mostly has two): every load
    // issued before the first add, then added in K order
    constexpr int kAhead = 3;
    const float *first[kAhead];
    int np = 0, c = c0;
    for (; c <= c1 && np < kAhead; ++c) {
        const float *pc = piece_of(c);
        if (pc != nullptr) first[np++] = pc;
    }
    float4 w[kAhead][V];
#pragma unroll
    for (int q = 0; q < kAhead; ++q)
        if (q < np)
#pragma unroll
            for (int r = 0; r < V; ++r) w[q][r] = *reinterpret_cast<const float4 *>(first[q] + 1024 * r);
#pragma unroll
    for (int q = 0; q < kAhead; ++q)
        if (q < np)
#pragma unroll
            for (int r = 0; r < V; ++r) {
                acc[r].x += w[q][r].x;
                acc[r].y += w[q][r].y;
                acc[r].z += w[q][r].z;
                acc[r].w += w[q][r].w;
            }
    for (; c <= c1; ++c) {
        const float *piece = piece_of(c);
        if (piece == nullptr) continue;
        float4 v[V];
#pragma unroll
        for (int r = 0; r < V; ++r) v[r] = *reinterpret_cast<const float4 *>(piece + 1024 * r);
#pragma unroll
        for (int r = 0; r < V; ++r) {
            acc[r].x += v[r].x;
            acc[r].y += v[r].y;
            acc[r].z += v[r].z;
            acc[r].w += v[r].w;
        }
    }
    int z, tm, tn;
    raster(p, sk.tiles_dp + tl, z, tm, tn);
    float *Cz = p.C + (int64_t)z * p.strideC;
    const bool plain = plain_epilogue(p);
#pragma unroll
    for (int r = 0; r < V; ++r) {
        const int e = e0 + 1024 * r;
        const int row = tm * BM + e / BN_, col = tn * BN_ + e % BN_;
        if (row < p.M) store_c4(p, Cz + (int64_t)row * p.ldc, col, acc[r], VEC, plain);
    }
}

}  // namespace simt
}  // namespace sgemm
