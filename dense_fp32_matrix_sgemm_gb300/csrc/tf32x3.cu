// FP32 GEMM on the tensor cores with the three-term TF32 split (3xTF32), and
// the plain single-term TF32 product.
//
// TF32 keeps 10 explicit mantissa bits, so one TF32 product loses about 750x
// in accuracy against FP32 FMA (the RRMSE comparison of 1.03e-6 vs 7.78e-4 on
// the ChetanC28/cuda-kernels page).  Writing every input as x = hi + lo with
// hi = x cut to TF32 (see tf32_hi) and lo = tf32_rn(x - hi), the product a*b
// is recovered to about 2^-20 relative by hi_a*hi_b + hi_a*lo_b + lo_a*hi_b
// (the lo*lo term is below that and dropped), each term a TF32 MMA
// accumulated in fp32 in TMEM.  With TERMS = 1 only hi_a*hi_b is formed, from
// hi = tf32_rn(x): the plain TF32 product.
//
// Stage 1 (one split launch for both operands): op(A) and op(B) are
//   rewritten into a caller-owned workspace as K-major planes
//   [batch][TERMS == 3 ? hi|lo : hi][rows][Kp] (Kp = K rounded up to 32 so
//   rows start on 128-byte boundaries).  M- or N-major operands are
//   corner-turned through a padded shared tile.  A K-contiguous operand with
//   aligned rows needs no hi plane for three terms (the GEMM loads the
//   caller's rows, which the MMA reads as hi), so only its lo plane is
//   written; for short reductions it needs no split at all (converter warps
//   make lo, or the rounded hi of one term, inside the GEMM).  The GEMM is
//   launched as a programmatic dependent of it and waits for it before
//   reading a plane.
// Stage 2 (persistent GEMM kernel, one CTA per SM walking 128 x BN output
//   tiles, BN = 256 or 128 picked per problem; 192 threads in three roles):
//   warp 0 / lane 0 issues TMA loads of the swizzled K slices (BK fp32 of K,
//   swizzle span = BK * 4 bytes; A planes 128 rows, B planes BN rows) into a
//   STAGES-deep ring that runs on across tiles; warp 1 owns TMEM and its lane
//   0 issues TERMS MMAs (M128 N=BN K8) per 8-wide K step into one of two
//   accumulator buffers where they fit, releasing each stage with
//   tcgen05.commit; warps 2-5 drain a finished accumulator 32 columns at a
//   time, add the two accumulators and store the tile while the MMAs of the
//   next one run.  For the plain product into a 16-byte-aligned C with N a
//   multiple of 4, each warp writes its 32 x 32 block into its own shared
//   staging buffers (128-byte swizzle, two per warp) and one lane stores it
//   with a TMA tensor store, which writes whole rows and clips the ragged
//   edges; otherwise the threads store their own rows.
//   This single-pass kernel serves reductions up to 256 deep (three terms)
//   and the plain product; longer three-term reductions run the K-chunked
//   kernel (tf32x3_chunked_kernel, below), same roles, same ring.
// The tensor cores add each MMA's partial sum into its fp32 accumulator with
// a rounding that is biased towards zero, so the error of a long K grows with
// the number of updates.  hi*hi therefore has an accumulator of its own (K/8
// updates) and the two small terms share the second one, whose values are
// 2^-10 smaller, so their rounding is negligible; one round-to-nearest add
// combines the two in the epilogue.  The K-chunked kernel goes further and
// adds the tensor cores' sums of every 128 of K in round-to-nearest fp32.
// Every mbarrier wait is bounded; a wait that runs out flags the CTA, the
// roles drain (copies in flight land, MMAs complete, TMEM is freed) and the
// library's device error word is raised.
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "gemm_args.h"
#include "tc_utils.cuh"
#include "tma_encode.h"

namespace sgemm {
namespace tf32x3 {

constexpr int BM = 128;
constexpr int THREADS = 128;   // the TF32 probe's CTA

// K-chunked kernel: K per chunk (the library's choice, see tf32x3_chunked_kernel)
// and the step a measurement may set it in (whole K blocks of both tile widths).
constexpr int kChunkK = 128;
constexpr int kChunkStep = 32;
std::atomic<int> g_chunk_k{kChunkK};

template <int BK_, int STAGES_, int TERMS_, int BN_ = 256>
struct Config {
    static constexpr int BK = BK_;             // fp32 of K per stage (one swizzled row)
    static constexpr int STAGES = STAGES_;
    static constexpr int TERMS = TERMS_;       // 3: hi/lo split; 1: plain TF32
    static constexpr int BN = BN_;             // output tile width (MMA N): 128 or 256
    static constexpr int ACC_COLS = BN;        // one fp32 accumulator column per output column
    static constexpr int PLANES = TERMS == 3 ? 2 : 1;
    static constexpr int ROW_BYTES = BK * 4;
    static constexpr int A_TILE = BM * ROW_BYTES;
    static constexpr int B_TILE = BN * ROW_BYTES;
    static constexpr int STAGE_BYTES = PLANES * (A_TILE + B_TILE);
    static_assert(BN == 128 || BN == 256, "tile width");
};

// The library's device status word (sgemm_device_status).  Bit 0: a
// pipeline wait in one of its kernels ran out.
__device__ unsigned int g_tf32x3_error = 0;

// ------------------------------------------------------------------ split

// The three-term split of an fp32 x.  A kind::tf32 MMA takes the upper 19
// bits of each 32-bit operand word (sign, exponent, 10 mantissa bits) and
// ignores the low 13, so hi is x with those bits cleared: the value the
// tensor core sees when it reads x itself, which lets a K-contiguous operand
// serve as its own hi plane.  x - hi is exact (the 13 dropped bits), and lo
// rounds it to TF32 (nearest, ties away).  |x - hi - lo| <= 2^-21 |x| and the
// dropped lo_a lo_b term is below 2^-20 |a b|.
__device__ __forceinline__ float tf32_hi(float x) {
    return __uint_as_float(__float_as_uint(x) & 0xffffe000u);
}
__device__ __forceinline__ float tf32_lo(float x, float hi) { return tc::to_tf32(x - hi); }

// One operand to split: rows r of op(X) (R of them per problem), element
// (r, k) at X[z*sX + r*ld + k] when kcontig, else at X[z*sX + k*ld + r];
// planes written to `out`.  `blocks` CTAs of the split grid serve it.
// lo_only (three terms, K-contiguous X): the GEMM reads X itself as the hi
// term, so only the lo plane is written, one plane per problem.
struct SplitJob {
    const float *X;
    int64_t ld, sX;
    float *out;
    int64_t blocks;
    int R;
    int kcontig;
    int vec;   // rows allow 16-byte loads (along K, or along r for M/N-major X)
    int lo_only;
};

struct SplitArgs {
    SplitJob job[2];   // op(A) and op(B)
    int K, Kp, batch;
};

// K-contiguous operand: one thread per four consecutive k of a row; 16-byte
// loads where the row allows, 16-byte stores always (rows of the planes are
// Kp long; the padding gets zeros).  CTA `b` of `blocks`, grid-stride.
template <int PLANES>
__device__ __forceinline__ void split_kcontig(const SplitJob &j, int K, int Kp, int batch,
                                              int64_t b) {
    const int64_t plane = (int64_t)j.R * Kp;
    const int quads = Kp / 4;
    const int64_t total = (int64_t)batch * j.R * quads;
    for (int64_t t = b * blockDim.x + threadIdx.x; t < total; t += j.blocks * blockDim.x) {
        const int64_t row = t / quads;
        const int k = (int)(t - row * quads) * 4;
        const int64_t z = row / j.R, r = row - z * j.R;
        const float *src = j.X + z * j.sX + r * j.ld + k;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j.vec && k + 3 < K) {
            x = __ldg(reinterpret_cast<const float4 *>(src));
        } else {
            if (k + 0 < K) x.x = __ldg(src + 0);
            if (k + 1 < K) x.y = __ldg(src + 1);
            if (k + 2 < K) x.z = __ldg(src + 2);
            if (k + 3 < K) x.w = __ldg(src + 3);
        }
        if constexpr (PLANES == 2) {
            const float4 h = make_float4(tf32_hi(x.x), tf32_hi(x.y), tf32_hi(x.z), tf32_hi(x.w));
            const float4 l = make_float4(tf32_lo(x.x, h.x), tf32_lo(x.y, h.y), tf32_lo(x.z, h.z),
                                         tf32_lo(x.w, h.w));
            if (j.lo_only) {
                *reinterpret_cast<float4 *>(j.out + z * plane + r * Kp + k) = l;
            } else {
                float *hi = j.out + (2 * z) * plane + r * Kp + k;
                *reinterpret_cast<float4 *>(hi) = h;
                *reinterpret_cast<float4 *>(hi + plane) = l;
            }
        } else {
            *reinterpret_cast<float4 *>(j.out + z * plane + r * Kp + k) =
                make_float4(tc::to_tf32(x.x), tc::to_tf32(x.y), tc::to_tf32(x.z),
                            tc::to_tf32(x.w));
        }
    }
}

// M/N-major operand: transposed through a 32 x 33 shared tile (one 32 x 32
// block of (k, r) per step, the 256 threads as 32 x 8) so both the read and
// the write are coalesced.  Plane columns k >= K are not written: the GEMM's
// tensor maps end at K.
template <int PLANES>
__device__ __forceinline__ void split_transpose(const SplitJob &j, int K, int Kp, int batch,
                                                int64_t b, float (*tile)[33]) {
    const int64_t plane = (int64_t)j.R * Kp;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int64_t rt_n = (j.R + 31) / 32, kt_n = (K + 31) / 32;
    const int64_t total = (int64_t)batch * kt_n * rt_n;
    for (int64_t t = b; t < total; t += j.blocks) {
        const int64_t z = t / (kt_n * rt_n), rem = t - z * kt_n * rt_n;
        const int k0 = (int)(rem / rt_n) * 32, r0 = (int)(rem % rt_n) * 32;
        const float *src = j.X + z * j.sX;
        float *hi = j.out + (PLANES * z) * plane;
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
            const int k = k0 + ty + i, r = r0 + tx;
            tile[ty + i][tx] = (k < K && r < j.R) ? src[(int64_t)k * j.ld + r] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
            const int r = r0 + ty + i, k = k0 + tx;
            if (r < j.R && k < K) {
                const float x = tile[tx][ty + i];
                if constexpr (PLANES == 2) {
                    const float h = tf32_hi(x);
                    hi[(int64_t)r * Kp + k] = h;
                    hi[plane + (int64_t)r * Kp + k] = tf32_lo(x, h);
                } else {
                    hi[(int64_t)r * Kp + k] = tc::to_tf32(x);
                }
            }
        }
        __syncthreads();
    }
}

// M/N-major operand with 16-byte aligned rows: 32 (k) x 128 (r) blocks.  Each
// thread loads four 16-byte row segments of X (4 consecutive r), the block
// passes through a shared tile of row stride 129 floats, and each thread
// writes 4 consecutive k of a plane row per 16-byte store: a quarter of the
// load and store instructions of the 32 x 32 form and four times the bytes
// per barrier.  Reads of the tile (tile[4q + e][r], q = thread % 8,
// r = thread / 8 + 32 i) fall in 32 distinct banks.  Plane columns from K up
// to the block's end get zeros (inside the row: Kp is a multiple of 32).
template <int PLANES>
__device__ __forceinline__ void split_transpose_wide(const SplitJob &j, int K, int Kp, int batch,
                                                     int64_t b, float (*tile)[129]) {
    const int64_t plane = (int64_t)j.R * Kp;
    const int tid = threadIdx.x;
    const int64_t rt_n = (j.R + 127) / 128, kt_n = (K + 31) / 32;
    const int64_t total = (int64_t)batch * kt_n * rt_n;
    const int lr = 4 * (tid & 31), lk = tid >> 5;   // load: r quad, k row (0..7)
    const int kq = tid & 7, sr = tid >> 3;          // store: k quad, plane row (0..31)
    for (int64_t t = b; t < total; t += j.blocks) {
        const int64_t z = t / (kt_n * rt_n), rem = t - z * kt_n * rt_n;
        const int k0 = (int)(rem / rt_n) * 32, r0 = (int)(rem % rt_n) * 128;
        const float *src = j.X + z * j.sX;
        float4 x[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = k0 + lk + 8 * i, r = r0 + lr;
            x[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k < K) {
                const float *row = src + (int64_t)k * j.ld + r;
                if (r + 3 < j.R) {
                    x[i] = __ldg(reinterpret_cast<const float4 *>(row));
                } else {
                    if (r + 0 < j.R) x[i].x = __ldg(row + 0);
                    if (r + 1 < j.R) x[i].y = __ldg(row + 1);
                    if (r + 2 < j.R) x[i].z = __ldg(row + 2);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float *trow = tile[lk + 8 * i] + lr;
            trow[0] = x[i].x;
            trow[1] = x[i].y;
            trow[2] = x[i].z;
            trow[3] = x[i].w;
        }
        __syncthreads();
        float *hi = j.out + (PLANES * z) * plane;
        const int k = k0 + 4 * kq;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = sr + 32 * i, r = r0 + c;
            if (r < j.R) {
                const float4 v = make_float4(tile[4 * kq][c], tile[4 * kq + 1][c],
                                             tile[4 * kq + 2][c], tile[4 * kq + 3][c]);
                float *dst = hi + (int64_t)r * Kp + k;
                if constexpr (PLANES == 2) {
                    const float4 h = make_float4(tf32_hi(v.x), tf32_hi(v.y), tf32_hi(v.z),
                                                 tf32_hi(v.w));
                    *reinterpret_cast<float4 *>(dst) = h;
                    *reinterpret_cast<float4 *>(dst + plane) =
                        make_float4(tf32_lo(v.x, h.x), tf32_lo(v.y, h.y), tf32_lo(v.z, h.z),
                                    tf32_lo(v.w, h.w));
                } else {
                    *reinterpret_cast<float4 *>(dst) =
                        make_float4(tc::to_tf32(v.x), tc::to_tf32(v.y), tc::to_tf32(v.z),
                                    tc::to_tf32(v.w));
                }
            }
        }
        __syncthreads();
    }
}

// Both operands in one launch: CTAs [0, job[0].blocks) split op(A), the rest
// op(B).  The GEMM that follows is launched as a programmatic dependent, so
// this grid lets it start its set-up early; the GEMM waits for this grid's
// completion before it reads a plane.
template <int PLANES>
__global__ void __launch_bounds__(256) split_kernel(const SplitArgs a) {
    __shared__ float tile[32 * 129];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int w = (int64_t)blockIdx.x < a.job[0].blocks ? 0 : 1;
    const int64_t b = (int64_t)blockIdx.x - (w ? a.job[0].blocks : 0);
    const SplitJob j = w ? a.job[1] : a.job[0];   // no dynamic index into the parameters
    if (j.kcontig)
        split_kcontig<PLANES>(j, a.K, a.Kp, a.batch, b);
    else if (j.vec)
        split_transpose_wide<PLANES>(j, a.K, a.Kp, a.batch, b,
                                     reinterpret_cast<float (*)[129]>(tile));
    else
        split_transpose<PLANES>(j, a.K, a.Kp, a.batch, b, reinterpret_cast<float (*)[33]>(tile));
}

// ------------------------------------------------------------------ GEMM

struct Tf32x3Params {
    float *C;
    int64_t ldc, strideC;
    int M, N, K;
    int tiles_m, tiles_n, group_m;
    int vec_c;   // C rows allow 16-byte stores
    int tma_c;   // store C through the tmC tensor map (plain epilogue, aligned C)
    int tma_n;   // with tma_c: 32-column blocks of C ending at or before column
                 // tma_n go through the map, the block holding the last
                 // columns of a width that is not a multiple of 4 does not
    int batch;
    float alpha, beta;      // epilogue C = alpha * acc + beta * C + bias[col]
    const float *bias;
    int kcb;                // K-chunked kernel: K blocks per chunk (>= 1)
    // K-chunked kernel schedule (see piece_of): the first tiles_dp tiles are
    // computed whole; each of the other `tail` tiles is split into `split`
    // K segments (tail = 0: every tile whole).  Segment j of tail tile t runs
    // on CTA j * tail + t, and its sum is partial tile j * tail + t of `part`.
    int tiles_dp, tail, split;
    float *part;            // [split * tail][BM * BN] partial tiles, row-major
};

__device__ __forceinline__ void raster(const Tf32x3Params &p, int bid, int &z, int &tm, int &tn) {
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

// Stores the 32 tile rows held in TMEM lanes 32q..32q+31 of the accumulator
// at `acc` (small-term accumulator ACC_COLS columns further) to C.  The
// calling warp must be a warp whose TMEM lane quarter is q.
//   TMA path (p.tma_c): 32 columns at a time through the warp's two 4 KB
//   staging buffers at `stage` (1024-byte aligned; the 128-byte swizzle puts
//   16-byte chunk j of row r at chunk j ^ (r & 7), so the eight rows a
//   quarter-warp writes hit distinct banks), one TMA store per chunk issued by
//   lane 0.  `cc` counts the chunks staged so far (across calls), picks the
//   buffer and says when to wait for the store two chunks back.
//   Otherwise: each thread stores its own row, with the epilogue applied.
template <class CFG>
__device__ __forceinline__ void store_tile_rows(const Tf32x3Params &p, const CUtensorMap *tmC,
                                                uint32_t acc, int q, int lane, int z, int m0,
                                                int n0, uint32_t stage, int &cc) {
    constexpr int BN = CFG::BN, ACC_COLS = CFG::ACC_COLS;
    const uint32_t lane_base = acc + ((uint32_t)(32 * q) << 16);
    if (p.tma_c) {
        const int row0 = m0 + 32 * q;
        for (int c = 0; row0 < p.M && c < BN / 32 && n0 + 32 * c < p.N; ++c) {
            float v[32];
            const uint32_t ta = lane_base + (uint32_t)(32 * c);
            tc::tmem_ld_32(ta, v);
            if constexpr (CFG::TERMS == 3) {
                float w[32];
                tc::tmem_ld_32(ta + ACC_COLS, w);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] += w[j];
            }
            if (n0 + 32 * c + 32 > p.tma_n) {
                // the last columns of a width that is not a multiple of 4:
                // each thread stores its own row (plain product)
                const int row = row0 + lane;
                if (row < p.M) {
                    float *crow = p.C + (int64_t)z * p.strideC + (int64_t)row * p.ldc;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (n0 + 32 * c + j < p.N) crow[n0 + 32 * c + j] = v[j];
                }
                continue;
            }
            const uint32_t buf = stage + (uint32_t)(cc & 1) * 4096u;
            if (cc >= 2) {
                if (lane == 0) tc::bulk_wait_group_read<1>();   // the store of chunk cc-2 has read it
                __syncwarp();
            }
            const uint32_t rbase = buf + (uint32_t)lane * 128u;
#pragma unroll
            for (int j = 0; j < 8; ++j)
                tc::st_shared_v4(rbase + ((uint32_t)(j ^ (lane & 7)) << 4), v[4 * j], v[4 * j + 1],
                                 v[4 * j + 2], v[4 * j + 3]);
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tc::tma_store_3d(tmC, buf, n0 + 32 * c, row0, z);
                tc::bulk_commit_group();
            }
            ++cc;
        }
        return;
    }
    const int row = m0 + 32 * q + lane;
    float *crow = p.C + (int64_t)z * p.strideC + (int64_t)row * p.ldc;
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        float v[32];
        const uint32_t ta = lane_base + (uint32_t)(32 * c);
        tc::tmem_ld_32(ta, v);
        if constexpr (CFG::TERMS == 3) {
            float w[32];
            tc::tmem_ld_32(ta + ACC_COLS, w);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += w[j];
        }
        if (row < p.M) {
            const int col0 = n0 + 32 * c;
            if (!(p.alpha == 1.f && p.beta == 0.f && p.bias == nullptr)) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int col = col0 + j;
                    const float old = (p.beta != 0.f && col < p.N) ? crow[col] : 0.f;
                    const float b = (p.bias != nullptr && col < p.N) ? p.bias[col] : 0.f;
                    v[j] = fmaf(p.beta, old, p.alpha * v[j]) + b;
                }
            }
            if (p.vec_c && col0 + 31 < p.N) {
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4 *>(crow + col0 + j) =
                        make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (col0 + j < p.N) crow[col0 + j] = v[j];
            }
        }
    }
}

// ------------------------------------------------------------------ GEMM

// Persistent GEMM kernel: one CTA per SM walks tiles
// blockIdx.x, blockIdx.x + gridDim.x, ... with warp-specialised roles.
//   warp 0, lane 0: TMA producer; the ring runs on across tile boundaries,
//                   so the next tile's slices load while this one finishes;
//   warp 1, lane 0: MMA issuer, into accumulator buffer i % ACC_BUFS; warp 1
//                   allocates and frees TMEM;
//   warps 2-5:      epilogue, warp w draining TMEM lane quarter w % 4 through
//                   its own staging buffers (outside the ring), then arriving
//                   on the buffer's "empty" barrier;
//   warps 6-9:      (CONV only) converters: wait for a stage to land, make
//                   the planes of its raw operand tiles in place, fence the
//                   async proxy and arrive on the stage's "converted" barrier,
//                   which the MMA issuer then waits on instead of "full".
// With ACC_BUFS = 2 the MMAs of tile i+1 overlap the epilogue of tile i; the
// 128 x 256 three-term tile needs all 512 TMEM columns for one tile
// (ACC_BUFS = 1), and there only the next tile's loads overlap its epilogue.
// Barrier phases: a ring stage's j-th fill is waited on with parity j & 1 and
// its (j-1)-th release with parity (j-1) & 1; accumulator buffer b's u-th
// result likewise.  Every wait is bounded and the abort word stops all roles.
constexpr int PTHREADS = 192;   // producer, MMA and 4 epilogue warps
constexpr int kConvWarps = 4;   // converter warps when an operand arrives raw

// RAW: bit 0 set when op(A), bit 1 when op(B), is loaded as the caller's
// fp32 (K-contiguous rows) into the stage's hi slot instead of a hi plane.
// CONV (a subset of RAW): converter warps make that operand's planes inside
// the stage (three terms: the lo slot from the raw values, which the MMAs
// read as hi as they are; one term: the hi slot rounded in place).  An
// operand in RAW but not CONV (three terms only) takes its lo slot from a
// lo-only plane the split kernel wrote.
template <class CFG, int ACC_BUFS, int RAW = 0, int CONV = 0>
struct Persist {
    static_assert((CONV & ~RAW) == 0, "converted operands are loaded raw");
    static_assert(CFG::PLANES == 2 || RAW == CONV, "one term rounds its raw operand in place");
    static constexpr int CONV_WARPS = CONV ? kConvWarps : 0;
    static constexpr int THREADS = PTHREADS + 32 * CONV_WARPS;
    static constexpr int BUF_COLS = CFG::TERMS == 3 ? 2 * CFG::BN : CFG::BN;
    static constexpr int TMEM_COLS = ACC_BUFS * BUF_COLS <= 256 ? 256 : 512;
    static constexpr int STAGING = 4 * 8192;   // 4 epilogue warps x two 4 KB buffers
    static constexpr int BARS = (CONV ? 3 : 2) * CFG::STAGES + 2 * ACC_BUFS + 1;
    // transaction bytes of one stage: a converted operand lands as one plane
    static constexpr int TX_BYTES = ((CONV & 1) ? CFG::A_TILE : CFG::PLANES * CFG::A_TILE) +
                                    ((CONV & 2) ? CFG::B_TILE : CFG::PLANES * CFG::B_TILE);
    static constexpr int SMEM_BYTES = CFG::STAGES * CFG::STAGE_BYTES + STAGING + 1024 + 256;
    static_assert(ACC_BUFS * BUF_COLS <= 512, "accumulators exceed tensor memory");
    static_assert(BARS * 8 + 8 <= 256, "barrier area");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// The converted operand tiles of one landed stage, each holding raw fp32 x in
// its hi slot.  Three terms: the same position of the lo slot (one tile
// further) gets tf32_lo(x, tf32_hi(x)) and the hi slot stays as it is (the
// MMAs read x as tf32_hi(x)).  One term: the hi slot becomes tf32_rn(x) in
// place.  These are the values the split kernel writes, so the MMAs see the
// same operands.  The swizzle moves whole 16-byte chunks, so position-wise
// work ignores it.  Thread t of NT takes 16-byte chunks t, t + NT, ... of
// each tile, and issues every load of the stage before its first store, so
// one shared-memory round trip covers the stage.
template <int PLANES, int CONV, int A_BYTES, int B_BYTES, int NT>
__device__ __forceinline__ void convert_stage(uint8_t *st, int t) {
    constexpr int NA = (CONV & 1) ? A_BYTES / (16 * NT) : 0;
    constexpr int NB = (CONV & 2) ? B_BYTES / (16 * NT) : 0;
    static_assert(A_BYTES % (16 * NT) == 0 && B_BYTES % (16 * NT) == 0, "whole chunks per thread");
    float4 *ahi = reinterpret_cast<float4 *>(st);
    float4 *bhi = reinterpret_cast<float4 *>(st + PLANES * A_BYTES);
    float4 *alo = PLANES == 2 ? reinterpret_cast<float4 *>(st + A_BYTES) : ahi;
    float4 *blo = PLANES == 2 ? reinterpret_cast<float4 *>(st + PLANES * A_BYTES + B_BYTES) : bhi;
    float4 xa[NA > 0 ? NA : 1], xb[NB > 0 ? NB : 1];
#pragma unroll
    for (int i = 0; i < NA; ++i) xa[i] = ahi[t + i * NT];
#pragma unroll
    for (int i = 0; i < NB; ++i) xb[i] = bhi[t + i * NT];
    auto conv = [](float4 x) {
        if constexpr (PLANES == 2)
            return make_float4(tf32_lo(x.x, tf32_hi(x.x)), tf32_lo(x.y, tf32_hi(x.y)),
                               tf32_lo(x.z, tf32_hi(x.z)), tf32_lo(x.w, tf32_hi(x.w)));
        else
            return make_float4(tc::to_tf32(x.x), tc::to_tf32(x.y), tc::to_tf32(x.z),
                               tc::to_tf32(x.w));
    };
#pragma unroll
    for (int i = 0; i < NA; ++i) alo[t + i * NT] = conv(xa[i]);
#pragma unroll
    for (int i = 0; i < NB; ++i) blo[t + i * NT] = conv(xb[i]);
}

// tmA / tmB: the operand's planes, or (RAW) its raw rows; tmAlo / tmBlo: the
// lo-only plane of an operand in RAW but not CONV (unused otherwise).
template <class CFG, int ACC_BUFS, int RAW, int CONV>
__global__ void __launch_bounds__(Persist<CFG, ACC_BUFS, RAW, CONV>::THREADS, 1)
tf32x3_persistent_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmAlo,
                         const __grid_constant__ CUtensorMap tmBlo,
                         const __grid_constant__ CUtensorMap tmC, const Tf32x3Params p) {
    using P = Persist<CFG, ACC_BUFS, RAW, CONV>;
    constexpr int BK = CFG::BK, STAGES = CFG::STAGES, PLANES = CFG::PLANES;
    constexpr int BN = CFG::BN, ACC_COLS = CFG::ACC_COLS;
    constexpr int A_TILE = CFG::A_TILE, B_TILE = CFG::B_TILE, STAGE_BYTES = CFG::STAGE_BYTES;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_addr = tc::smem_u32_generic(smem_raw);
    const uint32_t pad = (1024 - (raw_addr & 1023)) & 1023;
    uint8_t *smem = smem_raw + pad;
    const uint32_t ring = tc::smem_u32_generic(smem);
    const uint32_t staging = ring + STAGES * STAGE_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES + P::STAGING);
    const uint32_t full0 = tc::smem_u32_generic(bars);
    const uint32_t empty0 = full0 + 8 * STAGES;
    const uint32_t accf0 = empty0 + 8 * STAGES;     // accumulator b holds a finished tile
    const uint32_t acce0 = accf0 + 8 * ACC_BUFS;    // accumulator b has been drained
    const uint32_t done_bar = acce0 + 8 * ACC_BUFS;
    const uint32_t conv0 = done_bar + 8;            // (CONV) stage s converted
    const uint32_t ready0 = CONV ? conv0 : full0;   // what the MMA waits for
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + P::BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = p.batch * p.tiles_m * p.tiles_n;
    const int nlocal = ((int)blockIdx.x < total) ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int kblocks = (p.K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(full0 + 8 * s, 1);
            tc::mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < ACC_BUFS; ++b) {
            tc::mbar_init(accf0 + 8 * b, 1);
            tc::mbar_init(acce0 + 8 * b, 4);   // one arrival per epilogue warp
        }
        tc::mbar_init(done_bar, 1);
        if constexpr (CONV != 0)
            for (int s = 0; s < STAGES; ++s) tc::mbar_init(conv0 + 8 * s, P::CONV_WARPS);
        *abort_flag = 0;
        tc::fence_barrier_init();
        tc::tma_prefetch_desc(&tmA);
        tc::tma_prefetch_desc(&tmB);
        if constexpr ((RAW & ~CONV & 1) != 0) tc::tma_prefetch_desc(&tmAlo);
        if constexpr ((RAW & ~CONV & 2) != 0) tc::tma_prefetch_desc(&tmBlo);
    }
    if (warp == 1) tc::tmem_alloc(tc::smem_u32_generic(tmem_slot), P::TMEM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // Launched as a programmatic dependent of the split kernel: the set-up above
    // may overlap its tail; nothing below touches global memory before the
    // split grid has completed and its planes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            long long issued = 0;
            bool stop = false;
            for (int i = 0; i < nlocal && !stop; ++i) {
                int z, tm, tn;
                raster(p, (int)blockIdx.x + i * (int)gridDim.x, z, tm, tn);
                const int m0 = tm * BM, n0 = tn * BN;
                for (int kb = 0; kb < kblocks; ++kb) {
                    const long long g = (long long)i * kblocks + kb;
                    const int s = (int)(g % STAGES);
                    const int j = (int)(g / STAGES);
                    if (g >= STAGES && !tc::mbar_wait(empty0 + 8 * s, (j & 1) ^ 1, abort_flag)) {
                        stop = true;
                        break;
                    }
                    const uint32_t st = ring + s * STAGE_BYTES;
                    const uint32_t fb = full0 + 8 * s;
                    tc::mbar_arrive_expect_tx(fb, P::TX_BYTES);
                    const int k0 = kb * BK;
                    // a raw operand: the caller's rows into the hi slot (and,
                    // unless converted in the stage, its lo plane); else its planes
                    if constexpr (RAW & 1) {
                        tc::tma_load_3d(st, &tmA, fb, k0, m0, z);
                        if constexpr (!(CONV & 1))
                            tc::tma_load_3d(st + A_TILE, &tmAlo, fb, k0, m0, z);
                    } else {
#pragma unroll
                        for (int pl = 0; pl < PLANES; ++pl)
                            tc::tma_load_3d(st + pl * A_TILE, &tmA, fb, k0, m0, PLANES * z + pl);
                    }
                    if constexpr (RAW & 2) {
                        tc::tma_load_3d(st + PLANES * A_TILE, &tmB, fb, k0, n0, z);
                        if constexpr (!(CONV & 2))
                            tc::tma_load_3d(st + PLANES * A_TILE + B_TILE, &tmBlo, fb, k0, n0, z);
                    } else {
#pragma unroll
                        for (int pl = 0; pl < PLANES; ++pl)
                            tc::tma_load_3d(st + PLANES * A_TILE + pl * B_TILE, &tmB, fb, k0, n0,
                                            PLANES * z + pl);
                    }
                    issued = g + 1;
                }
            }
            if (*abort_flag) {
                // let this thread's copies in flight land before the CTA exits
                for (long long g = (issued > STAGES ? issued - STAGES : 0); g < issued; ++g) {
                    const int s = (int)(g % STAGES);
                    const long long t0 = clock64();
                    while (!tc::mbar_try_wait(full0 + 8 * s, (int)((g / STAGES) & 1)) &&
                           clock64() - t0 < tc::kWaitLimitCycles) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            constexpr uint32_t idesc = tc::tf32_idesc<BM, BN>();
            bool stop = false;
            for (int i = 0; i < nlocal && !stop; ++i) {
                const int b = i % ACC_BUFS, u = i / ACC_BUFS;
                if (i >= ACC_BUFS && !tc::mbar_wait(acce0 + 8 * b, (u - 1) & 1, abort_flag)) break;
                tc::fence_after_sync();
                const uint32_t acc = tmem + (uint32_t)(b * P::BUF_COLS);
                for (int kb = 0; kb < kblocks; ++kb) {
                    const long long g = (long long)i * kblocks + kb;
                    const int s = (int)(g % STAGES);
                    if (!tc::mbar_wait(ready0 + 8 * s, (int)((g / STAGES) & 1), abort_flag)) {
                        stop = true;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t st = ring + s * STAGE_BYTES;
                    const uint64_t ahi = tc::kmajor_desc<CFG::ROW_BYTES>(st);
                    const uint64_t bhi = tc::kmajor_desc<CFG::ROW_BYTES>(st + PLANES * A_TILE);
#pragma unroll
                    for (int kk = 0; kk < BK / 8; ++kk) {
                        const uint64_t step = (uint64_t)(kk * 32) >> 4;
                        const uint32_t first = (kb == 0 && kk == 0) ? 0u : 1u;
                        if constexpr (CFG::TERMS == 3) {
                            const uint64_t alo = tc::kmajor_desc<CFG::ROW_BYTES>(st + A_TILE);
                            const uint64_t blo =
                                tc::kmajor_desc<CFG::ROW_BYTES>(st + 2 * A_TILE + B_TILE);
                            tc::mma_tf32(acc + ACC_COLS, alo + step, bhi + step, idesc, first);
                            tc::mma_tf32(acc + ACC_COLS, ahi + step, blo + step, idesc, 1u);
                        }
                        tc::mma_tf32(acc, ahi + step, bhi + step, idesc, first);
                    }
                    tc::mma_commit(empty0 + 8 * s);
                }
                if (!stop) tc::mma_commit(accf0 + 8 * b);
            }
            tc::mma_commit(done_bar);   // tracks every MMA issued above, also on abort
        }
    } else if (warp < 6) {
        // ---------------- epilogue warps 2-5: TMEM lane quarter warp % 4
        const int q = warp & 3;
        const uint32_t stage = staging + (uint32_t)(warp - 2) * 8192u;
        int cc = 0;
        for (int i = 0; i < nlocal; ++i) {
            const int b = i % ACC_BUFS, u = i / ACC_BUFS;
            const bool ok = tc::mbar_wait(accf0 + 8 * b, u & 1, abort_flag);
            __syncwarp();
            // one warp-uniform decision: the TMEM loads are warp-collective
            if (!__all_sync(0xffffffffu, ok && !*abort_flag)) break;
            tc::fence_after_sync();
            int z, tm, tn;
            raster(p, (int)blockIdx.x + i * (int)gridDim.x, z, tm, tn);
            store_tile_rows<CFG>(p, &tmC, tmem + (uint32_t)(b * P::BUF_COLS), q, lane, z, tm * BM,
                                 tn * BN, stage, cc);
            tc::fence_before_sync();   // the TMEM loads above precede the release
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(acce0 + 8 * b);
        }
        if (lane == 0 && cc > 0) tc::bulk_wait_group_read<0>();
    } else if constexpr (CONV != 0) {
        // ---------------- converter warps 6..: raw operand tiles -> planes
        constexpr int NT = 32 * P::CONV_WARPS;
        const int t = (int)threadIdx.x - PTHREADS;
        for (int i = 0; i < nlocal; ++i) {
            bool stop = false;
            for (int kb = 0; kb < kblocks; ++kb) {
                const long long g = (long long)i * kblocks + kb;
                const int s = (int)(g % STAGES);
                const bool ok = tc::mbar_wait(full0 + 8 * s, (int)((g / STAGES) & 1), abort_flag);
                // one warp-uniform decision
                if (!__all_sync(0xffffffffu, ok && !*abort_flag)) {
                    stop = true;
                    break;
                }
                uint8_t *st = smem + s * STAGE_BYTES;
                convert_stage<PLANES, CONV, A_TILE, B_TILE, NT>(st, t);
                // the planes are read by the tensor cores (async proxy)
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(conv0 + 8 * s);
            }
            if (stop) break;
        }
    }
    __syncwarp();

    tc::fence_before_sync();
    __syncthreads();
    // after every role has finished, so a wait that ran out late is reported too
    if (*abort_flag && threadIdx.x == 0) atomicOr(&g_tf32x3_error, 1u);
    if (warp == 1) {
        // every MMA issued has completed before TMEM is freed
        int local_abort = 0;
        (void)tc::mbar_wait(done_bar, 0, &local_abort);
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, P::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ K-chunked GEMM

// The three-term product over long reductions, with the tensor cores' sums
// promoted to round-to-nearest fp32 adds every 128 of K.
//
// The tensor cores add each MMA's result into its fp32 TMEM accumulator with
// a rounding biased towards zero, so over K/8 updates the errors add up with
// one sign: 3072^3 came out at an RRMSE of 7.3e-6 with hi*hi in an accumulator
// of its own, seven times that of sequential FP32 FMA.  Here no accumulator
// absorbs more than 16 K steps.  The MMAs of K chunk c of a tile go into chunk
// accumulator c % 2 (TMEM columns [256 (c % 2), 256 (c % 2) + 256)), starting
// from zero; once a chunk is complete, the epilogue warps load it and add it
// into a running sum held in their registers with ordinary fp32 adds
// (round to nearest even), and hand the accumulator back to the MMA issuer,
// which meanwhile fills the other one.  After the last chunk the running sum
// is the tile's result and is stored.  The chunk sums are added in ascending
// chunk order, so results stay deterministic, and small-integer inputs stay
// exact (every partial sum is an exact float).
//
// Chunk length: measured at 3072^3 (RRMSE / time of the whole call), 64 of K
// 5.6e-7 / +2.7 %, 128 1.0e-6 / +1.1 %, 256 1.9e-6 / +0.3 %, against the same
// kernel with one chunk per tile (2.2e-5).  What a chunk costs is the MMA
// issuer waiting at the chunk boundary for the previous chunk's drain: the
// epilogue's TMEM loads of one accumulator complete slowly while the tensor
// cores write the other (the same kernel with the loads removed, or with the
// issuer not waiting, runs as fast as one chunk per tile; halving the loaded
// columns changes nothing).  128 gives the FP32-FMA path's accuracy (RRMSE
// 9.9e-7 at 3072^3) for about 1 %.
//
// TMEM layout of one chunk accumulator (256 columns, lane = tile row):
//   128-wide tile: hi*hi in columns [0, 128), the two small terms in
//     [128, 256) (as in the single-pass kernel);
//   256-wide tile: all three terms in one 256-column block (the small terms'
//     updates round at hi*hi's magnitude, three per K step instead of one,
//     which the chunking keeps well below the bound).
// Warps: 0 TMA producer (as in the persistent kernel), 1 MMA issuer and TMEM
// owner, 2-9 epilogue: warp w drains TMEM lane quarter w % 4 and column half
// (w - 2) / 4, i.e. 32 rows x BN/2 columns of the running sum per warp.
template <class CFG>
struct Chunked {
    static constexpr int BN = CFG::BN;
    static constexpr bool SEP = BN == 128;   // hi*hi apart from the small terms
    static constexpr int SLOT_COLS = 256;
    static constexpr int NSLOT = 2;
    static constexpr int KC = kChunkK;            // K per chunk unless measured otherwise (Tf32x3Params::kcb)
    static constexpr int EPI_WARPS = 8;
    static constexpr int COLS = BN / 2;           // running-sum columns per epilogue thread
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int STAGING = EPI_WARPS * 4096;   // one 32 x 32 fp32 block per warp
    static constexpr int BARS = 2 * CFG::STAGES + 2 * NSLOT + 1;
    static constexpr int SMEM_BYTES = CFG::STAGES * CFG::STAGE_BYTES + STAGING + 1024 + 256;
    static_assert(CFG::TERMS == 3, "the chunked kernel forms the three-term product");
    static_assert(KC % CFG::BK == 0, "chunks are whole K blocks");
    static_assert(kChunkStep % CFG::BK == 0, "every chunk length is whole K blocks");
    static_assert(NSLOT * SLOT_COLS == 512, "two chunk accumulators fill tensor memory");
    static_assert((SEP ? 2 * BN : BN) == SLOT_COLS, "chunk accumulator width");
    static_assert(BARS * 8 + 8 <= 256, "barrier area");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// Stores 32 rows x COLS columns of running sums from the calling warp's
// threads (thread `lane` holds row m0 + 32q + lane, columns n0 .. n0 + COLS
// - 1 of a rows x cols matrix), 32 columns at a time through the warp's 4 KB
// staging block (128-byte swizzle: 16-byte chunk j of row r at chunk
// j ^ (r & 7), so the eight rows a quarter-warp writes, and the 32 columns of
// one row the warp reads back, hit distinct banks).
//   tma: one lane stores the block with a TMA tensor store through `map`
//   (C, or the partial tiles as [slot][BM][BN]) at (n0 + 32c, row, z), after
//   the previous block's store has read the staging block, for blocks that
//   end at or before column tma_n; `cc` counts the blocks stored this way so
//   far.
//   Otherwise (C only) the warp reads the block back a row at a time, lane j
//   taking column j, and stores it with the epilogue: each store is one
//   128-byte row segment.
template <int COLS>
__device__ __forceinline__ void store_running_rows(const Tf32x3Params &p, const CUtensorMap *map,
                                                   bool tma, int tma_n, const float (&run)[COLS],
                                                   int q, int lane, int z, int m0, int n0,
                                                   int rows, int cols, uint32_t stage, int &cc) {
    const int row0 = m0 + 32 * q;
    if (row0 >= rows) return;
    const uint32_t rbase = stage + (uint32_t)lane * 128u;
#pragma unroll
    for (int c = 0; c < COLS / 32; ++c) {
        if (n0 + 32 * c >= cols) break;
        if (cc > 0) {
            if (lane == 0) tc::bulk_wait_group_read<0>();   // the previous store has read the block
        }
        __syncwarp();   // (and, without TMA, the warp's reads of the previous block are done)
#pragma unroll
        for (int j = 0; j < 8; ++j)
            tc::st_shared_v4(rbase + ((uint32_t)(j ^ (lane & 7)) << 4), run[32 * c + 4 * j],
                             run[32 * c + 4 * j + 1], run[32 * c + 4 * j + 2],
                             run[32 * c + 4 * j + 3]);
        if (tma && n0 + 32 * c + 32 <= tma_n) {
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tc::tma_store_3d(map, stage, n0 + 32 * c, row0, z);
                tc::bulk_commit_group();
            }
            ++cc;
            continue;
        }
        __syncwarp();
        const int col = n0 + 32 * c + lane;
        const uint32_t cofs = (uint32_t)((lane & 3) * 4);
        const int rows = min(32, p.M - row0);
#pragma unroll 1
        for (int r = 0; r < rows; ++r) {
            float v;
            asm volatile("ld.shared.f32 %0, [%1];"
                         : "=f"(v)
                         : "r"(stage + (uint32_t)r * 128u +
                               ((uint32_t)((lane >> 2) ^ (r & 7)) << 4) + cofs)
                         : "memory");
            if (col < p.N) {
                float *cp = p.C + (int64_t)z * p.strideC + (int64_t)(row0 + r) * p.ldc + col;
                if (!(p.alpha == 1.f && p.beta == 0.f && p.bias == nullptr)) {
                    const float old = p.beta != 0.f ? *cp : 0.f;
                    const float b = p.bias != nullptr ? p.bias[col] : 0.f;
                    v = fmaf(p.beta, old, p.alpha * v) + b;
                }
                *cp = v;
            }
        }
    }
}

// The K-chunked kernel's schedule over its G CTAs.  The first tiles_dp tiles
// (whole waves) are computed whole, tile c + i*G on CTA c.  The remaining
// `tail` tiles, fewer than G, would leave G - tail SMs idle for a whole tile
// time; instead each is split into `split` = G / tail segments of K blocks
// [j * kblocks / split, (j+1) * kblocks / split), and segment j of tail tile
// t runs on CTA j * tail + t, after its whole tiles.  The segments of one
// index start together and walk K in step, so tiles sharing an operand
// panel read the same K slices at about the same time and L2 serves the
// repeats, as it does for the whole-tile waves.  (Dealing the tail's K
// blocks out evenly over all CTAs, stream-K style, starts every CTA at a
// different K offset: at 3072^3 that read 637 MB from DRAM against 251 MB
// and ran 12 % slower.)  A segment's sum is a partial tile, which
// tf32x3_fixup_kernel adds in K order.
struct Piece {
    int t;          // tile index (batch-major, as raster() takes it)
    int kb0, kb1;   // K blocks [kb0, kb1)
    int slot;       // -1: the whole tile, stored to C; else its partial tile
};

__device__ __forceinline__ int piece_count(const Tf32x3Params &p, int c, int G) {
    const int ndp = c < p.tiles_dp ? (p.tiles_dp - 1 - c) / G + 1 : 0;
    return ndp + (c < p.split * p.tail ? 1 : 0);
}

__device__ __forceinline__ Piece piece_of(const Tf32x3Params &p, int c, int G, int kblocks,
                                          int i) {
    Piece pc;
    const int ndp = c < p.tiles_dp ? (p.tiles_dp - 1 - c) / G + 1 : 0;
    if (i < ndp) {
        pc.t = c + i * G;
        pc.kb0 = 0;
        pc.kb1 = kblocks;
        pc.slot = -1;
        return pc;
    }
    const int j = c / p.tail, tl = c - j * p.tail;
    pc.t = p.tiles_dp + tl;
    pc.kb0 = (int)((long long)j * kblocks / p.split);
    pc.kb1 = (int)(((long long)j + 1) * kblocks / p.split);
    pc.slot = c;
    return pc;
}

// Adds the `split` partial tiles of every tail tile and stores the sums to C
// with the epilogue: grid (BM * BN / (1024 * V), tail) x 256 threads, V
// float4 per thread 1024 floats apart (each load and store instruction
// coalesced across the warp).  A thread reads 8 / V segments at a time,
// every load of such a batch issued before its adds, so a long split costs
// split * V / 8 round trips; the adds go in K order starting from zero.  The
// launcher takes V = 4 when that still gives a CTA per SM, else V = 1.
// Launched as a programmatic dependent of the GEMM kernel.
template <int BN, int V>
__global__ void __launch_bounds__(256) tf32x3_fixup_kernel(const Tf32x3Params p) {
    constexpr int NB = 8 / V;   // segments per batch
    static_assert((BM * BN) % (1024 * V) == 0, "whole float4 groups per CTA");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int tl = blockIdx.y;
    const int e0 = (blockIdx.x * 256 * V + threadIdx.x) * 4;   // element of the BM x BN tile
    const long long seg = (long long)p.tail * (BM * BN);        // floats between segments
    const float *base = p.part + (long long)tl * (BM * BN) + e0;
    float4 acc[V];
#pragma unroll
    for (int r = 0; r < V; ++r) acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j0 = 0; j0 < p.split; j0 += NB) {
        float4 v[NB][V];
#pragma unroll
        for (int b = 0; b < NB; ++b)
            if (j0 + b < p.split) {
#pragma unroll
                for (int r = 0; r < V; ++r)
                    v[b][r] = *reinterpret_cast<const float4 *>(base + (j0 + b) * seg + 1024 * r);
            }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if (j0 + b < p.split) {
#pragma unroll
                for (int r = 0; r < V; ++r) {
                    acc[r].x += v[b][r].x;
                    acc[r].y += v[b][r].y;
                    acc[r].z += v[b][r].z;
                    acc[r].w += v[b][r].w;
                }
            }
        }
    }
    int z, tm, tn;
    raster(p, p.tiles_dp + tl, z, tm, tn);
    const bool plain = p.alpha == 1.f && p.beta == 0.f && p.bias == nullptr;
#pragma unroll
    for (int r = 0; r < V; ++r) {
        const int e = e0 + 1024 * r;
        const int row = tm * BM + e / BN, col = tn * BN + e % BN;
        if (row >= p.M || col >= p.N) continue;
        float *cp = p.C + (int64_t)z * p.strideC + (int64_t)row * p.ldc + col;
        float o[4] = {acc[r].x, acc[r].y, acc[r].z, acc[r].w};
        if (!plain) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (col + j >= p.N) break;
                const float old = p.beta != 0.f ? cp[j] : 0.f;
                const float b = p.bias != nullptr ? p.bias[col + j] : 0.f;
                o[j] = fmaf(p.beta, old, p.alpha * o[j]) + b;
            }
        }
        if (p.vec_c && col + 3 < p.N) {
            *reinterpret_cast<float4 *>(cp) = make_float4(o[0], o[1], o[2], o[3]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (col + j < p.N) cp[j] = o[j];
        }
    }
}

// One CTA per SM walks its pieces (piece_of: whole tiles blockIdx.x,
// blockIdx.x + gridDim.x, ..., then at most one K segment of a tail tile).  A piece's K
// blocks split into chunks at the multiples of the chunk length (kcb blocks),
// so a piece that starts or ends inside a chunk has a shorter first or last
// chunk; the CTA's chunks are counted across pieces (gc) and chunk gc goes to
// accumulator gc % 2, and its K blocks are counted across pieces (g) for the
// ring.  Barriers: a ring stage's j-th fill is waited on with
// parity j & 1 and its (j-1)-th release with parity (j-1) & 1 (as in the
// persistent kernel); accumulator s's u-th chunk ("chunk full", one
// tcgen05.commit) with parity u & 1 and its (u-1)-th drain ("chunk free", one
// arrival per epilogue warp) with parity (u-1) & 1.  Every wait is bounded
// and the abort word stops all roles.  RAW as in the persistent kernel (no
// converter warps: chunking applies to K > 256, where operands come from lo
// planes).
template <class CFG, int RAW>
__global__ void __launch_bounds__(Chunked<CFG>::THREADS, 1)
tf32x3_chunked_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmAlo,
                      const __grid_constant__ CUtensorMap tmBlo,
                      const __grid_constant__ CUtensorMap tmC,
                      const __grid_constant__ CUtensorMap tmP, const Tf32x3Params p) {
    using P = Chunked<CFG>;
    constexpr int BK = CFG::BK, STAGES = CFG::STAGES, PLANES = CFG::PLANES;
    constexpr int BN = CFG::BN;
    constexpr int A_TILE = CFG::A_TILE, B_TILE = CFG::B_TILE, STAGE_BYTES = CFG::STAGE_BYTES;
    constexpr int NSLOT = P::NSLOT, COLS = P::COLS;
    const int KCB = p.kcb;   // K blocks per chunk
    constexpr int TX_BYTES = PLANES * (A_TILE + B_TILE);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_addr = tc::smem_u32_generic(smem_raw);
    const uint32_t pad = (1024 - (raw_addr & 1023)) & 1023;
    uint8_t *smem = smem_raw + pad;
    const uint32_t ring = tc::smem_u32_generic(smem);
    const uint32_t staging = ring + STAGES * STAGE_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES + P::STAGING);
    const uint32_t full0 = tc::smem_u32_generic(bars);
    const uint32_t empty0 = full0 + 8 * STAGES;
    const uint32_t chf0 = empty0 + 8 * STAGES;     // chunk accumulator s holds a finished chunk
    const uint32_t che0 = chf0 + 8 * NSLOT;        // chunk accumulator s has been drained
    const uint32_t done_bar = che0 + 8 * NSLOT;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + P::BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kblocks = (p.K + BK - 1) / BK;
    const int cta = (int)blockIdx.x, G = (int)gridDim.x;
    const int npieces = piece_count(p, cta, G);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            tc::mbar_init(full0 + 8 * s, 1);
            tc::mbar_init(empty0 + 8 * s, 1);
        }
        for (int s = 0; s < NSLOT; ++s) {
            tc::mbar_init(chf0 + 8 * s, 1);
            tc::mbar_init(che0 + 8 * s, P::EPI_WARPS);
        }
        tc::mbar_init(done_bar, 1);
        *abort_flag = 0;
        tc::fence_barrier_init();
        tc::tma_prefetch_desc(&tmA);
        tc::tma_prefetch_desc(&tmB);
        if constexpr ((RAW & 1) != 0) tc::tma_prefetch_desc(&tmAlo);
        if constexpr ((RAW & 2) != 0) tc::tma_prefetch_desc(&tmBlo);
    }
    if (warp == 1) tc::tmem_alloc(tc::smem_u32_generic(tmem_slot), 512);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // a programmatic dependent of the split kernel: no global access before
    // its planes are complete and visible
    asm volatile("griddepcontrol.wait;" ::: "memory");

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (the ring runs on across tiles)
            long long issued = 0;
            long long g = 0;   // the CTA's K blocks so far
            bool stop = false;
            for (int i = 0; i < npieces && !stop; ++i) {
                const Piece pc = piece_of(p, cta, G, kblocks, i);
                int z, tm, tn;
                raster(p, pc.t, z, tm, tn);
                const int m0 = tm * BM, n0 = tn * BN;
                for (int kb = pc.kb0; kb < pc.kb1; ++kb, ++g) {
                    const int s = (int)(g % STAGES);
                    const int j = (int)(g / STAGES);
                    if (g >= STAGES && !tc::mbar_wait(empty0 + 8 * s, (j & 1) ^ 1, abort_flag)) {
                        stop = true;
                        break;
                    }
                    if (*abort_flag) {
                        stop = true;
                        break;
                    }
                    const uint32_t st = ring + s * STAGE_BYTES;
                    const uint32_t fb = full0 + 8 * s;
                    tc::mbar_arrive_expect_tx(fb, TX_BYTES);
                    const int k0 = kb * BK;
                    if constexpr (RAW & 1) {
                        tc::tma_load_3d(st, &tmA, fb, k0, m0, z);
                        tc::tma_load_3d(st + A_TILE, &tmAlo, fb, k0, m0, z);
                    } else {
#pragma unroll
                        for (int pl = 0; pl < PLANES; ++pl)
                            tc::tma_load_3d(st + pl * A_TILE, &tmA, fb, k0, m0, PLANES * z + pl);
                    }
                    if constexpr (RAW & 2) {
                        tc::tma_load_3d(st + PLANES * A_TILE, &tmB, fb, k0, n0, z);
                        tc::tma_load_3d(st + PLANES * A_TILE + B_TILE, &tmBlo, fb, k0, n0, z);
                    } else {
#pragma unroll
                        for (int pl = 0; pl < PLANES; ++pl)
                            tc::tma_load_3d(st + PLANES * A_TILE + pl * B_TILE, &tmB, fb, k0, n0,
                                            PLANES * z + pl);
                    }
                    issued = g + 1;
                }
            }
            if (*abort_flag) {
                // the latest fill of every stage lands before the CTA exits
                for (long long f = (issued > STAGES ? issued - STAGES : 0); f < issued; ++f) {
                    const int s = (int)(f % STAGES);
                    const long long t0 = clock64();
                    while (!tc::mbar_try_wait(full0 + 8 * s, (int)((f / STAGES) & 1)) &&
                           clock64() - t0 < tc::kWaitLimitCycles) {
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            constexpr uint32_t idesc = tc::tf32_idesc<BM, BN>();
            bool stop = false;
            long long gc = 0;   // the CTA's chunk counter
            long long g = 0;    // the CTA's K blocks so far
            for (int i = 0; i < npieces && !stop; ++i) {
                const Piece pc = piece_of(p, cta, G, kblocks, i);
                for (int c = pc.kb0 / KCB; c <= (pc.kb1 - 1) / KCB; ++c, ++gc) {
                    const int sl = (int)(gc % NSLOT);
                    const long long u = gc / NSLOT;
                    if (gc >= NSLOT && !tc::mbar_wait(che0 + 8 * sl, (int)((u - 1) & 1), abort_flag)) {
                        stop = true;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t acc = tmem + (uint32_t)(sl * P::SLOT_COLS);
                    const int kb0 = max(pc.kb0, c * KCB);
                    const int kb1 = min(pc.kb1, (c + 1) * KCB);
                    for (int kb = kb0; kb < kb1; ++kb, ++g) {
                        const int s = (int)(g % STAGES);
                        if (!tc::mbar_wait(full0 + 8 * s, (int)((g / STAGES) & 1), abort_flag)) {
                            stop = true;
                            break;
                        }
                        tc::fence_after_sync();
                        const uint32_t st = ring + s * STAGE_BYTES;
                        const uint64_t ahi = tc::kmajor_desc<CFG::ROW_BYTES>(st);
                        const uint64_t alo = tc::kmajor_desc<CFG::ROW_BYTES>(st + A_TILE);
                        const uint64_t bhi = tc::kmajor_desc<CFG::ROW_BYTES>(st + 2 * A_TILE);
                        const uint64_t blo =
                            tc::kmajor_desc<CFG::ROW_BYTES>(st + 2 * A_TILE + B_TILE);
#pragma unroll
                        for (int kk = 0; kk < BK / 8; ++kk) {
                            const uint64_t step = (uint64_t)(kk * 32) >> 4;
                            const uint32_t first = (kb == kb0 && kk == 0) ? 0u : 1u;
                            if constexpr (P::SEP) {
                                tc::mma_tf32(acc + BN, alo + step, bhi + step, idesc, first);
                                tc::mma_tf32(acc + BN, ahi + step, blo + step, idesc, 1u);
                                tc::mma_tf32(acc, ahi + step, bhi + step, idesc, first);
                            } else {
                                tc::mma_tf32(acc, alo + step, bhi + step, idesc, first);
                                tc::mma_tf32(acc, ahi + step, blo + step, idesc, 1u);
                                tc::mma_tf32(acc, ahi + step, bhi + step, idesc, 1u);
                            }
                        }
                        tc::mma_commit(empty0 + 8 * s);
                    }
                    if (stop) break;
                    tc::mma_commit(chf0 + 8 * sl);
                }
            }
            tc::mma_commit(done_bar);   // tracks every MMA issued above, also on abort
        }
    } else {
        // ---------------- epilogue warps 2-9: lane quarter warp % 4, column half
        const int q = warp & 3;
        const int h = (warp - 2) >> 2;
        const uint32_t stage = staging + (uint32_t)(warp - 2) * 4096u;
        const uint32_t lane_off = ((uint32_t)(32 * q) << 16) + (uint32_t)(h * COLS);
        int cc = 0;
        long long gc = 0;
        bool stop = false;
        for (int i = 0; i < npieces && !stop; ++i) {
            const Piece pc = piece_of(p, cta, G, kblocks, i);
            float run[COLS];
#pragma unroll
            for (int j = 0; j < COLS; ++j) run[j] = 0.f;
            for (int c = pc.kb0 / KCB; c <= (pc.kb1 - 1) / KCB; ++c, ++gc) {
                const int sl = (int)(gc % NSLOT);
                const long long u = gc / NSLOT;
                const bool ok = tc::mbar_wait(chf0 + 8 * sl, (int)(u & 1), abort_flag);
                __syncwarp();
                // one warp-uniform decision: the TMEM loads are warp-collective
                if (!__all_sync(0xffffffffu, ok && !*abort_flag)) {
                    stop = true;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t base = tmem + (uint32_t)(sl * P::SLOT_COLS) + lane_off;
#pragma unroll
                for (int b = 0; b < COLS / 16; ++b) {
                    float v[16];
                    tc::tmem_ld_16(base + 16 * b, v);
                    if constexpr (P::SEP) {
                        float w[16];
                        tc::tmem_ld_16(base + BN + 16 * b, w);
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] += w[j];
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) run[16 * b + j] += v[j];
                }
                tc::fence_before_sync();   // the TMEM loads above precede the release
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(che0 + 8 * sl);
            }
            if (stop) break;
            // a whole tile to C, a segment's sum to its partial tile (whole)
            int z, tm, tn;
            raster(p, pc.t, z, tm, tn);
            const bool part = pc.slot >= 0;
            store_running_rows<COLS>(p, part ? &tmP : &tmC, part || p.tma_c,
                                     part ? INT_MAX : p.tma_n, run, q, lane,
                                     part ? pc.slot : z, part ? 0 : tm * BM,
                                     (part ? 0 : tn * BN) + h * COLS, part ? BM : p.M,
                                     part ? BN : p.N, stage, cc);
        }
        // the stores' global writes are done before the CTA ends (the fix-up
        // kernel reads the partial tiles)
        if (lane == 0 && cc > 0) tc::bulk_wait_group<0>();
    }
    __syncwarp();

    tc::fence_before_sync();
    __syncthreads();
    // after every role has finished, so a wait that ran out late is reported too
    if (*abort_flag && threadIdx.x == 0) atomicOr(&g_tf32x3_error, 1u);
    if (warp == 1) {
        // every MMA issued has completed before TMEM is freed
        int local_abort = 0;
        (void)tc::mbar_wait(done_bar, 0, &local_abort);
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ self-test

// Exercises the failure path of the pipeline waits: one CTA waits, with the
// same bounded wait the GEMM kernel uses, on an mbarrier that nothing ever
// arrives on.  The wait gives up after `limit` cycles, the CTA raises the
// library's device status word and exits normally.
__global__ void wait_timeout_selftest_kernel(long long limit) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_word;
    const uint32_t b = tc::smem_u32_generic(&bar);
    if (threadIdx.x == 0) {
        tc::mbar_init(b, 1);
        abort_word = 0;
        tc::fence_barrier_init();
    }
    __syncthreads();
    const bool ok = tc::mbar_wait(b, 0, &abort_word, limit);
    __syncthreads();
    if (threadIdx.x == 0 && (!ok || abort_word)) atomicOr(&g_tf32x3_error, 1u);
}

// ------------------------------------------------------------------ TF32 probe

// Tensor-pipe throughput probe for kind::tf32: every CTA (one per SM) issues
// `iters` rounds of four M128 N256 K8 MMAs on operand tiles that stay in
// shared memory (128-byte swizzle, as the GEMM's 32-float slices), all
// accumulating into one 256-column TMEM accumulator; no global traffic.  The
// single issuing thread is held back by the MMA queue, not by a spin.  The
// completion wait is bounded; if it runs out the CTA raises the status word
// and waits once more before freeing TMEM.
constexpr int kProbeA = BM * 128;          // 128 rows x 32 fp32
constexpr int kProbeB = 256 * 128;         // 256 rows x 32 fp32
constexpr int kProbeSmem = kProbeA + kProbeB + 1024 + 64;

__global__ void __launch_bounds__(THREADS, 1) tf32_mma_probe_kernel(long long iters, float *out) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw_addr = tc::smem_u32_generic(smem_raw);
    const uint32_t pad = (1024 - (raw_addr & 1023)) & 1023;
    uint8_t *smem = smem_raw + pad;
    float *ops = reinterpret_cast<float *>(smem);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kProbeA + kProbeB);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 1);
    const uint32_t bar_addr = tc::smem_u32_generic(bar);
    const int warp = threadIdx.x >> 5;

    // small TF32 values (low 13 bits zero), so the accumulator stays finite
    for (int i = threadIdx.x; i < (kProbeA + kProbeB) / 4; i += blockDim.x)
        ops[i] = (float)((i * 7) % 17 - 8) * 0.0078125f;
    if (threadIdx.x == 0) {
        tc::mbar_init(bar_addr, 1);
        tc::fence_barrier_init();
    }
    if (warp == 1) tc::tmem_alloc(tc::smem_u32_generic(tmem_slot), 256);
    // the operand tiles were written by the generic proxy; the MMAs read them
    // through the async proxy
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t base = tc::smem_u32_generic(smem);

    if (warp == 1 && (threadIdx.x & 31) == 0) {
        constexpr uint32_t idesc = tc::tf32_idesc<BM, 256>();
        const uint64_t adesc = tc::kmajor_desc<128>(base);
        const uint64_t bdesc = tc::kmajor_desc<128>(base + kProbeA);
        for (long long it = 0; it < iters; ++it) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t step = (uint64_t)(kk * 32) >> 4;
                tc::mma_tf32(tmem, adesc + step, bdesc + step, idesc, (it | kk) ? 1u : 0u);
            }
        }
        tc::mma_commit(bar_addr);
    }
    __syncwarp();
    // every thread waits for the MMAs (bounded); nothing sets an abort word here
    int never = 0;
    bool done = tc::mbar_wait(bar_addr, 0, &never);
    if (!done) {
        if (threadIdx.x == 0) atomicOr(&g_tf32x3_error, 1u);
        never = 0;
        done = tc::mbar_wait(bar_addr, 0, &never);
    }
    tc::fence_after_sync();
    if (warp == 0 && __all_sync(0xffffffffu, done)) {
        float v[32];
        tc::tmem_ld_32(tmem, v);   // lanes 0-31, columns 0-31
        if ((threadIdx.x & 31) == 0) out[blockIdx.x] = v[0];
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 256);
    }
}

// ------------------------------------------------------------------ host side

// Planes [planes*batch][rows][Kp] of fp32, box BK (K) x box_rows x 1, with
// the swizzle whose span equals the BK-float row.
template <class CFG>
bool make_plane_map(CUtensorMap *map, const float *base, int rows, int K, int Kp, int batch,
                    int box_rows, int planes = CFG::PLANES) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)(planes * batch)};
    const cuuint64_t strides[2] = {(cuuint64_t)Kp * 4, (cuuint64_t)rows * Kp * 4};
    const cuuint32_t box[3] = {(cuuint32_t)CFG::BK, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapSwizzle sw = CFG::ROW_BYTES == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : CFG::ROW_BYTES == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                         : CU_TENSOR_MAP_SWIZZLE_32B;
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The caller's K-contiguous operand as [batch][rows][K] fp32 (row stride ld,
// batch stride zstride), box BK x box_rows x 1 in the planes' swizzle: the
// raw slice lands where the hi plane would.  False when the driver rejects
// the description (the operand is then split as usual).
template <class CFG>
bool make_raw_map(CUtensorMap *map, const float *base, int rows, int K, int64_t ld,
                  int64_t zstride, int batch, int box_rows) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const int64_t zs = batch > 1 ? zstride : ld * (int64_t)rows;
    if (zs <= 0) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)batch};
    const cuuint64_t strides[2] = {(cuuint64_t)ld * 4, (cuuint64_t)zs * 4};
    const cuuint32_t box[3] = {(cuuint32_t)CFG::BK, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapSwizzle sw = CFG::ROW_BYTES == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : CFG::ROW_BYTES == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                         : CU_TENSOR_MAP_SWIZZLE_32B;
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// C as a [batch][M][N] tensor (row stride ldc, batch stride strideC), box
// 32 x 32 x 1 with the 128-byte swizzle the epilogue writes in.
bool make_c_map(CUtensorMap *map, float *C, int M, int N, int64_t ldc, int64_t strideC,
                int batch) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)N, (cuuint64_t)M, (cuuint64_t)batch};
    const int64_t zstride = batch > 1 ? strideC : (int64_t)M * ldc;
    const cuuint64_t strides[2] = {(cuuint64_t)ldc * 4, (cuuint64_t)zstride * 4};
    const cuuint32_t box[3] = {32, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, C, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The partial tiles as a [slots][BM][bn] tensor, box 32 x 32 x 1 with the
// 128-byte swizzle the epilogue stages in.
bool make_part_map(CUtensorMap *map, float *part, int slots, int bn) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)bn, (cuuint64_t)BM, (cuuint64_t)slots};
    const cuuint64_t strides[2] = {(cuuint64_t)bn * 4, (cuuint64_t)BM * bn * 4};
    const cuuint32_t box[3] = {32, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, part, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Floats per row of a TF32 plane: K rounded up to 32, so every row starts on
// a 128-byte boundary.  TMA moves a K slice of a row as one 64- or 128-byte
// piece; on rows only 16-byte aligned (K rounded up to 4) each piece straddled
// 32-byte sectors, and 3000 x 2000 x 1500 ran at 142 TFLOP/s against 163 with
// 128-byte rows.
int64_t plane_row_floats(int64_t K) { return (K + 31) / 32 * 32; }

size_t plane_bytes(int64_t rows, int64_t K, int64_t batch, int planes) {
    const size_t Kp = (size_t)plane_row_floats(K);
    return align_up((size_t)planes * (size_t)batch * (size_t)rows * Kp * 4, 256);
}

// Encodes the tensor maps, launches the split kernel into `ws` for the
// operands that need planes and fills the GEMM kernel's parameters.  `raw`
// and `conv` (bits as in Persist) mark operands the GEMM loads as they are
// (their maps are already in tmA / tmB) and those converted in the stage;
// a raw operand that is not converted gets a lo-only plane and its map in
// tmAlo / tmBlo (which are left empty otherwise).
template <class CFG>
cudaError_t prepare(const GemmArgs &a, bool transA, bool transB, int raw, int conv, void *ws,
                    cudaStream_t s, CUtensorMap &tmA, CUtensorMap &tmB, CUtensorMap &tmAlo,
                    CUtensorMap &tmBlo, CUtensorMap &tmC, Tf32x3Params &p) {
    constexpr int PLANES = CFG::PLANES;
    const int Kp = plane_row_floats(a.K);
    float *wsA = static_cast<float *>(ws);
    float *wsB = wsA + plane_bytes(a.M, a.K, a.batch, PLANES) / 4;
    const int lo_only = raw & ~conv;

    // tensor maps first (they depend only on the workspace and the sizes), so
    // no host work separates the split launch from the GEMM launch
    tmAlo = CUtensorMap{};
    tmBlo = CUtensorMap{};
    if ((!(raw & 1) && !make_plane_map<CFG>(&tmA, wsA, a.M, a.K, Kp, a.batch, BM)) ||
        (!(raw & 2) && !make_plane_map<CFG>(&tmB, wsB, a.N, a.K, Kp, a.batch, CFG::BN)) ||
        ((lo_only & 1) && !make_plane_map<CFG>(&tmAlo, wsA, a.M, a.K, Kp, a.batch, BM, 1)) ||
        ((lo_only & 2) && !make_plane_map<CFG>(&tmBlo, wsB, a.N, a.K, Kp, a.batch, CFG::BN, 1)))
        return cudaErrorInvalidValue;

    // stage 1: split op(A) (rows M) and op(B) (rows N) into K-major TF32 planes,
    // one launch for both; a converted operand gets no CTAs, a raw one only
    // its lo plane
    SplitArgs sa;
    sa.K = a.K;
    sa.Kp = Kp;
    sa.batch = a.batch;
    auto job = [&](SplitJob &j, const float *X, int64_t ld, int64_t sX, int R, bool kcontig,
                   float *out, bool skip, bool lo) {
        j.X = X;
        j.ld = ld;
        j.sX = sX;
        j.out = out;
        j.R = R;
        j.kcontig = kcontig;
        j.lo_only = lo;
        j.vec = (reinterpret_cast<uintptr_t>(X) % 16 == 0) && ld % 4 == 0 &&
                (a.batch == 1 || sX % 4 == 0);
        const int64_t work =
            kcontig ? ((int64_t)a.batch * R * (Kp / 4) + 255) / 256
                    : (int64_t)a.batch * ((R + (j.vec ? 127 : 31)) / (j.vec ? 128 : 32)) *
                          ((a.K + 31) / 32);
        j.blocks = skip ? 0 : (work < 152 * 16 ? (work > 0 ? work : 1) : 152 * 16);
    };
    job(sa.job[0], a.A, a.lda, a.strideA, a.M, !transA, wsA, (conv & 1) != 0, (lo_only & 1) != 0);
    job(sa.job[1], a.B, a.ldb, a.strideB, a.N, transB, wsB, (conv & 2) != 0, (lo_only & 2) != 0);
    const int64_t split_blocks = sa.job[0].blocks + sa.job[1].blocks;
    if (split_blocks > 0) {
        split_kernel<PLANES><<<(unsigned)split_blocks, 256, 0, s>>>(sa);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }

    p.C = a.C;
    p.ldc = a.ldc;
    p.strideC = a.strideC;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.batch = a.batch;
    p.tiles_m = (a.M + BM - 1) / BM;
    p.tiles_n = (a.N + CFG::BN - 1) / CFG::BN;
    p.group_m = a.group_m;
    p.vec_c = (reinterpret_cast<uintptr_t>(a.C) % 16 == 0) && a.ldc % 4 == 0 && a.strideC % 4 == 0;
    p.alpha = a.alpha;
    p.beta = a.beta;
    p.bias = a.bias;
    p.kcb = 1;
    p.tiles_dp = a.batch * p.tiles_m * p.tiles_n;
    p.tail = 0;
    p.split = 0;
    p.part = nullptr;
    // The TMA store takes the plain product into a C whose base, rows and
    // batches are 16-byte aligned.  A store was seen to write whole 16-byte
    // granules: with N not a multiple of 4 it wrote the padding column next
    // to column N-1.  So the map is N rounded down to a multiple of 4 wide,
    // and the 32-column block holding the last columns of such a width is
    // stored by the threads themselves (tma_n).  The map is only read when
    // tma_c is set.
    tmC = CUtensorMap{};
    const int n4 = a.N / 4 * 4;
    p.tma_c = p.vec_c && n4 > 0 && plain_epilogue(a) &&
              make_c_map(&tmC, a.C, a.M, n4, a.ldc, a.strideC, a.batch);
    p.tma_n = a.N % 4 == 0 ? INT_MAX : n4;
    return cudaSuccess;
}

// Sets the opt-in dynamic shared-memory size of `kern` once per context.
template <typename Kern>
cudaError_t ensure_smem(Kern kern, int bytes, PerContext<bool> &configured) {
    const unsigned long long ctx = current_context_id();
    bool done = false;
    if (configured.get(ctx, done)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    configured.put(current_context_id(), true);
    return cudaSuccess;
}

// One CTA per SM, walking the tiles (see tf32x3_persistent_kernel).
template <class CFG, int ACC_BUFS, int RAW, int CONV>
cudaError_t launch_persistent_raw(const GemmArgs &a, bool transA, bool transB, void *ws,
                                  cudaStream_t s, CUtensorMap &tmA, CUtensorMap &tmB) {
    using P = Persist<CFG, ACC_BUFS, RAW, CONV>;
    static PerContext<bool> configured;
    cudaError_t e = ensure_smem(tf32x3_persistent_kernel<CFG, ACC_BUFS, RAW, CONV>, P::SMEM_BYTES,
                                configured);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    CUtensorMap tmC, tmAlo, tmBlo;
    Tf32x3Params p;
    e = prepare<CFG>(a, transA, transB, RAW, CONV, ws, s, tmA, tmB, tmAlo, tmBlo, tmC, p);
    if (e != cudaSuccess) return e;
    const long long tiles = (long long)a.batch * p.tiles_m * p.tiles_n;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(tiles < sms ? tiles : sms));
    cfg.blockDim = dim3(P::THREADS);
    cfg.dynamicSmemBytes = P::SMEM_BYTES;
    cfg.stream = s;
    // a programmatic dependent of the split launch (or, with no split, of
    // whatever precedes): every global access waits on griddepcontrol.wait
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, tf32x3_persistent_kernel<CFG, ACC_BUFS, RAW, CONV>, tmA, tmB,
                           tmAlo, tmBlo, tmC, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Operands stored K-contiguous (row-major A, B stored transposed) with
// 16-byte aligned rows and batches are loaded as they are.  With three terms
// the caller's rows are the hi term and the lo term comes either from
// converter warps inside the GEMM or from a lo-only plane the split kernel
// writes (half the split's output for that operand).  With one term the
// operand is rounded in the stage where it would be converted (below), else
// split.  Everything else goes through the split kernel's full planes.
//
// Converting in the GEMM saves the split's HBM round trip of that operand
// but adds shared-memory traffic and a step to every stage of a ring that is
// already latency-bound, and each operand panel is converted once per tile
// that reads it (A once per tile column, B once per tile row).  Measured
// (results bit-identical either way), three terms, lo plane -> converted:
//   96 x 512 x 512 x K (4 x 4 tiles): K = 96 NT 84.0 -> 104.1, K = 256 NN
//   103.6 -> 115.2, NT 112.5 -> 138.3 TFLOP/s;
//   24 x 1024 x 1024 x 128 (8 x 8 tiles): NN 108.1 -> 113.9;
//   4096 x 4096 x 128 (32 x 32): NN 119.9 -> 112.3, NT 119.3 -> 105.2;
//   3072^3: NN 257.8 -> 244.5, NT 271.4 -> 195.5.
// So an operand is converted when K <= kRawMaxK, or when K <= kConvMaxK and
// at most kConvMaxReuse tiles read each of its panels (for three terms on
// the 128-wide tile, which every K <= 256 takes).  The one-term product
// gains the same way: 96 x 512 x 512 x 256 NT 160.3 -> 217.1, K = 128 NT
// 121.1 -> 159.2, 24 x 1024 x 1024 x 128 NN 142.1 -> 151.5; 4096 x 4096 x 128
// and 3072^3 unchanged.
constexpr int kRawMaxK = 64;
constexpr int kConvMaxK = 256;
constexpr int kConvMaxReuse = 8;
// Longer three-term reductions take the K-chunked kernel.
constexpr int kChunkMinK = 256;

// Launches with the runtime choice `conv` (a subset of RAW) of converted
// operands; a combination the configuration does not provide launches
// nothing and returns an error (the caller never asks for one).
template <class CFG, int ACC_BUFS, int RAW>
cudaError_t launch_conv(const GemmArgs &a, bool transA, bool transB, void *ws, cudaStream_t s,
                        CUtensorMap &tmA, CUtensorMap &tmB, int conv) {
    if constexpr (CFG::PLANES == 1) {
        // one term: an operand is raw only when it is rounded in the stage
        if (conv == RAW)
            return launch_persistent_raw<CFG, ACC_BUFS, RAW, RAW>(a, transA, transB, ws, s, tmA, tmB);
    } else if constexpr (CFG::BN == 128) {
        switch (conv) {
            case 0:
                return launch_persistent_raw<CFG, ACC_BUFS, RAW, 0>(a, transA, transB, ws, s, tmA, tmB);
            case 1:
                if constexpr ((RAW & 1) != 0)
                    return launch_persistent_raw<CFG, ACC_BUFS, RAW, 1>(a, transA, transB, ws, s, tmA,
                                                                        tmB);
                break;
            case 2:
                if constexpr ((RAW & 2) != 0)
                    return launch_persistent_raw<CFG, ACC_BUFS, RAW, 2>(a, transA, transB, ws, s, tmA,
                                                                        tmB);
                break;
            case 3:
                if constexpr (RAW == 3)
                    return launch_persistent_raw<CFG, ACC_BUFS, 3, 3>(a, transA, transB, ws, s, tmA, tmB);
                break;
            default:
                break;
        }
    } else {
        // the 256-wide three-term tile (K > 256 only): lo planes, no converters
        if (conv == 0)
            return launch_persistent_raw<CFG, ACC_BUFS, RAW, 0>(a, transA, transB, ws, s, tmA, tmB);
    }
    return cudaErrorInvalidValue;
}

template <class CFG, int ACC_BUFS>
cudaError_t launch_persistent(const GemmArgs &a, bool transA, bool transB, void *ws,
                              cudaStream_t s) {
    const int64_t tiles_m = (a.M + BM - 1) / BM, tiles_n = (a.N + CFG::BN - 1) / CFG::BN;
    // converting an operand whose panels `reuse` tiles read
    auto convert = [&](int64_t reuse) {
        return a.K <= kRawMaxK || (a.K <= kConvMaxK && reuse <= kConvMaxReuse);
    };
    // one term: raw only when converted (rounded in the stage)
    auto raw_ok = [&](const float *X, int64_t ld, int64_t sX, bool kcontig, int64_t reuse) {
        return (CFG::PLANES == 2 || convert(reuse)) && kcontig &&
               reinterpret_cast<uintptr_t>(X) % 16 == 0 && ld % 4 == 0 &&
               (a.batch == 1 || (sX > 0 && sX % 4 == 0));
    };
    CUtensorMap tmA, tmB;
    int raw = 0;
    if (raw_ok(a.A, a.lda, a.strideA, !transA, tiles_n) &&
        make_raw_map<CFG>(&tmA, a.A, a.M, a.K, a.lda, a.strideA, a.batch, BM))
        raw |= 1;
    if (raw_ok(a.B, a.ldb, a.strideB, transB, tiles_m) &&
        make_raw_map<CFG>(&tmB, a.B, a.N, a.K, a.ldb, a.strideB, a.batch, CFG::BN))
        raw |= 2;
    int conv = 0;
    if (CFG::PLANES == 1) {
        conv = raw;
    } else if (CFG::BN == 128) {
        if ((raw & 1) && convert(tiles_n)) conv |= 1;
        if ((raw & 2) && convert(tiles_m)) conv |= 2;
    }
    switch (raw) {
        case 1: return launch_conv<CFG, ACC_BUFS, 1>(a, transA, transB, ws, s, tmA, tmB, conv);
        case 2: return launch_conv<CFG, ACC_BUFS, 2>(a, transA, transB, ws, s, tmA, tmB, conv);
        case 3: return launch_conv<CFG, ACC_BUFS, 3>(a, transA, transB, ws, s, tmA, tmB, conv);
        default: return launch_persistent_raw<CFG, ACC_BUFS, 0, 0>(a, transA, transB, ws, s, tmA, tmB);
    }
}

// The K-chunked kernel for three terms over K > kChunkMinK: one CTA per SM.
// An operand stored K-contiguous with 16-byte aligned rows is loaded raw as
// its own hi term with a lo-only plane from the split kernel; other operands
// get hi and lo planes.
// The K-chunked kernel's schedule for `tiles` output tiles BN wide of
// `kblocks` K blocks on `sms` SMs, one CTA per SM (see piece_of): whole waves
// of tiles, then the tail split into G / tail K segments when that is at
// least two, each segment at least two K blocks; the segments' partial
// tiles take split * tail * BM * BN floats of workspace.
struct ChunkedPlan {
    int G, tiles_dp, tail, split;
    size_t part_bytes;
};

ChunkedPlan chunked_plan(long long tiles, int kblocks, int bn, int sms) {
    ChunkedPlan pl = {};
    pl.G = (int)(tiles < sms ? tiles : sms);
    pl.tiles_dp = (int)tiles;
    const long long tail = tiles % sms;
    if (sms < 2 || tail == 0) return pl;
    int split = (int)(sms / tail);
    if (split > kblocks / 2) split = kblocks / 2;
    if (split < 2) return pl;
    pl.G = sms;
    pl.tiles_dp = (int)(tiles - tail);
    pl.tail = (int)tail;
    pl.split = split;
    pl.part_bytes = (size_t)split * (size_t)tail * BM * (size_t)bn * sizeof(float);
    return pl;
}

template <class CFG>
ChunkedPlan chunked_plan_for(const GemmArgs &a, int sms) {
    const long long tiles =
        (long long)a.batch * ((a.M + BM - 1) / BM) * ((a.N + CFG::BN - 1) / CFG::BN);
    return chunked_plan(tiles, (a.K + CFG::BK - 1) / CFG::BK, CFG::BN, sms);
}

template <class CFG, int RAW>
cudaError_t launch_chunked_raw(const GemmArgs &a, bool transA, bool transB, void *ws,
                               size_t ws_bytes, cudaStream_t s, CUtensorMap &tmA,
                               CUtensorMap &tmB) {
    using P = Chunked<CFG>;
    static PerContext<bool> configured;
    cudaError_t e = ensure_smem(tf32x3_chunked_kernel<CFG, RAW>, P::SMEM_BYTES, configured);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    CUtensorMap tmC, tmAlo, tmBlo;
    Tf32x3Params p;
    e = prepare<CFG>(a, transA, transB, RAW, 0, ws, s, tmA, tmB, tmAlo, tmBlo, tmC, p);
    if (e != cudaSuccess) return e;
    p.kcb = g_chunk_k.load(std::memory_order_relaxed) / CFG::BK;
    // the partial tiles follow the planes; a workspace without room for them
    // keeps the whole-tile schedule
    const size_t planes = plane_bytes(a.M, a.K, a.batch, 2) + plane_bytes(a.N, a.K, a.batch, 2);
    ChunkedPlan pl = chunked_plan_for<CFG>(a, sms);
    if (pl.split > 0 && ws_bytes >= planes + pl.part_bytes) {
        p.tiles_dp = pl.tiles_dp;
        p.tail = pl.tail;
        p.split = pl.split;
        p.part = reinterpret_cast<float *>(static_cast<char *>(ws) + planes);
    } else {
        const long long tiles = (long long)a.batch * p.tiles_m * p.tiles_n;
        pl.G = (int)(tiles < sms ? tiles : sms);
        pl.split = 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.G);
    cfg.blockDim = dim3(P::THREADS);
    cfg.dynamicSmemBytes = P::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    CUtensorMap tmP = {};
    if (pl.split > 0 && !make_part_map(&tmP, p.part, pl.split * pl.tail, CFG::BN))
        return cudaErrorInvalidValue;
    e = cudaLaunchKernelEx(&cfg, tf32x3_chunked_kernel<CFG, RAW>, tmA, tmB, tmAlo, tmBlo, tmC, tmP,
                           p);
    if (e != cudaSuccess) return e;
    if (pl.split == 0) return cudaGetLastError();
    // the tail tiles' sums, as a programmatic dependent of the GEMM
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    if ((long long)pl.tail * (BM * CFG::BN / 4096) >= sms) {
        cfg.gridDim = dim3((unsigned)(BM * CFG::BN / 4096), (unsigned)pl.tail);
        e = cudaLaunchKernelEx(&cfg, tf32x3_fixup_kernel<CFG::BN, 4>, p);
    } else {
        cfg.gridDim = dim3((unsigned)(BM * CFG::BN / 1024), (unsigned)pl.tail);
        e = cudaLaunchKernelEx(&cfg, tf32x3_fixup_kernel<CFG::BN, 1>, p);
    }
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// An operand is read raw only when its rows start on 128-byte boundaries
// (base and leading dimension): a K slice of a row is then whole 32-byte
// sectors, as in the planes (plane_row_floats).  On rows only 16-byte aligned
// each slice straddles sectors, and the split kernel's planes are the cheaper
// route (3000 x 2000 x 1500 with row-major A of ld 1500).
template <class CFG>
cudaError_t launch_chunked(const GemmArgs &a, bool transA, bool transB, void *ws, size_t ws_bytes,
                           cudaStream_t s) {
    static_assert(CFG::PLANES == 2, "three terms");
    auto raw_ok = [&](const float *X, int64_t ld, int64_t sX, bool kcontig) {
        return kcontig && reinterpret_cast<uintptr_t>(X) % 128 == 0 && ld % 32 == 0 &&
               (a.batch == 1 || (sX > 0 && sX % 32 == 0));
    };
    CUtensorMap tmA, tmB;
    int raw = 0;
    if (raw_ok(a.A, a.lda, a.strideA, !transA) &&
        make_raw_map<CFG>(&tmA, a.A, a.M, a.K, a.lda, a.strideA, a.batch, BM))
        raw |= 1;
    if (raw_ok(a.B, a.ldb, a.strideB, transB) &&
        make_raw_map<CFG>(&tmB, a.B, a.N, a.K, a.ldb, a.strideB, a.batch, CFG::BN))
        raw |= 2;
    switch (raw) {
        case 1: return launch_chunked_raw<CFG, 1>(a, transA, transB, ws, ws_bytes, s, tmA, tmB);
        case 2: return launch_chunked_raw<CFG, 2>(a, transA, transB, ws, ws_bytes, s, tmA, tmB);
        case 3: return launch_chunked_raw<CFG, 3>(a, transA, transB, ws, ws_bytes, s, tmA, tmB);
        default: return launch_chunked_raw<CFG, 0>(a, transA, transB, ws, ws_bytes, s, tmA, tmB);
    }
}

}  // namespace tf32x3

// Tuned configurations (K slice, stages, terms, tile width) and accumulator
// buffers.  The ring is latency-bound, so what counts is the bytes in flight:
// for the 128 x 256 three-term tile, 4 stages of 48 KB (64-byte swizzle) beat 2
// stages of 96 KB by 13-16 %; the 128 x 128 tile does best with 32-float slices.
using Tf32x3Wide = tf32x3::Config<16, 4, 3, 256>;     // one accumulator buffer (512 columns)
using Tf32x3Narrow = tf32x3::Config<32, 3, 3, 128>;   // two buffers of 256 columns
using Tf32Wide = tf32x3::Config<32, 4, 1, 256>;       // two buffers of 256 columns
using Tf32Narrow = tf32x3::Config<32, 6, 1, 128>;     // two buffers of 128 columns

namespace {

// Tile width.  Plain TF32 (the persistent kernel): a 128 x 256 tile costs
// about 1.75 128 x 128 tiles (8192 x 8192 x 4096, where the wave tail is
// negligible); count tiles per SM and take the cheaper tiling, the wide one
// on ties.  Three terms: a short K (at most 256) takes the narrow tile
// whatever the count: only it has two accumulator buffers, and with few K
// steps per tile the overlapped epilogue matters most (96 x 512 x 512 x 64:
// 54.8 us narrow, 61.0 us wide).  A longer K runs the K-chunked kernel,
// costed in microseconds by chunked_cost_us: a 128 x 128 tile takes about
// 0.019 us per unit of K on one SM and a 128 x 256 tile 1.5 times that
// (8192 x 8192 x 4096: 287 TFLOP/s wide, 220 narrow); a tail split in K
// costs 1 / split of a tile plus writing and reading back its partial tiles
// at about 20 TB/s (they stay in L2).  Fitted to the whole call on GB300 with
// each width forced: 2049 x 3071 x 1537 takes a wave of wide tiles and a
// tail in halves (183 TFLOP/s; three waves of narrow ones, 151), 700 x 900 x
// 300 takes 48 narrow tiles in 3 segments (21.3; 24 wide in 6, 19.5), and
// 512 x 512 x 4096 8 wide tiles in 19 (72.6; 16 narrow in 9, 68.8).
double chunked_cost_us(long long tiles, int K, int kblocks, int bn, int sms) {
    const tf32x3::ChunkedPlan pl = tf32x3::chunked_plan(tiles, kblocks, bn, sms);
    const double tile_us = 0.019 * K * (bn == 256 ? 1.5 : 1.0);
    const double waves = (double)(tiles / sms);
    if (pl.split > 0) return (waves + 1.0 / pl.split) * tile_us + 2.0 * pl.part_bytes / 20e6;
    return (waves + (tiles % sms != 0 ? 1.0 : 0.0)) * tile_us;
}

bool tc_wide_tile(const GemmArgs &a, int terms) {
    if (terms == 3 && a.K <= 256) return false;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        sms = 1;
    const long long tm = (a.M + tf32x3::BM - 1) / tf32x3::BM;
    const long long wide = (long long)a.batch * tm * ((a.N + 255) / 256);
    const long long narrow = (long long)a.batch * tm * ((a.N + 127) / 128);
    if (terms == 3)
        return chunked_cost_us(wide, a.K, (a.K + Tf32x3Wide::BK - 1) / Tf32x3Wide::BK, 256, sms) <=
               chunked_cost_us(narrow, a.K, (a.K + Tf32x3Narrow::BK - 1) / Tf32x3Narrow::BK, 128,
                               sms);
    const double cost_wide = 1.75 * (double)((wide + sms - 1) / sms);
    const double cost_narrow = (double)((narrow + sms - 1) / sms);
    return cost_wide <= cost_narrow;
}

}  // namespace

size_t tf32x3_workspace_min_bytes(int64_t M, int64_t N, int64_t K, int64_t batch) {
    return tf32x3::plane_bytes(M, K, batch, 2) + tf32x3::plane_bytes(N, K, batch, 2);
}

// The planes, then (K-chunked kernel whose tail tiles are split in K on this
// device) the segments' partial tiles.
size_t tf32x3_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t batch) {
    const size_t planes = tf32x3_workspace_min_bytes(M, N, K, batch);
    if (K <= tf32x3::kChunkMinK || M <= 0 || N <= 0 || batch <= 0) return planes;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return planes;
    GemmArgs a = {};
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.batch = (int)batch;
    const tf32x3::ChunkedPlan pl = tc_wide_tile(a, 3) ? tf32x3::chunked_plan_for<Tf32x3Wide>(a, sms)
                                                      : tf32x3::chunked_plan_for<Tf32x3Narrow>(a, sms);
    return planes + pl.part_bytes;
}

size_t tf32_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t batch) {
    return tf32x3::plane_bytes(M, K, batch, 1) + tf32x3::plane_bytes(N, K, batch, 1);
}

// Three terms: reductions up to kChunkMinK run the single-pass persistent
// kernel (128-wide tiles, converter warps where they pay); longer ones the
// K-chunked kernel, whose sums are promoted to round-to-nearest fp32 adds
// every 128 of K, on the tile width the wave count favours.
cudaError_t launch_tf32x3(const GemmArgs &a, bool transA, bool transB, void *ws, size_t ws_bytes,
                          cudaStream_t s) {
    if (a.K <= tf32x3::kChunkMinK)
        return tf32x3::launch_persistent<Tf32x3Narrow, 2>(a, transA, transB, ws, s);
    return tc_wide_tile(a, 3)
               ? tf32x3::launch_chunked<Tf32x3Wide>(a, transA, transB, ws, ws_bytes, s)
               : tf32x3::launch_chunked<Tf32x3Narrow>(a, transA, transB, ws, ws_bytes, s);
}

cudaError_t launch_tf32(const GemmArgs &a, bool transA, bool transB, void *ws, cudaStream_t s) {
    return tc_wide_tile(a, 1) ? tf32x3::launch_persistent<Tf32Wide, 2>(a, transA, transB, ws, s)
                              : tf32x3::launch_persistent<Tf32Narrow, 2>(a, transA, transB, ws, s);
}

int set_tf32x3_chunk_k(int chunk_k) {
    if (chunk_k == 0) chunk_k = tf32x3::kChunkK;
    if (chunk_k < tf32x3::kChunkStep || chunk_k > (1 << 30) || chunk_k % tf32x3::kChunkStep != 0)
        return -1;
    return tf32x3::g_chunk_k.exchange(chunk_k);
}

cudaError_t launch_tf32_mma_probe(long long iters, float *out, int ctas, cudaStream_t s) {
    static PerContext<bool> configured;
    cudaError_t e = tf32x3::ensure_smem(tf32x3::tf32_mma_probe_kernel, tf32x3::kProbeSmem,
                                        configured);
    if (e != cudaSuccess) return e;
    tf32x3::tf32_mma_probe_kernel<<<ctas, tf32x3::THREADS, tf32x3::kProbeSmem, s>>>(iters, out);
    return cudaGetLastError();
}

double tf32_mma_probe_flops_per_iteration() { return 4.0 * 2.0 * tf32x3::BM * 256 * 8; }

cudaError_t launch_wait_timeout_selftest(long long limit_cycles, cudaStream_t s) {
    tf32x3::wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(limit_cycles);
    return cudaGetLastError();
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (get_current == nullptr || get_id == nullptr) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// The status word's device address in the current context: looked up in each
// context once (the lookup also makes the runtime set up a context that is
// not yet current), so a kernel never gets an address from another context.
unsigned int *device_error_word() {
    static PerContext<unsigned int *> cached;
    unsigned int *w = nullptr;
    if (cached.get(current_context_id(), w)) return w;
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, tf32x3::g_tf32x3_error) != cudaSuccess) return nullptr;
    w = static_cast<unsigned int *>(p);
    cached.put(current_context_id(), w);
    return w;
}

cudaError_t tf32x3_read_error(unsigned int *flags, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(flags, tf32x3::g_tf32x3_error, sizeof(unsigned int));
    if (e != cudaSuccess || !reset) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(tf32x3::g_tf32x3_error, &zero, sizeof(unsigned int));
}

}  // namespace sgemm
