// SIMT FP32 SGEMM fed by TMA, for row-major B with A either stored
// transposed (K x M, contiguous along M) or row-major (contiguous along K),
// and for both operands stored transposed: a K slice of either operand is
// then a plain 2-D box of global memory.
//
// Same arithmetic as sgemm_simt_kernel (each output accumulated by one thread
// in ascending k with packed fp32 FMAs, 8 x 8 register tile of 4 x 4
// sub-blocks, Z-order warps; "CUDA GEMM operator performance optimization",
// sections 4-8), so results are bit-identical to it.  What changes is the
// operand pipeline (sections 9-10 of that page, with Hopper-and-later bulk
// copies in place of per-thread loads):
//   * one thread issues each stage as two cp.async.bulk.tensor loads (an A
//     box of 128 x 32 and a B box of 128 x 32) that complete on the stage's
//     "full" mbarrier; nobody else computes a global address;
//   * no CTA-wide barrier in the main loop: each warp, done with a stage,
//     arrives on the stage's "empty" mbarrier, and only the issuing thread
//     waits for all eight arrivals before it refills the stage, so warps
//     drift apart by up to a stage instead of meeting every 32 k steps;
//   * B boxes and M-contiguous A boxes land K-major ([32][128]) with no
//     swizzle: a warp's fragment loads touch 4 (A) and 8 (B) consecutive
//     16-byte chunks of one row, so they are conflict-free as they are;
//   * a K-contiguous (row-major) A box lands M-major ([128][32], one 128-byte
//     row per m) with the 128-byte swizzle (16-byte chunk c of row m stored
//     at c ^ (m % 8)).  Instead of a corner turn, each thread owns rows
//     ty + 16 j (j = 0..7) and reads 4 consecutive k of a row with one
//     16-byte load; all of a thread's rows share m % 8 = ty % 8, and the 4
//     row groups of a warp land in 4 different chunks: conflict-free, and as
//     many loads per k step as the K-major layout;
//   * a K-contiguous B (stored transposed, with A stored transposed) lands
//     the same way, [128][32] per n, each thread owning columns tx + 16 j;
//     its packed FMAs pair outputs along m (see slice_fma);
//   * the tensor map zero-fills rows, columns and K beyond the operand, so
//     ragged tiles need no per-element predicates;
//   * without per-thread copy state the kernel fits 128 registers: two CTAs
//     (16 warps) per SM, 4 warps per scheduler to hide the FMA and
//     shared-load latencies.  The cp.async kernel needs 8 x 16 tiles and one
//     CTA per SM to avoid spilling.
// Three kernels:
//   * sgemm_simt_tma_kernel: one tile per CTA (sgemm_f32; strided batches
//     are the third tensor dimension);
//   * sgemm_simt_persist_tma_kernel: the same tiles walked by one CTA per
//     resident slot, the loads running ahead across tile boundaries (short
//     reductions with A stored transposed);
//   * sgemm_simt_streamk_tma_kernel: the stream-K schedule
//     (sgemm_f32_streamk) as one grid, whole waves of tiles one per CTA,
//     then one CTA per stream-K range.
// Every mbarrier wait is bounded; once one runs out the CTA waits no more,
// except for the issuing thread's own copies in flight (again bounded), and
// bit 0 of the library's device status word is raised.
#include <atomic>
#include <cstdint>

#include "simt_launch.cuh"
#include "tc_utils.cuh"
#include "tma_encode.h"

namespace sgemm {
namespace simt {

constexpr int kTmaBK = 32;       // K slice per stage
constexpr int kTmaStages = 3;    // 3 x 32 KB of operands per CTA
constexpr int kTmaBN = 128;      // tile 128 x 128
constexpr int kTmaMinBlocks = 2;
constexpr int kPersistMaxSlices = 8;   // K <= 256: the persistent form (see below)

template <int BK, int STAGES, int BN_>
constexpr int tma_smem_bytes() {
    // 1 KB to align the ring to the 1024-byte swizzle atom, the operand ring,
    // then STAGES "full" and STAGES "empty" mbarriers, the CTA's abort word and
    // the slice last issued into each stage
    return 1024 + STAGES * BK * (BM + BN_) * (int)sizeof(float) + 16 * STAGES +
           (4 + 4 * STAGES + 15) / 16 * 16;
}

// The operand ring starts at the first 1024-byte boundary of the dynamic
// shared memory (the 128-byte swizzle pattern repeats every 8 rows of 128
// bytes and is laid out relative to such a boundary).
__device__ __forceinline__ float *align_ring(float *raw) {
    const uint32_t a = smem_u32(raw);
    return raw + ((1024u - (a & 1023u)) & 1023u) / sizeof(float);
}

// Initialises the stage barriers and the abort word: "full" barriers take one
// arrival (the issuing thread's expect_tx) plus the stage's bytes, "empty"
// barriers one arrival per warp.  Returns the shared address of full barrier
// 0; the empty barriers follow the full ones.
template <int BK, int STAGES, int BN_>
__device__ __forceinline__ uint32_t tma_pipeline_init(float *smem, volatile int *&abort) {
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * BK * (BM + BN_));
    abort = reinterpret_cast<volatile int *>(bars + 2 * STAGES);
    const uint32_t full0 = smem_u32(bars);
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) tc::mbar_init(full0 + 8 * s, 1);
        for (int s = 0; s < STAGES; ++s) tc::mbar_init(full0 + 8 * (STAGES + s), THREADS / 32);
        abort[0] = 0;
        for (int s = 0; s < STAGES; ++s) abort[1 + s] = -1;   // nothing issued (last_issued)
        tc::fence_barrier_init();
    }
    __syncthreads();
    return full0;
}

// The slice whose copies the issuing thread last started into stage `st`
// (the words after the abort word; 0xffffffff: none yet).
__device__ __forceinline__ volatile uint32_t &last_issued(volatile int *abort, uint32_t st) {
    return *reinterpret_cast<volatile uint32_t *>(abort + 1 + st);
}

// One K slice of the tile from a landed stage (A part `at`, B part `bt`):
// acc[i][j] += a[i] * b[j] for its BK k steps, k ascending.  A fragments come
// K-major (4 + 4 rows per 16-byte load) or, with KA, from the M-major swizzled
// stage (4 k of a row per 16-byte load).  B fragments come K-major (4 + 4
// columns per 16-byte load) or, with KB, from the N-major swizzled stage (4 k
// of a column per 16-byte load).  A packed FMA takes one operand pair from
// adjacent registers and the other as one value twice: pairs run along n
// (b[j], b[j+1] from one K-major float4) unless B comes N-major, whose 8
// values of a k step sit in 8 different registers; then pairs run along m
// (a[i], a[i+1] from one K-major float4).  Moving values into pairs costs
// about a third of the throughput, so both operands M/N-major (A row-major
// with B stored transposed) is not a form of this kernel.
template <int BK, int BN_, bool KA, bool KB>
__device__ __forceinline__ void slice_fma(const float *at, const float *bt, int a_col, int b_col,
                                          float (&acc)[8][BN_ / 16]) {
    constexpr int TN = BN_ / 16;
    static_assert(!(KA && KB), "no packed-FMA pairs when both operands come M/N-major");
    static_assert(!KB || BN_ == 128, "N-major B fragments assume 128-column tiles");
    static_assert(!(KA || KB) || BK == 32, "the 128-byte swizzle spans one 32-float row");
    auto fma8 = [&](const float (&a)[8], const float (&b)[TN]) {
        if constexpr (KB) {   // pairs along m, b[j] twice
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                const float2 bj = make_float2(b[j], b[j]);
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    float2 c = make_float2(acc[i][j], acc[i + 1][j]);
                    c = __ffma2_rn(make_float2(a[i], a[i + 1]), bj, c);
                    acc[i][j] = c.x;
                    acc[i + 1][j] = c.y;
                }
            }
        } else {              // pairs along n, a[i] twice
            // column pair outer, rows inner: the pair operand stays the same
            // for 8 consecutive FMAs and the broadcast one changes (measured:
            // 3072^3 A^T by B 65.5 -> 68.8 TFLOP/s one tile per CTA, the
            // stream-K step 66.5 -> 68.9, 96 x 512^2 x 64 persistent 48.7 ->
            // 51.9; the rows-outer order of the cp.async kernels stays, it
            // lost 14 % there).  Every output still takes its k in order.
#pragma unroll
            for (int j = 0; j < TN; j += 2) {
                const float2 bj = make_float2(b[j], b[j + 1]);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float2 c = make_float2(acc[i][j], acc[i][j + 1]);
                    c = __ffma2_rn(make_float2(a[i], a[i]), bj, c);
                    acc[i][j] = c.x;
                    acc[i][j + 1] = c.y;
                }
            }
        }
    };
    // fragments of k step kk from a K-major stage: columns col..col+3, +64, ...
    auto a_kmajor = [&](int kk, float (&a)[8]) {
        const float *ar = at + kk * BM;
        const float4 a0 = *reinterpret_cast<const float4 *>(ar + a_col);
        const float4 a1 = *reinterpret_cast<const float4 *>(ar + 64 + a_col);
        a[0] = a0.x; a[1] = a0.y; a[2] = a0.z; a[3] = a0.w;
        a[4] = a1.x; a[5] = a1.y; a[6] = a1.z; a[7] = a1.w;
    };
    auto b_kmajor = [&](int kk, float (&b)[TN]) {
        const float *br = bt + kk * BN_;
#pragma unroll
        for (int h = 0; h < BN_ / 64; ++h) {
            const float4 bv = *reinterpret_cast<const float4 *>(br + 64 * h + b_col);
            b[4 * h + 0] = bv.x;
            b[4 * h + 1] = bv.y;
            b[4 * h + 2] = bv.z;
            b[4 * h + 3] = bv.w;
        }
    };
    if constexpr (KA || KB) {
        // rows ty + 16 j (columns tx + 16 j) of the [128][32] swizzled stage:
        // they share ty % 8 (tx % 8), hence the 16-byte chunk of k quad kq;
        // four k per load, the other operand K-major one k at a time
        const int t = KA ? a_col >> 2 : b_col >> 2;
        const float *qrow = (KA ? at : bt) + t * BK;
#pragma unroll
        for (int kq = 0; kq < BK / 4; ++kq) {
            float4 qv[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                qv[j] = *reinterpret_cast<const float4 *>(qrow + j * 16 * BK + 4 * (kq ^ (t & 7)));
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float q[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    q[j] = e == 0 ? qv[j].x : e == 1 ? qv[j].y : e == 2 ? qv[j].z : qv[j].w;
                if constexpr (KA) {
                    float b[TN];
                    b_kmajor(4 * kq + e, b);
                    fma8(q, b);
                } else {
                    float a[8];
                    a_kmajor(4 * kq + e, a);
                    fma8(a, q);
                }
            }
        }
    } else {
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[8], b[TN];
            a_kmajor(kk, a);
            b_kmajor(kk, b);
            fma8(a, b);
        }
    }
}

// Accumulates slices [0, ktiles) of one piece, starting at K offset kbeg, of
// the tile at (m0, n0) of problem z into acc (zeroed first).  gk counts the
// slices this CTA has consumed before the piece: slice g lives in stage
// g % STAGES during its round g / STAGES, so the phase parity of the stage's
// barriers is (g / STAGES) & 1.  Every thread keeps the same count.
// Thread 0 issues slice g only after every warp has released slice
// g - STAGES from the same stage; each warp releases a slice once its lanes
// have read it.  On return no copy of this piece is in flight (every issued
// slice has been waited on), and the next piece may start at once.
// The issuing thread records the slice it last started into each stage in
// the words after the abort word (last_issued), so finish_abort knows which
// copies can still be in flight.  A stage is refilled only after all eight
// warps released it, and a warp does not release it once the abort word is
// set (a wait that gave up sets the word before the warp gets to its release,
// so every release in an aborted run follows a copy that landed), so a stage
// never gets a second
// fill in one phase, also after an abort; after an abort a slice may be
// skipped while a later one whose stage was already released still goes out,
// hence a record per stage.  The records live in shared memory, not in
// registers held across the loop.
// GUARD_FLAG picks how a warp decides to skip its release after an abort:
// by reading the abort word at the release (false) or by keeping its own
// wait's result (true).  Both are exact; they differ only in the registers
// the compiler gives the loop, and every kernel now runs fastest with its own
// wait's result (3072^3, CUDA events, against the word: stream-K step 68.9 ->
// 69.2 TFLOP/s, A^T by B 68.7 -> 69.0, both transposed 59.5 -> 60.5, row-major
// A 60.2 against 58.9).
template <int BK, int STAGES, int BN_, bool KA, bool KB, bool GUARD_FLAG>
__device__ __forceinline__ void tma_mainloop(const CUtensorMap *tmA, const CUtensorMap *tmB,
                                             float *As, float *Bs, uint32_t full0, uint32_t &gk,
                                             int m0, int n0, int z, int kbeg, int ktiles,
                                             int a_col, int b_col, float (&acc)[8][BN_ / 16],
                                             volatile int *abort) {
    constexpr int TN = BN_ / 16;
    constexpr int ATILE = BK * BM;
    constexpr int BTILE = BK * BN_;
    constexpr uint32_t STAGE_BYTES = (ATILE + BTILE) * sizeof(float);
    const uint32_t empty0 = full0 + 8 * STAGES;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

    const bool issuer = threadIdx.x == 0;
    const uint32_t g0 = gk;          // the piece's slice j is the CTA's slice g0 + j
    auto issue = [&](int slice) {
        const uint32_t g = g0 + (uint32_t)slice;
        const uint32_t st = g % STAGES;
        // slice g - STAGES released by every warp.  No warp releases a stage
        // after the abort word is set, so a completed release means the
        // stage holds no copy in flight; once the word is set the wait gives
        // up instead of waiting for releases that will not come.
        if (g >= STAGES && !tc::mbar_wait(empty0 + 8 * st, ((g / STAGES) - 1) & 1, abort)) return;
        last_issued(abort, st) = g;
        const uint32_t bar = full0 + 8 * st;
        tc::mbar_arrive_expect_tx(bar, STAGE_BYTES);
        if constexpr (KA)   // box (k, m): 32 k x 128 rows
            tc::tma_load_3d(smem_u32(As + st * ATILE), tmA, bar, kbeg + slice * BK, m0, z);
        else                // box (m, k): 128 m x 32 k
            tc::tma_load_3d(smem_u32(As + st * ATILE), tmA, bar, m0, kbeg + slice * BK, z);
        if constexpr (KB)   // box (k, n): 32 k x 128 columns
            tc::tma_load_3d(smem_u32(Bs + st * BTILE), tmB, bar, kbeg + slice * BK, n0, z);
        else                // box (n, k): 128 n x 32 k
            tc::tma_load_3d(smem_u32(Bs + st * BTILE), tmB, bar, n0, kbeg + slice * BK, z);
    };
    if (issuer) {
#pragma unroll
        for (int s = 0; s < STAGES - 1; ++s)
            if (s < ktiles) issue(s);
    }
    for (int kt = 0; kt < ktiles; ++kt) {
        const uint32_t rs = gk % STAGES;
        const bool landed = tc::mbar_wait(full0 + 8 * rs, (gk / STAGES) & 1, abort);
        ++gk;
        slice_fma<BK, BN_, KA, KB>(As + rs * ATILE, Bs + rs * BTILE, a_col, b_col, acc);
        // the warp's lanes have all read the stage: release it, unless the
        // abort word is set (a wait that gave up sets it first, and its copy
        // may still be in flight)
        __syncwarp();
        if ((threadIdx.x & 31) == 0 && (GUARD_FLAG ? landed : !*abort))
            tc::mbar_arrive(empty0 + 8 * rs);
        if (issuer && kt + STAGES - 1 < ktiles) issue(kt + STAGES - 1);
    }
}

// After a wait ran out (the abort word is set; every later wait returned at
// once, and no stage was refilled unless its last copy had landed), thread 0
// raises bit 0 of the status word and waits, with a limit, for the latest
// copy it issued into each stage to land, so that none writes into shared
// memory after the CTA has exited.  Does nothing in a run whose waits all
// completed.
template <int STAGES>
__device__ __forceinline__ void finish_abort(uint32_t full0, volatile int *abort,
                                             unsigned int *status) {
    if (threadIdx.x != 0 || !*abort) return;
    if (status != nullptr) atomicOr(status, 1u);
    for (uint32_t st = 0; st < STAGES; ++st) {
        const uint32_t g = last_issued(abort, st);
        if (g == 0xffffffffu) continue;
        const long long t0 = clock64();
        while (!tc::mbar_try_wait(full0 + 8 * st, (g / STAGES) & 1) &&
               clock64() - t0 < tc::kWaitLimitCycles) {
        }
    }
}

// The thread's place in the tile: rows a_col..a_col+3 and +64, columns
// b_col..b_col+3 and +64 (Z-order 4 x 8 warps, 2 warps across).
__device__ __forceinline__ void thread_coords(int &a_col, int &b_col) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int lane_row = (lane & 1) | ((lane >> 4) << 1);
    const int lane_col = (lane >> 1) & 7;
    a_col = 4 * ((warp >> 1) * 4 + lane_row);
    b_col = 4 * ((warp & 1) * 8 + lane_col);
}

// Tile row of accumulator row r: a_col + r and 64 + a_col + r - 4 when A
// fragments come K-major, ty + 16 r (ty = a_col / 4) when they come M-major.
template <bool KA>
__device__ __forceinline__ int acc_row(int a_col, int r) {
    if constexpr (KA) return (a_col >> 2) + 16 * r;
    return r < 4 ? a_col + r : 64 + a_col + (r - 4);
}

// Stores the thread's outputs with the epilogue.  Columns b_col..b_col+3
// (and +64) go out as 16-byte stores; with KB the thread's columns are
// tx + 16 j (tx = b_col / 4), stored one by one with the same arithmetic as
// store_c4, a warp writing 32 consecutive bytes of each of its rows per j.
template <int BN_, bool KA, bool KB = false>
__device__ __forceinline__ void store_tile(const GemmArgs &p, int z, int m0, int n0, int a_col,
                                           int b_col, const float (&acc)[8][BN_ / 16]) {
    constexpr int NSB = BN_ / 64;
    float *Cz = p.C + (int64_t)z * p.strideC;
    const bool plain = plain_epilogue(p);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int row = m0 + acc_row<KA>(a_col, r);
        if (row >= p.M) continue;
        float *crow = Cz + (int64_t)row * p.ldc;
        if constexpr (KB) {
            const int tx = b_col >> 2;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int col = n0 + tx + 16 * j;
                if (col >= p.N) continue;
                float v = acc[r][j];
                if (!plain) {
                    const float o = p.beta != 0.f ? crow[col] : 0.f;
                    const float b = p.bias != nullptr ? p.bias[col] : 0.f;
                    v = fmaf(p.beta, o, p.alpha * v) + b;
                }
                crow[col] = v;
            }
        } else {
#pragma unroll
            for (int h = 0; h < NSB; ++h)
                store_c4(p, crow, n0 + h * 64 + b_col,
                         make_float4(acc[r][4 * h], acc[r][4 * h + 1], acc[r][4 * h + 2],
                                     acc[r][4 * h + 3]),
                         true, plain);
        }
    }
}

// One 128 x BN_ tile per CTA, all of K.
template <int BK, int STAGES, int BN_, bool KA, bool KB, int MINB>
__global__ void __launch_bounds__(THREADS, MINB)
sgemm_simt_tma_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB, const GemmArgs p,
                      unsigned int *status) {
    extern __shared__ __align__(128) float smem_raw[];
    float *smem = align_ring(smem_raw);
    float *As = smem;
    float *Bs = smem + STAGES * BK * BM;
    volatile int *abort;
    const uint32_t full0 = tma_pipeline_init<BK, STAGES, BN_>(smem, abort);
    if (threadIdx.x == 0) {
        tc::tma_prefetch_desc(&tmA);
        tc::tma_prefetch_desc(&tmB);
    }
    // launched as a programmatic dependent (of the transpose that turned an
    // operand, say): the set-up above overlaps its tail; memory after this
    pdl_wait();
    pdl_trigger();
    int z, tm, tn;
    raster(p, (int)blockIdx.x, z, tm, tn);
    int a_col, b_col;
    thread_coords(a_col, b_col);
    float acc[8][BN_ / 16];
    uint32_t gk = 0;
    tma_mainloop<BK, STAGES, BN_, KA, KB, true>(&tmA, &tmB, As, Bs, full0, gk, tm * BM, tn * BN_, z,
                                              0, (p.K + BK - 1) / BK, a_col, b_col, acc, abort);
    finish_abort<STAGES>(full0, abort, status);
    store_tile<BN_, KA, KB>(p, z, tm * BM, tn * BN_, a_col, b_col, acc);
}

// Persistent form for short reductions: CTA c of G walks tiles c, c + G, ...
// of the whole grid, all of K each.  Slice g of the CTA (tile g / ktiles,
// K slice g % ktiles) uses stage g % STAGES, and the issuing thread stays
// STAGES - 1 slices ahead across tile boundaries: the next tile's first
// slices are in flight while this tile's last ones compute and its results
// are stored.  With 2 K slices per tile (K = 64) a CTA of the plain kernel
// spends most of its life on set-up, the first load's latency and the store.
template <int BK, int STAGES, int BN_, bool KA, int MINB>
__global__ void __launch_bounds__(THREADS, MINB)
sgemm_simt_persist_tma_kernel(const __grid_constant__ CUtensorMap tmA,
                              const __grid_constant__ CUtensorMap tmB, const GemmArgs p,
                              unsigned int *status) {
    constexpr int ATILE = BK * BM;
    constexpr int BTILE = BK * BN_;
    constexpr uint32_t STAGE_BYTES = (ATILE + BTILE) * sizeof(float);
    extern __shared__ __align__(128) float smem_raw[];
    float *smem = align_ring(smem_raw);
    float *As = smem;
    float *Bs = smem + STAGES * BK * BM;
    volatile int *abort;
    const uint32_t full0 = tma_pipeline_init<BK, STAGES, BN_>(smem, abort);
    const uint32_t empty0 = full0 + 8 * STAGES;
    if (threadIdx.x == 0) {
        tc::tma_prefetch_desc(&tmA);
        tc::tma_prefetch_desc(&tmB);
    }
    pdl_wait();
    pdl_trigger();
    int a_col, b_col;
    thread_coords(a_col, b_col);
    const int c = blockIdx.x, G = gridDim.x;
    const int tiles = p.batch * p.tiles_m * p.tiles_n;
    const int mine = c < tiles ? (tiles - 1 - c) / G + 1 : 0;
    const int ktiles = (p.K + BK - 1) / BK;
    const int total = mine * ktiles;   // slices of this CTA
    const bool issuer = threadIdx.x == 0;
    auto issue = [&](int g) {
        const int i = g / ktiles, j = g - i * ktiles;
        int z, tm, tn;
        raster(p, c + i * G, z, tm, tn);
        const uint32_t st = (uint32_t)g % STAGES;
        // as in tma_mainloop: released stages hold no copy in flight
        if (g >= STAGES && !tc::mbar_wait(empty0 + 8 * st, ((uint32_t)g / STAGES - 1) & 1, abort))
            return;
        last_issued(abort, st) = (uint32_t)g;
        const uint32_t bar = full0 + 8 * st;
        tc::mbar_arrive_expect_tx(bar, STAGE_BYTES);
        if constexpr (KA)
            tc::tma_load_3d(smem_u32(As + st * ATILE), &tmA, bar, j * BK, tm * BM, z);
        else
            tc::tma_load_3d(smem_u32(As + st * ATILE), &tmA, bar, tm * BM, j * BK, z);
        tc::tma_load_3d(smem_u32(Bs + st * BTILE), &tmB, bar, tn * BN_, j * BK, z);
    };
    if (issuer)
        for (int g = 0; g < STAGES - 1 && g < total; ++g) issue(g);
    int g = 0;
#pragma unroll 1
    for (int i = 0; i < mine; ++i) {
        float acc[8][BN_ / 16];
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int q = 0; q < BN_ / 16; ++q) acc[r][q] = 0.f;
#pragma unroll 1
        for (int j = 0; j < ktiles; ++j, ++g) {
            const uint32_t rs = (uint32_t)g % STAGES;
            (void)tc::mbar_wait(full0 + 8 * rs, ((uint32_t)g / STAGES) & 1, abort);
            slice_fma<BK, BN_, KA, false>(As + rs * ATILE, Bs + rs * BTILE, a_col, b_col, acc);
            __syncwarp();
            if ((threadIdx.x & 31) == 0 && !*abort) tc::mbar_arrive(empty0 + 8 * rs);
            if (issuer && g + STAGES - 1 < total) issue(g + STAGES - 1);
        }
        int z, tm, tn;
        raster(p, c + i * G, z, tm, tn);
        store_tile<BN_, KA>(p, z, tm * BM, tn * BN_, a_col, b_col, acc);
    }
    finish_abort<STAGES>(full0, abort, status);
}

// The stream-K schedule (see StreamK) as one grid of tiles_dp + G CTAs:
// CTA b < tiles_dp computes tile b whole, like sgemm_simt_tma_kernel; CTA
// tiles_dp + c takes stream-K range c (units [c*U/G, (c+1)*U/G) of the
// remaining tiles' K slices, at most two pieces), so the whole-wave tiles
// run one per CTA and the ranges fill the last wave.  Pieces that are not a
// whole tile go to workspace slots [c][0|1] for streamk_fixup_kernel.
template <int BK, int STAGES, int BN_, bool KA, int MINB>
__global__ void __launch_bounds__(THREADS, MINB)
sgemm_simt_streamk_tma_kernel(const __grid_constant__ CUtensorMap tmA,
                              const __grid_constant__ CUtensorMap tmB, const GemmArgs p,
                              const StreamK sk, unsigned int *status) {
    constexpr int NSB = BN_ / 64;
    extern __shared__ __align__(128) float smem_raw[];
    float *smem = align_ring(smem_raw);
    float *As = smem;
    float *Bs = smem + STAGES * BK * BM;
    volatile int *abort;
    const uint32_t full0 = tma_pipeline_init<BK, STAGES, BN_>(smem, abort);
    if (threadIdx.x == 0) {
        tc::tma_prefetch_desc(&tmA);
        tc::tma_prefetch_desc(&tmB);
    }
    // launched as a programmatic dependent (of the transpose that turned an
    // operand, say): the set-up above overlaps its tail; memory after this
    pdl_wait();
    pdl_trigger();
    int a_col, b_col;
    thread_coords(a_col, b_col);
    uint32_t gk = 0;
    const int b = blockIdx.x;
    if (b < sk.tiles_dp) {
        int z, tm, tn;
        raster(p, b, z, tm, tn);
        float acc[8][BN_ / 16];
        tma_mainloop<BK, STAGES, BN_, KA, false, true>(&tmA, &tmB, As, Bs, full0, gk, tm * BM,
                                                        tn * BN_, z, 0, sk.kslices, a_col, b_col,
                                                        acc, abort);
        finish_abort<STAGES>(full0, abort, status);
        store_tile<BN_, KA>(p, z, tm * BM, tn * BN_, a_col, b_col, acc);
        return;
    }
    const int c = b - sk.tiles_dp;
    const int64_t u0 = (int64_t)c * sk.units / sk.G, u1 = ((int64_t)c + 1) * sk.units / sk.G;
    // tiles_sk < G, so a range is at most kslices units long: at most two pieces
    const int nsk = u0 == u1 ? 0 : (u0 / sk.kslices == (u1 - 1) / sk.kslices ? 1 : 2);
#pragma unroll 1
    // After a wait of the first piece ran out, the second piece issues no copy
    // (tma_mainloop issues nothing once the abort word is set) and its waits
    // return at once; skipping it explicitly cost registers in the main loop.
    for (int k = 0; k < nsk; ++k) {   // 0: the range's first piece, 1: its last
        const int64_t ub = k == 0 ? u0 : (u0 / sk.kslices + 1) * sk.kslices;
        const int tl = (int)(ub / sk.kslices);
        const int s0 = (int)(ub - (int64_t)tl * sk.kslices);
        const int s1 = (int)min((int64_t)sk.kslices, s0 + (u1 - ub));
        int z, tm, tn;
        raster(p, sk.tiles_dp + tl, z, tm, tn);
        float acc[8][BN_ / 16];
        tma_mainloop<BK, STAGES, BN_, KA, false, true>(&tmA, &tmB, As, Bs, full0, gk, tm * BM,
                                                        tn * BN_, z, s0 * BK, s1 - s0, a_col,
                                                        b_col, acc, abort);
        if (!(s0 == 0 && s1 == sk.kslices)) {
            // the whole 128 x BN_ block, unmasked: the workspace holds full tiles
            float *part = sk.ws + ((int64_t)c * 2 + k) * (BM * BN_);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int row = acc_row<KA>(a_col, r);
#pragma unroll
                for (int h = 0; h < NSB; ++h)
                    *reinterpret_cast<float4 *>(part + row * BN_ + h * 64 + b_col) =
                        make_float4(acc[r][4 * h], acc[r][4 * h + 1], acc[r][4 * h + 2],
                                    acc[r][4 * h + 3]);
            }
        } else {
            store_tile<BN_, KA>(p, z, tm * BM, tn * BN_, a_col, b_col, acc);
        }
    }
    finish_abort<STAGES>(full0, abort, status);
}

namespace {

// [batch][K][cols] fp32 with row stride ld and batch stride zstride (elements),
// boxes of box_cols x BK x 1, zero fill outside: an operand contiguous along
// M or N.  False when the driver rejects the description (the caller then
// uses the cp.async kernels).
bool make_operand_map(CUtensorMap *map, const float *base, int cols, int K, int64_t ld,
                      int64_t zstride, int batch, int box_cols) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const int64_t zs = batch > 1 ? zstride : ld * (int64_t)K;
    if (zs <= 0) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)K, (cuuint64_t)batch};
    const cuuint64_t strides[2] = {(cuuint64_t)ld * 4, (cuuint64_t)zs * 4};
    const cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)kTmaBK, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// [batch][rows][K] fp32 (contiguous along K) with row stride ld, boxes of
// BK x box_rows x 1 with the 128-byte swizzle (BK floats = 128 bytes).
bool make_kmajor_map(CUtensorMap *map, const float *base, int rows, int K, int64_t ld,
                     int64_t zstride, int batch, int box_rows) {
    auto fn = tensor_map_encoder();
    if (!fn) return false;
    const int64_t zs = batch > 1 ? zstride : ld * (int64_t)rows;
    if (zs <= 0) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)batch};
    const cuuint64_t strides[2] = {(cuuint64_t)ld * 4, (cuuint64_t)zs * 4};
    const cuuint32_t box[3] = {(cuuint32_t)kTmaBK, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_maps(const GemmArgs &a, bool ka, bool kb, CUtensorMap &tmA, CUtensorMap &tmB) {
    const bool okA = ka ? make_kmajor_map(&tmA, a.A, a.M, a.K, a.lda, a.strideA, a.batch, BM)
                        : make_operand_map(&tmA, a.A, a.M, a.K, a.lda, a.strideA, a.batch, BM);
    const bool okB = kb ? make_kmajor_map(&tmB, a.B, a.N, a.K, a.ldb, a.strideB, a.batch, kTmaBN)
                        : make_operand_map(&tmB, a.B, a.N, a.K, a.ldb, a.strideB, a.batch, kTmaBN);
    return okA && okB;
}

template <bool KA, bool KB>
cudaError_t launch_tile_kernel(const CUtensorMap &tmA, const CUtensorMap &tmB, const GemmArgs &g,
                               cudaStream_t s) {
    auto kern = sgemm_simt_tma_kernel<kTmaBK, kTmaStages, kTmaBN, KA, KB, kTmaMinBlocks>;
    constexpr int smem = tma_smem_bytes<kTmaBK, kTmaStages, kTmaBN>();
    static PerContext<bool> configured;
    cudaError_t err = ensure_smem_attribute(kern, smem, configured);
    if (err != cudaSuccess) return err;
    const long long blocks = (long long)g.batch * g.tiles_m * g.tiles_n;
    return launch_pdl(kern, dim3((unsigned)blocks), dim3(THREADS), smem, s, tmA, tmB, g,
                      device_error_word());
}

template <bool KA>
cudaError_t launch_persist_kernel(const CUtensorMap &tmA, const CUtensorMap &tmB,
                                  const GemmArgs &g, int ctas, cudaStream_t s) {
    auto kern = sgemm_simt_persist_tma_kernel<kTmaBK, kTmaStages, kTmaBN, KA, kTmaMinBlocks>;
    constexpr int smem = tma_smem_bytes<kTmaBK, kTmaStages, kTmaBN>();
    static PerContext<bool> configured;
    cudaError_t err = ensure_smem_attribute(kern, smem, configured);
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3((unsigned)ctas), dim3(THREADS), smem, s, tmA, tmB, g,
                      device_error_word());
}

template <bool KA>
cudaError_t launch_streamk_kernel(const CUtensorMap &tmA, const CUtensorMap &tmB,
                                  const GemmArgs &g, const StreamK &sk, cudaStream_t s) {
    auto kern = sgemm_simt_streamk_tma_kernel<kTmaBK, kTmaStages, kTmaBN, KA, kTmaMinBlocks>;
    constexpr int smem = tma_smem_bytes<kTmaBK, kTmaStages, kTmaBN>();
    static PerContext<bool> configured;
    cudaError_t err = ensure_smem_attribute(kern, smem, configured);
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3((unsigned)(sk.tiles_dp + sk.G)), dim3(THREADS), smem, s, tmA, tmB,
                      g, sk, device_error_word());
}

}  // namespace
}  // namespace simt

bool simt_tma_eligible(const GemmArgs &a, bool transA, bool transB, bool vec) {
    // 16-byte aligned bases and rows (vec), whole problems (no split-K
    // chunks), distinct batches (a zero batch stride is not a tensor stride);
    // any layout but row-major A with B stored transposed, which would leave
    // the packed FMAs no operand pair in adjacent registers (see slice_fma)
    return vec && (transA || !transB) && a.kchunk == 0 &&
           (a.batch == 1 || (a.strideA > 0 && a.strideB > 0));
}

int simt_tma_ctas_per_sm() {
    using namespace simt;
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
    int v = cached[dev & 63].load();
    if (v <= 0) {
        auto kern = sgemm_simt_streamk_tma_kernel<kTmaBK, kTmaStages, kTmaBN, false, kTmaMinBlocks>;
        constexpr int smem = tma_smem_bytes<kTmaBK, kTmaStages, kTmaBN>();
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, THREADS, smem) != cudaSuccess ||
            v <= 0) {
            (void)cudaGetLastError();
            v = 1;
        }
        cached[dev & 63].store(v);
    }
    return v;
}

bool launch_simt_tma(const GemmArgs &a, bool transA, bool transB, cudaStream_t s,
                     cudaError_t &err) {
    using namespace simt;
    CUtensorMap tmA, tmB;
    if (!make_maps(a, !transA, transB, tmA, tmB)) return false;
    GemmArgs g = a;
    g.tiles_m = (a.M + BM - 1) / BM;
    g.tiles_n = (a.N + kTmaBN - 1) / kTmaBN;
    // A stored transposed, short reductions over at least two waves of
    // resident CTAs: the persistent form, which prefetches across tile
    // boundaries (96 x 512 x 512 x 64: 42.3 -> 45.9 TFLOP/s; 48 x 1024^2 x 64:
    // 48.2 -> 52.0).  With row-major A it spills and gained nothing (96 x
    // 512^2 x 128: 50.2 -> 47.5), so that layout keeps one tile per CTA.
    const long long tiles = (long long)g.batch * g.tiles_m * g.tiles_n;
    const long long G = (long long)sm_count() * simt_tma_ctas_per_sm();
    if (transA && !transB && (a.K + kTmaBK - 1) / kTmaBK <= kPersistMaxSlices && tiles >= 2 * G) {
        err = launch_persist_kernel<false>(tmA, tmB, g, (int)G, s);
        return true;
    }
    if (transB)   // A stored transposed (see simt_tma_eligible)
        err = launch_tile_kernel<false, true>(tmA, tmB, g, s);
    else
        err = transA ? launch_tile_kernel<false, false>(tmA, tmB, g, s)
                     : launch_tile_kernel<true, false>(tmA, tmB, g, s);
    return true;
}

bool launch_simt_streamk_tma(const GemmArgs &a, bool transA, const StreamKPlan &pl, void *ws,
                             cudaStream_t s, cudaError_t &err) {
    using namespace simt;
    // the stream-K plan covers A stored transposed only (see streamk_plan)
    if (!transA) return false;
    CUtensorMap tmA, tmB;
    if (!make_maps(a, false, false, tmA, tmB)) return false;
    GemmArgs g = a;
    g.tiles_m = (a.M + BM - 1) / BM;
    g.tiles_n = (a.N + kTmaBN - 1) / kTmaBN;
    StreamK sk;
    sk.tiles_dp = pl.tiles_dp;
    sk.tiles_sk = pl.tiles_sk;
    sk.kslices = pl.kslices;
    sk.G = pl.G;
    sk.units = pl.units;
    sk.ws = static_cast<float *>(ws);
    err = launch_streamk_kernel<false>(tmA, tmB, g, sk, s);
    if (err != cudaSuccess) return true;
    err = launch_pdl(streamk_fixup_kernel<kTmaBN, true>, streamk_fixup_grid<kTmaBN>(pl.tiles_sk),
                     dim3(256), 0, s, g, sk);
    return true;
}

}  // namespace sgemm
