// C ABI of the SGEMM library: argument validation, kernel selection, launch.
// The public contract (layout, ownership, errors) is documented in
// include/sgemm_gb300.h.
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>

#include <cuda_runtime.h>

#include "gemm_args.h"
#include "sgemm_gb300.h"

namespace sgemm {

cudaError_t launch_simt_nn(const GemmArgs &a, bool vec, cudaStream_t s);
cudaError_t launch_simt_nt(const GemmArgs &a, bool vec, cudaStream_t s);
cudaError_t launch_simt_tn(const GemmArgs &a, bool vec, cudaStream_t s);
cudaError_t launch_simt_tt(const GemmArgs &a, bool vec, cudaStream_t s);

cudaError_t launch_simt(const GemmArgs &a, bool transA, bool transB, bool vec, cudaStream_t s) {
    if (!transA && !transB) return launch_simt_nn(a, vec, s);
    if (!transA && transB) return launch_simt_nt(a, vec, s);
    if (transA && !transB) return launch_simt_tn(a, vec, s);
    return launch_simt_tt(a, vec, s);
}

cudaError_t launch_simt_streamk_nn(const GemmArgs &, bool, const StreamKPlan &, void *, cudaStream_t);
cudaError_t launch_simt_streamk_nt(const GemmArgs &, bool, const StreamKPlan &, void *, cudaStream_t);
cudaError_t launch_simt_streamk_tn(const GemmArgs &, bool, const StreamKPlan &, void *, cudaStream_t);
cudaError_t launch_simt_streamk_tt(const GemmArgs &, bool, const StreamKPlan &, void *, cudaStream_t);

cudaError_t launch_simt_streamk(const GemmArgs &a, bool transA, bool transB, bool vec,
                                const StreamKPlan &pl, void *ws, cudaStream_t s) {
    if (pl.tma) {
        // the same schedule on the cp.async kernel (128 x 128 tiles) if the
        // operands cannot be described as tensor maps
        cudaError_t e = cudaSuccess;
        if (launch_simt_streamk_tma(a, transA, pl, ws, s, e)) return e;
    }
    if (!transA && !transB) return launch_simt_streamk_nn(a, vec, pl, ws, s);
    if (!transA && transB) return launch_simt_streamk_nt(a, vec, pl, ws, s);
    if (transA && !transB) return launch_simt_streamk_tn(a, vec, pl, ws, s);
    return launch_simt_streamk_tt(a, vec, pl, ws, s);
}

// Only for A stored transposed with row-major B: the one layout whose
// operands both arrive without a corner turn.  Where an operand is
// corner-turned through registers (row-major A, or B^T), a CTA that runs tile
// after tile left those 16-byte global loads exposed (long-scoreboard stalls
// 0.007 -> 0.75 per instruction, 15 % slower per tile on 2048 x 4864 x 4096),
// more than the wave tail stream-K removes.  With 16-byte aligned operands
// the TMA-fed kernel runs it on 128 x 128 tiles with G = every resident CTA
// (two per SM), and only below four waves of G: two CTAs per SM already
// absorb most of a wave tail (a lone CTA runs faster), so beyond that the
// partial tiles and the fix-up cost more than the tail (8192^3: 70.9 TFLOP/s
// plain, 69.3 with stream-K; 2048 x 3072 x 1536: 56.9 plain, 62.8 with it).
// Otherwise the cp.async kernel on one CTA per SM, with 128 x 256 tiles where
// it can use 16-byte access.
StreamKPlan streamk_plan(const GemmArgs &a, bool transA, bool transB, bool vec) {
    StreamKPlan pl = {};
    if (!transA || transB) return pl;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return pl;
    pl.tma = simt_tma_eligible(a, transA, transB, vec);
    pl.wide = !pl.tma && vec && !transB;
    const int64_t bn = pl.wide ? 256 : 128;
    const int64_t tiles = (int64_t)a.batch * ((a.M + 127) / 128) * ((a.N + bn - 1) / bn);
    pl.G = sms * (pl.tma ? simt_tma_ctas_per_sm() : 1);
    pl.kslices = (a.K + 31) / 32;
    pl.use = tiles > pl.G && tiles % pl.G != 0 && pl.kslices >= 2 && tiles <= (1LL << 30) &&
             (!pl.tma || tiles < 4LL * pl.G);
    if (!pl.use) return pl;
    pl.tiles_dp = (int)(tiles / pl.G * pl.G);
    pl.tiles_sk = (int)(tiles - pl.tiles_dp);
    pl.units = (int64_t)pl.tiles_sk * pl.kslices;
    pl.ws_bytes = (size_t)pl.G * 2 * 128 * (size_t)bn * sizeof(float);
    return pl;
}

namespace {

__global__ void epilogue_only_kernel(float *C, int64_t ldc, int64_t strideC, int M, int N,
                                     int batch, float beta, const float *bias) {
    const int64_t total = (int64_t)batch * M * N;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t z = t / ((int64_t)M * N);
        const int64_t r = t - z * (int64_t)M * N;
        const int64_t i = r / N, j = r - i * N;
        float *c = C + z * strideC + i * ldc + j;
        float v = beta != 0.f ? beta * *c : 0.f;
        if (bias) v += bias[j];
        *c = v;
    }
}

thread_local char g_last_error[512] = "";

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return code;
}

constexpr int64_t kMaxDim = (int64_t)1 << 30;    // kernels index within a problem in int32
constexpr int64_t kMaxLd = (int64_t)1 << 40;
constexpr int64_t kMaxStride = (int64_t)1 << 60;
constexpr int64_t kMaxBlocks = ((int64_t)1 << 31) - 1;

bool aligned(const void *p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

// Is the current device an sm_103 part?  Cached per device ordinal.
int check_device() {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0)
        return fail(SGEMM_EDEVICE, "no CUDA device: %s", cudaGetErrorString(e));
    static int cc_cache[64];   // 0 = unknown, else 10*major + minor
    int cc = dev < 64 ? cc_cache[dev] : 0;
    if (cc == 0) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cc = 10 * major + minor;
        if (dev < 64) cc_cache[dev] = cc;
    }
    if (cc != 103)
        return fail(SGEMM_EDEVICE, "device %d has compute capability %d.%d; this library is built "
                    "for sm_103a (GB300) only", dev, cc / 10, cc % 10);
    return SGEMM_OK;
}

// Validates a strided-batched problem.  Returns SGEMM_OK and fills `a` when
// there is work to do; `nothing` is set when the call is a no-op.
int validate(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, int64_t strideA,
             const float *B, int64_t ldb, int64_t strideB, float *C, int64_t ldc,
             int64_t strideC, int64_t batch, int transA, int transB, GemmArgs &a,
             bool &nothing) {
    nothing = false;
    if ((transA != 0 && transA != 1) || (transB != 0 && transB != 1))
        return fail(SGEMM_EINVAL_TRANS, "transA=%d transB=%d: each must be 0 or 1", transA, transB);
    if (M < 0 || N < 0 || K < 0)
        return fail(SGEMM_EINVAL_DIM, "negative size M=%lld N=%lld K=%lld", (long long)M,
                    (long long)N, (long long)K);
    if (batch < 0) return fail(SGEMM_EINVAL_BATCH, "batch=%lld is negative", (long long)batch);
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim)
        return fail(SGEMM_EINVAL_DIM, "a size exceeds 2^30 (M=%lld N=%lld K=%lld)", (long long)M,
                    (long long)N, (long long)K);
    const int64_t min_lda = transA ? (M > 1 ? M : 1) : (K > 1 ? K : 1);
    const int64_t min_ldb = transB ? (K > 1 ? K : 1) : (N > 1 ? N : 1);
    const int64_t min_ldc = N > 1 ? N : 1;
    if (lda < min_lda || ldb < min_ldb || ldc < min_ldc)
        return fail(SGEMM_EINVAL_LD, "leading dimension too small: lda=%lld (min %lld) ldb=%lld "
                    "(min %lld) ldc=%lld (min %lld)", (long long)lda, (long long)min_lda,
                    (long long)ldb, (long long)min_ldb, (long long)ldc, (long long)min_ldc);
    if (lda > kMaxLd || ldb > kMaxLd || ldc > kMaxLd)
        return fail(SGEMM_EINVAL_LD, "leading dimension above 2^40");
    if (M == 0 || N == 0 || batch == 0) {
        nothing = true;
        return SGEMM_OK;
    }
    if (batch > 1) {
        if (strideA < 0 || strideB < 0 || strideC < 0 || strideA > kMaxStride ||
            strideB > kMaxStride || strideC > kMaxStride)
            return fail(SGEMM_EINVAL_BATCH, "batch strides must be non-negative");
        const int64_t c_extent = (M - 1) * ldc + N;
        if (strideC < c_extent)
            return fail(SGEMM_EINVAL_BATCH, "strideC=%lld lets the C matrices of two batches "
                        "overlap (need >= %lld)", (long long)strideC, (long long)c_extent);
    }
    if (C == nullptr) return fail(SGEMM_EINVAL_PTR, "C is NULL");
    if (!aligned(C, 4)) return fail(SGEMM_EINVAL_PTR, "C is not 4-byte aligned");
    if (K > 0) {
        if (A == nullptr || B == nullptr) return fail(SGEMM_EINVAL_PTR, "A or B is NULL");
        if (!aligned(A, 4) || !aligned(B, 4))
            return fail(SGEMM_EINVAL_PTR, "A or B is not 4-byte aligned");
    }
    const int64_t tiles_m = (M + kSimtTileM - 1) / kSimtTileM;
    const int64_t tiles_n = (N + kSimtTileN - 1) / kSimtTileN;
    if (batch * tiles_m * tiles_n > kMaxBlocks)
        return fail(SGEMM_EINVAL_DIM, "problem needs more than 2^31-1 thread blocks");
    a.A = A;
    a.B = B;
    a.C = C;
    a.lda = lda;
    a.ldb = ldb;
    a.ldc = ldc;
    a.strideA = batch > 1 ? strideA : 0;
    a.strideB = batch > 1 ? strideB : 0;
    a.strideC = batch > 1 ? strideC : 0;
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.batch = (int)batch;
    a.tiles_m = (int)tiles_m;
    a.tiles_n = (int)tiles_n;
    a.group_m = raster_group();
    a.kchunk = 0;
    a.alpha = 1.f;
    a.beta = 0.f;
    a.bias = nullptr;
    return SGEMM_OK;
}

// 16-byte accesses are legal when every base, leading dimension and batch
// stride keeps float4 groups aligned.
bool vector_ok(const GemmArgs &a) {
    return aligned(a.A, 16) && aligned(a.B, 16) && aligned(a.C, 16) && a.lda % 4 == 0 &&
           a.ldb % 4 == 0 && a.ldc % 4 == 0 && a.strideA % 4 == 0 && a.strideB % 4 == 0 &&
           a.strideC % 4 == 0;
}

enum class Path { Simt, Tf32x3, Tf32 };

struct Epi {
    float alpha = 1.f, beta = 0.f;
    const float *bias = nullptr;
};

int run(Path path, int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, int64_t strideA,
        const float *B, int64_t ldb, int64_t strideB, float *C, int64_t ldc, int64_t strideC,
        int64_t batch, int transA, int transB, void *workspace, uint64_t workspace_bytes,
        void *stream, const Epi &epi = Epi()) {
    g_last_error[0] = '\0';
    GemmArgs a;
    bool nothing = false;
    int st = validate(M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc, strideC, batch, transA,
                      transB, a, nothing);
    if (st != SGEMM_OK || nothing) return st;
    if (epi.bias != nullptr && !aligned(epi.bias, 4))
        return fail(SGEMM_EINVAL_PTR, "bias is not 4-byte aligned");
    a.alpha = epi.alpha;
    a.beta = epi.beta;
    a.bias = epi.bias;
    if (a.alpha == 0.f) K = 0;   // the product term vanishes: A and B are not read
    if (path != Path::Simt && K > 0) {
        const uint64_t need = path == Path::Tf32x3 ? tf32x3_workspace_min_bytes(M, N, K, batch)
                                                   : tf32_workspace_bytes(M, N, K, batch);
        if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < need)
            return fail(SGEMM_EWORKSPACE, "workspace %p of %llu bytes: need %llu bytes, 256-byte "
                        "aligned", workspace, (unsigned long long)workspace_bytes,
                        (unsigned long long)need);
    }
    st = check_device();
    if (st != SGEMM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (K == 0) {
        e = launch_epilogue_only(a, s);
    } else if (path == Path::Tf32x3) {
        e = launch_tf32x3(a, transA != 0, transB != 0, workspace, workspace_bytes, s);
    } else if (path == Path::Tf32) {
        e = launch_tf32(a, transA != 0, transB != 0, workspace, s);
    } else if (gemv_shape(a)) {
        e = launch_gemv(a, transA != 0, transB != 0, s);
    } else {
        e = launch_simt(a, transA != 0, transB != 0, vector_ok(a), s);
    }
    if (e != cudaSuccess)
        return fail(SGEMM_ELAUNCH, "kernel launch failed: %s", cudaGetErrorString(e));
    return SGEMM_OK;
}

}  // namespace

int run_splitk(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
               int64_t ldb, float *C, int64_t ldc, int transA, int transB, int splits,
               void *workspace, uint64_t workspace_bytes, void *stream);

// Records a failure detail for sgemm_last_error() on behalf of another
// translation unit and returns `code`.
int record_error(int code, const char *msg) { return fail(code, "%s", msg); }

// The workspace plan of sgemm_f32_streamk.  A K-contiguous operand (row-major
// A, B stored transposed) of a large problem is first turned into an
// M/N-contiguous copy, so the tile kernel sees A^T with row-major B (both
// operands by cp.async, and the layout stream-K runs well on); the copy costs
// about 8 bytes per element against 2N (for A) or 2M (for B) flops.  The
// stream-K partial tiles follow the copies.
struct TurnPlan {
    bool turnA = false, turnB = false;
    int64_t ldA = 0, ldB = 0;     // leading dimensions of the copies
    size_t offA = 0, offB = 0, offP = 0, bytes = 0;
    StreamKPlan sk = {};
};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// `vec`: whether the problem the tile kernel sees allows 16-byte access
// (callers that do not know pass true: the larger workspace).
TurnPlan turn_plan(const GemmArgs &a, bool transA, bool transB, bool vec) {
    TurnPlan tp;
    const bool big = 2.0 * a.M * (double)a.N * a.K >= 1.6e10;
    tp.turnA = big && !transA && a.N >= 1024;
    tp.turnB = big && transB && a.M >= 1024;
    size_t off = 0;
    if (tp.turnA) {
        tp.ldA = ((int64_t)a.M + 3) / 4 * 4;
        tp.offA = off;
        off += round256((size_t)a.K * tp.ldA * sizeof(float));
    }
    if (tp.turnB) {
        tp.ldB = ((int64_t)a.N + 3) / 4 * 4;
        tp.offB = off;
        off += round256((size_t)a.K * tp.ldB * sizeof(float));
    }
    tp.sk = streamk_plan(a, transA || tp.turnA, transB && !tp.turnB, vec);
    if (tp.sk.use) {
        tp.offP = off;
        off += tp.sk.ws_bytes;
    }
    tp.bytes = off;
    return tp;
}

// The workspace the call may need: whether the tile kernel gets 16-byte access
// is only known from the pointers, and both the tile width and whether
// stream-K applies follow from it, so the larger need of the two.
size_t turn_plan_bytes(const GemmArgs &a, bool transA, bool transB) {
    const size_t wide = turn_plan(a, transA, transB, true).bytes;
    const size_t narrow = turn_plan(a, transA, transB, false).bytes;
    return wide > narrow ? wide : narrow;
}

// sgemm_f32 with turned operands and the stream-K schedule (see TurnPlan and
// StreamKPlan); problems neither helps run exactly as sgemm_f32 and need no
// workspace.
int run_streamk(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
                int64_t ldb, float *C, int64_t ldc, int transA, int transB, void *workspace,
                uint64_t workspace_bytes, void *stream) {
    g_last_error[0] = '\0';
    GemmArgs a;
    bool nothing = false;
    int st = validate(M, N, K, A, lda, 0, B, ldb, 0, C, ldc, 0, 1, transA, transB, a, nothing);
    if (st != SGEMM_OK || nothing) return st;
    const bool matvec = K == 0 || gemv_shape(a);
    const TurnPlan need = matvec ? TurnPlan{} : turn_plan(a, transA != 0, transB != 0, true);
    const size_t need_bytes = matvec ? 0 : turn_plan_bytes(a, transA != 0, transB != 0);
    if (need_bytes > 0 && (workspace == nullptr || !aligned(workspace, 256) ||
                           workspace_bytes < need_bytes))
        return fail(SGEMM_EWORKSPACE, "workspace %p of %llu bytes: this problem needs %llu bytes, "
                    "256-byte aligned", workspace, (unsigned long long)workspace_bytes,
                    (unsigned long long)need_bytes);
    st = check_device();
    if (st != SGEMM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (K == 0) {
        e = launch_epilogue_only(a, s);
    } else if (gemv_shape(a)) {
        e = launch_gemv(a, transA != 0, transB != 0, s);
    } else {
        // the problem the tile kernel sees: turned copies in the workspace
        GemmArgs t = a;
        bool tA = transA != 0, tB = transB != 0;
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        if (need.turnA) {
            float *copy = reinterpret_cast<float *>(ws + need.offA);
            e = launch_transpose(a.A, a.lda, a.M, a.K, copy, need.ldA, s);   // M x K -> K x M
            t.A = copy;
            t.lda = need.ldA;
            tA = true;
        }
        if (e == cudaSuccess && need.turnB) {
            float *copy = reinterpret_cast<float *>(ws + need.offB);
            e = launch_transpose(a.B, a.ldb, a.N, a.K, copy, need.ldB, s);   // N x K -> K x N
            t.B = copy;
            t.ldb = need.ldB;
            tB = false;
        }
        if (e == cudaSuccess) {
            const bool vec = vector_ok(t);
            const StreamKPlan sk = streamk_plan(t, tA, tB, vec);
            if (sk.use)
                e = launch_simt_streamk(t, tA, tB, vec, sk, ws + need.offP, s);
            else
                e = launch_simt(t, tA, tB, vec, s);
        }
    }
    if (e != cudaSuccess)
        return fail(SGEMM_ELAUNCH, "kernel launch failed: %s", cudaGetErrorString(e));
    return SGEMM_OK;
}

int run_splitk(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
               int64_t ldb, float *C, int64_t ldc, int transA, int transB, int splits,
               void *workspace, uint64_t workspace_bytes, void *stream) {
    g_last_error[0] = '\0';
    if (splits < 0 || splits > 4096)
        return fail(SGEMM_EINVAL_DIM, "splits=%d: must be 0 (automatic) or 1..4096", splits);
    GemmArgs a;
    bool nothing = false;
    int st = validate(M, N, K, A, lda, 0, B, ldb, 0, C, ldc, 0, 1, transA, transB, a, nothing);
    if (st != SGEMM_OK || nothing) return st;
    if (K > 0 && splits == 0) splits = splitk_auto_splits(M, N, K);
    // the number of K-chunks actually used (chunks are whole 32-wide slices)
    const int64_t chunk = K > 0 ? ((K + splits - 1) / splits + 31) / 32 * 32 : 0;
    const int used = K > 0 ? (int)((K + chunk - 1) / chunk) : 1;
    if (K > 0 && used > 1) {
        const uint64_t need = splitk_workspace_bytes(M, N, K, splits);
        if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < need)
            return fail(SGEMM_EWORKSPACE, "workspace %p of %llu bytes: split-K needs %llu bytes, "
                        "256-byte aligned", workspace, (unsigned long long)workspace_bytes,
                        (unsigned long long)need);
    }
    st = check_device();
    if (st != SGEMM_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (K == 0)
        e = launch_epilogue_only(a, s);
    else if (used <= 1)
        e = launch_simt(a, transA != 0, transB != 0, vector_ok(a), s);
    else {
        const bool vec = aligned(A, 16) && aligned(B, 16) && lda % 4 == 0 && ldb % 4 == 0;
        e = launch_simt_splitk(a, transA != 0, transB != 0, vec, splits, workspace, s);
    }
    if (e != cudaSuccess)
        return fail(SGEMM_ELAUNCH, "kernel launch failed: %s", cudaGetErrorString(e));
    return SGEMM_OK;
}

cudaError_t launch_epilogue_only(const GemmArgs &a, cudaStream_t s) {
    const int64_t total = (int64_t)a.batch * a.M * a.N;
    int blocks = (int)((total + 255) / 256);
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    epilogue_only_kernel<<<blocks, 256, 0, s>>>(a.C, a.ldc, a.strideC, a.M, a.N, a.batch, a.beta,
                                                a.bias);
    return cudaGetLastError();
}

}  // namespace sgemm

extern "C" {

int sgemm_f32(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
              int64_t ldb, float *C, int64_t ldc, int transA, int transB, void *stream) {
    return sgemm::run(sgemm::Path::Simt, M, N, K, A, lda, 0, B, ldb, 0, C, ldc, 0, 1, transA,
                      transB, nullptr, 0, stream);
}

int sgemm_f32_strided_batched(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                              int64_t strideA, const float *B, int64_t ldb, int64_t strideB,
                              float *C, int64_t ldc, int64_t strideC, int64_t batch, int transA,
                              int transB, void *stream) {
    return sgemm::run(sgemm::Path::Simt, M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc,
                      strideC, batch, transA, transB, nullptr, 0, stream);
}

int sgemm_f32_tf32x3(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
                     int64_t ldb, float *C, int64_t ldc, int transA, int transB, void *workspace,
                     uint64_t workspace_bytes, void *stream) {
    return sgemm::run(sgemm::Path::Tf32x3, M, N, K, A, lda, 0, B, ldb, 0, C, ldc, 0, 1, transA,
                      transB, workspace, workspace_bytes, stream);
}

int sgemm_f32_tf32x3_strided_batched(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                                     int64_t strideA, const float *B, int64_t ldb, int64_t strideB,
                                     float *C, int64_t ldc, int64_t strideC, int64_t batch,
                                     int transA, int transB, void *workspace,
                                     uint64_t workspace_bytes, void *stream) {
    return sgemm::run(sgemm::Path::Tf32x3, M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc,
                      strideC, batch, transA, transB, workspace, workspace_bytes, stream);
}

int sgemm_f32_tf32(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
                   int64_t ldb, float *C, int64_t ldc, int transA, int transB, void *workspace,
                   uint64_t workspace_bytes, void *stream) {
    return sgemm::run(sgemm::Path::Tf32, M, N, K, A, lda, 0, B, ldb, 0, C, ldc, 0, 1, transA,
                      transB, workspace, workspace_bytes, stream);
}

int sgemm_f32_tf32_strided_batched(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                                   int64_t strideA, const float *B, int64_t ldb, int64_t strideB,
                                   float *C, int64_t ldc, int64_t strideC, int64_t batch,
                                   int transA, int transB, void *workspace,
                                   uint64_t workspace_bytes, void *stream) {
    return sgemm::run(sgemm::Path::Tf32, M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc,
                      strideC, batch, transA, transB, workspace, workspace_bytes, stream);
}

int sgemm_f32_ex(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                 const float *B, int64_t ldb, float beta, float *C, int64_t ldc, const float *bias,
                 int transA, int transB, void *stream) {
    sgemm::Epi e;
    e.alpha = alpha;
    e.beta = beta;
    e.bias = bias;
    return sgemm::run(sgemm::Path::Simt, M, N, K, A, lda, 0, B, ldb, 0, C, ldc, 0, 1, transA,
                      transB, nullptr, 0, stream, e);
}

int sgemm_f32_ex_strided_batched(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                                 int64_t lda, int64_t strideA, const float *B, int64_t ldb,
                                 int64_t strideB, float beta, float *C, int64_t ldc,
                                 int64_t strideC, const float *bias, int64_t batch, int transA,
                                 int transB, void *stream) {
    sgemm::Epi e;
    e.alpha = alpha;
    e.beta = beta;
    e.bias = bias;
    return sgemm::run(sgemm::Path::Simt, M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc,
                      strideC, batch, transA, transB, nullptr, 0, stream, e);
}

int sgemm_f32_tf32x3_ex(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                        const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                        const float *bias, int transA, int transB, void *workspace,
                        uint64_t workspace_bytes, void *stream) {
    sgemm::Epi e;
    e.alpha = alpha;
    e.beta = beta;
    e.bias = bias;
    return sgemm::run(sgemm::Path::Tf32x3, M, N, K, A, lda, 0, B, ldb, 0, C, ldc, 0, 1, transA,
                      transB, workspace, workspace_bytes, stream, e);
}

int sgemm_f32_splitk(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda, const float *B,
                     int64_t ldb, float *C, int64_t ldc, int transA, int transB, int splits,
                     void *workspace, uint64_t workspace_bytes, void *stream) {
    return sgemm::run_splitk(M, N, K, A, lda, B, ldb, C, ldc, transA, transB, splits, workspace,
                             workspace_bytes, stream);
}

int sgemm_f32_streamk(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                      const float *B, int64_t ldb, float *C, int64_t ldc, int transA, int transB,
                      void *workspace, uint64_t workspace_bytes, void *stream) {
    return sgemm::run_streamk(M, N, K, A, lda, B, ldb, C, ldc, transA, transB, workspace,
                              workspace_bytes, stream);
}

uint64_t sgemm_f32_streamk_workspace_size(int64_t M, int64_t N, int64_t K, int transA, int transB) {
    if (M <= 1 || N <= 1 || K <= 0 || M > (1 << 30) || N > (1 << 30) || K > (1 << 30) ||
        (transA != 0 && transA != 1) || (transB != 0 && transB != 1))
        return 0;
    sgemm::GemmArgs a = {};
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.batch = 1;
    return sgemm::turn_plan_bytes(a, transA != 0, transB != 0);
}

int sgemm_f32_splitk_auto_splits(int64_t M, int64_t N, int64_t K) {
    if (M <= 0 || N <= 0 || K <= 0 || M > (1 << 30) || N > (1 << 30) || K > (1 << 30)) return 1;
    return sgemm::splitk_auto_splits(M, N, K);
}

uint64_t sgemm_f32_splitk_workspace_size(int64_t M, int64_t N, int64_t K, int splits) {
    if (M <= 0 || N <= 0 || K <= 0 || splits < 0) return 0;
    if (splits == 0) splits = sgemm_f32_splitk_auto_splits(M, N, K);
    return sgemm::splitk_workspace_bytes(M, N, K, splits);
}

uint64_t sgemm_f32_tf32_workspace_size(int64_t M, int64_t N, int64_t K, int64_t batch) {
    if (M <= 0 || N <= 0 || K <= 0 || batch <= 0) return 0;
    return sgemm::tf32_workspace_bytes(M, N, K, batch);
}

uint64_t sgemm_f32_tf32x3_workspace_size(int64_t M, int64_t N, int64_t K, int64_t batch) {
    if (M <= 0 || N <= 0 || K <= 0 || batch <= 0) return 0;
    return sgemm::tf32x3_workspace_bytes(M, N, K, batch);
}

int sgemm_device_status(unsigned int *flags, int reset) {
    if (flags == nullptr) return SGEMM_EINVAL_PTR;
    int st = sgemm::check_device();
    if (st != SGEMM_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = sgemm::tf32x3_read_error(flags, reset != 0);
    if (e != cudaSuccess)
        return sgemm::fail(SGEMM_ELAUNCH, "device status read failed: %s", cudaGetErrorString(e));
    return SGEMM_OK;
}

const char *sgemm_status_string(int status) {
    switch (status) {
        case SGEMM_OK: return "SGEMM_OK";
        case SGEMM_EINVAL_DIM: return "SGEMM_EINVAL_DIM: invalid size";
        case SGEMM_EINVAL_LD: return "SGEMM_EINVAL_LD: invalid leading dimension";
        case SGEMM_EINVAL_PTR: return "SGEMM_EINVAL_PTR: invalid pointer";
        case SGEMM_EINVAL_TRANS: return "SGEMM_EINVAL_TRANS: invalid transpose flag";
        case SGEMM_EINVAL_BATCH: return "SGEMM_EINVAL_BATCH: invalid batch or stride";
        case SGEMM_ELAUNCH: return "SGEMM_ELAUNCH: kernel launch failed";
        case SGEMM_EDEVICE: return "SGEMM_EDEVICE: no usable sm_103 device";
        case SGEMM_EWORKSPACE: return "SGEMM_EWORKSPACE: workspace missing, misaligned or too small";
        default: return "unknown sgemm status";
    }
}

const char *sgemm_last_error(void) { return sgemm::g_last_error; }

int sgemm_version(void) { return 200; }

}  // extern "C"
