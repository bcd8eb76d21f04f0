// Internal launch interface between the C ABI (api.cu) and the kernel
// translation units.  Not part of the public header.
#pragma once

#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

namespace sgemm {

// Unique id of the CUDA context current on the calling thread (the driver's
// context id), 0 when none is current or the driver cannot say.  Ids are never
// reused within a process: a context created after cudaDeviceReset, or another
// context made current on the same device, never matches a value cached for an
// earlier one.  Defined in tf32x3.cu, next to the other driver entry points.
unsigned long long current_context_id();

// A value looked up once per CUDA context (a device address, or the fact that
// a kernel's shared-memory attribute has been set), keyed on the context id.
// Id 0 (unknown context) is never cached, so the caller looks the value up
// again.  A few contexts are kept; the oldest entry is replaced after that.
template <class T>
class PerContext {
  public:
    bool get(unsigned long long ctx, T &out) const {
        if (ctx == 0) return false;
        std::lock_guard<std::mutex> lock(mu_);
        for (int i = 0; i < kSlots; ++i)
            if (ids_[i] == ctx) {
                out = vals_[i];
                return true;
            }
        return false;
    }
    void put(unsigned long long ctx, const T &v) {
        if (ctx == 0) return;
        std::lock_guard<std::mutex> lock(mu_);
        for (int i = 0; i < kSlots; ++i)
            if (ids_[i] == ctx) {
                vals_[i] = v;
                return;
            }
        ids_[next_] = ctx;
        vals_[next_] = v;
        next_ = (next_ + 1) % kSlots;
    }

  private:
    static constexpr int kSlots = 16;
    mutable std::mutex mu_;
    unsigned long long ids_[kSlots] = {};
    T vals_[kSlots] = {};
    int next_ = 0;
};

// One (possibly batched) problem after host-side validation.  All pointers are
// device pointers; strides and leading dimensions are in elements.
struct GemmArgs {
    const float *A;
    const float *B;
    float *C;
    int64_t lda, ldb, ldc;
    int64_t strideA, strideB, strideC;
    int M, N, K;
    int batch;
    int tiles_m, tiles_n;   // output tiles per problem (each launcher sets its own)
    int group_m;            // tile rows per raster group (L2 reuse)
    int kchunk;             // split-K: > 0 means problem z covers k in [z*kchunk, (z+1)*kchunk)
                            // (A/B strides step by one chunk, C by one partial plane)
    // epilogue: C = alpha * op(A) op(B) + beta * C + bias[col]; beta == 0 never
    // reads C, bias may be null.  alpha = 1, beta = 0, bias = null is the plain
    // product and stores the accumulators unchanged.
    float alpha, beta;
    const float *bias;
};

__host__ __device__ inline bool plain_epilogue(const GemmArgs &a) {
    return a.alpha == 1.f && a.beta == 0.f && a.bias == nullptr;
}

// SIMT FP32 kernel family (CUDA cores).  vec: every base pointer, leading
// dimension and batch stride allows 16-byte accesses.
cudaError_t launch_simt(const GemmArgs &a, bool transA, bool transB, bool vec, cudaStream_t s);

// Tensor-core 3xTF32 path: split kernels into `ws` (ws_bytes long, at least
// tf32x3_workspace_min_bytes: the planes), then the tcgen05 GEMM.  With
// tf32x3_workspace_bytes, a problem whose last wave of tiles leaves at least
// half the SMs idle also gets partial tiles for splitting those tiles in K.
cudaError_t launch_tf32x3(const GemmArgs &a, bool transA, bool transB, void *ws, size_t ws_bytes,
                          cudaStream_t s);
size_t tf32x3_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t batch);
size_t tf32x3_workspace_min_bytes(int64_t M, int64_t N, int64_t K, int64_t batch);
cudaError_t tf32x3_read_error(unsigned int *flags, bool reset);
cudaError_t launch_wait_timeout_selftest(long long limit_cycles, cudaStream_t s);
// TF32 tensor-pipe probe: `ctas` CTAs (one per SM), `iters` rounds each.
cudaError_t launch_tf32_mma_probe(long long iters, float *out, int ctas, cudaStream_t s);
double tf32_mma_probe_flops_per_iteration();

// Plain single-term TF32 tensor-core product (hi only), same workspace scheme.
cudaError_t launch_tf32(const GemmArgs &a, bool transA, bool transB, void *ws, cudaStream_t s);
size_t tf32_workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t batch);

// Split-K on the SIMT kernel: `splits` K-chunks into partial planes in `ws`,
// then a fixed-order sum into C.  batch must be 1.
cudaError_t launch_simt_splitk(const GemmArgs &a, bool transA, bool transB, bool vec, int splits,
                               void *ws, cudaStream_t s);
size_t splitk_workspace_bytes(int64_t M, int64_t N, int64_t K, int splits);
int splitk_auto_splits(int64_t M, int64_t N, int64_t K);

// Stream-K schedule of the SIMT kernel (sgemm_f32_streamk): whole waves of
// tiles computed whole, the K slices of the remaining tiles dealt out evenly
// over every resident CTA, shared tiles finished by a fix-up pass from the
// caller's workspace.  `use` is false where it cannot help (the tiles fill
// the SMs a whole number of times, or fewer tiles than SMs) and for layouts
// that corner-turn an operand through registers (see streamk_plan).
struct StreamKPlan {
    bool use, wide;                      // wide: 128 x 256 tiles
    bool tma;                            // the TMA-fed kernel (128 x 128 tiles)
    int tiles_dp, tiles_sk, kslices, G;  // G: CTAs (SMs x resident CTAs per SM)
    int64_t units;                       // tiles_sk * kslices
    size_t ws_bytes;                     // G * 2 partial tiles
};
StreamKPlan streamk_plan(const GemmArgs &a, bool transA, bool transB, bool vec);
cudaError_t launch_simt_streamk(const GemmArgs &a, bool transA, bool transB, bool vec,
                                const StreamKPlan &plan, void *ws, cudaStream_t s);

// The SIMT kernel fed by TMA (row-major B with A either way, or both stored
// transposed; 16-byte aligned operands, no split-K chunks): one 128 x 128
// tile per CTA, two CTAs per SM.  Its stream-K form takes A stored transposed
// and row-major B.
// The launchers return false, launching nothing, when the operands cannot be
// described as tensor maps; else they launch and store the status in `err`.
bool simt_tma_eligible(const GemmArgs &a, bool transA, bool transB, bool vec);
int simt_tma_ctas_per_sm();
bool launch_simt_tma(const GemmArgs &a, bool transA, bool transB, cudaStream_t s,
                     cudaError_t &err);
bool launch_simt_streamk_tma(const GemmArgs &a, bool transA, const StreamKPlan &plan, void *ws,
                             cudaStream_t s, cudaError_t &err);

// Device address of the library's status word (bit 0: a bounded pipeline
// wait ran out), for kernels that report into it; null if unavailable.
unsigned int *device_error_word();

// Y = X^T for a rows x cols row-major X (leading dimension ldx) into Y
// (cols x rows, leading dimension ldy): exact copy, coalesced both ways.
cudaError_t launch_transpose(const float *X, int64_t ldx, int rows, int cols, float *Y, int64_t ldy,
                             cudaStream_t s);

// Matrix-vector shapes (N == 1 or M == 1): bandwidth-bound kernels.
bool gemv_shape(const GemmArgs &a);
cudaError_t launch_gemv(const GemmArgs &a, bool transA, bool transB, cudaStream_t s);

// C[0:M, 0:N] = beta * C + bias for every batch: the whole result when the
// product term vanishes (K == 0 or alpha == 0); zeros for the plain epilogue.
cudaError_t launch_epilogue_only(const GemmArgs &a, cudaStream_t s);

// Tile rows per raster group for the launches that follow (the library's
// choice is 8; sgemm_set_raster_group changes it for measurements).
int raster_group();

// K per chunk of the K-chunked three-term kernel for the launches that follow
// (0: the library's 128; else a multiple of 32); returns the previous value,
// or -1 when chunk_k is not allowed (sgemm_set_tf32x3_chunk_k).
int set_tf32x3_chunk_k(int chunk_k);

// Smallest block tile of any kernel: bounds the grid size during validation.
constexpr int kSimtTileM = 128;
constexpr int kSimtTileN = 128;

}  // namespace sgemm
