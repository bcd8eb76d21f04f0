/*
 * sgemm_gb300.h -- single-precision GEMM on NVIDIA GB300 (sm_103a).
 *
 * The operation is the GEMM of "CUDA GEMM operator performance optimization",
 * section 1.1: C = A x B with A of size M x K, B of size K x N and C of size
 * M x N, all float32, 2*M*N*K floating-point operations.  The batched form
 * ("Batched GEMM: batched matmul in multi-head attention", same page, section
 * 1.2) applies it to independent problems at fixed strides, e.g. Q K^T.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layout.  All matrices are ROW-MAJOR, as in the page's kernels
 *   (element (r, c) of an R x C matrix with leading dimension ld at X[r*ld + c]).
 *   op(X) = X when trans == 0 and X^T when trans == 1, where trans describes
 *   how the operand is STORED:
 *     A, transA == 0: stored M x K, opA(i,k) = A[i*lda + k], lda >= max(1, K)
 *     A, transA == 1: stored K x M, opA(i,k) = A[k*lda + i], lda >= max(1, M)
 *     B, transB == 0: stored K x N, opB(k,j) = B[k*ldb + j], ldb >= max(1, N)
 *     B, transB == 1: stored N x K, opB(k,j) = B[j*ldb + k], ldb >= max(1, K)
 *     C:              stored M x N, C(i,j)   = C[i*ldc + j], ldc >= max(1, N)
 *   The result OVERWRITES C[0:M, 0:N]: C = op(A) op(B).  There is no alpha or
 *   beta (the operation on the pages has none).  Padding columns
 *   (c >= N of C, and likewise for A and B) are never read or written.
 *
 * Pointers and ownership.  A, B and C are DEVICE pointers (cudaMalloc, torch
 *   tensors, ...) owned by the caller, 4-byte aligned.  A and C, or B and C,
 *   must not overlap.  The library keeps no pointer after the call returns
 *   and allocates no device memory per call.
 *
 * Streams.  `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *   default stream).  Work is enqueued on it and the call returns without
 *   synchronising; the result is visible to later work on that stream.
 *
 * Precision.  sgemm_f32*: every product and sum is an fp32 FMA on the CUDA
 *   cores, each output's terms accumulated in ascending k by one thread (when
 *   the problem is too small to fill the GPU, K is first cut into chunks, each
 *   chunk accumulated that way and the chunk sums added in chunk order); the
 *   result is deterministic (bit-identical across calls).  sgemm_f32_tf32x3*:
 *   tensor cores with the three-term TF32 split (see below).
 *
 * Errors.  Arguments are validated on the host before anything is enqueued;
 *   on a violation the call returns a nonzero sgemm_status, enqueues nothing,
 *   and sgemm_last_error() describes it.  Launch failures return
 *   SGEMM_ELAUNCH.  Errors of the asynchronous execution itself surface, as
 *   usual in CUDA, at the caller's next synchronisation.  The library never
 *   exits or aborts the process.
 *
 * Degenerate sizes.  M == 0, N == 0 or batch == 0: nothing is done, SGEMM_OK
 *   (pointers may then be NULL).  K == 0: C[0:M,0:N] is set to zero (the
 *   empty sum); A and B are not read and may be NULL.
 */
#ifndef SGEMM_GB300_H
#define SGEMM_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The library is built with hidden symbol visibility; only the entry points
 * declared here are exported. */
#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

typedef enum {
    SGEMM_OK = 0,
    SGEMM_EINVAL_DIM = 1,    /* M, N or K negative, or too large for the grid */
    SGEMM_EINVAL_LD = 2,     /* a leading dimension below its minimum */
    SGEMM_EINVAL_PTR = 3,    /* NULL where data is needed, or not 4-byte aligned */
    SGEMM_EINVAL_TRANS = 4,  /* transA/transB not 0 or 1 */
    SGEMM_EINVAL_BATCH = 5,  /* batch < 0, or strideC lets two problems' C overlap */
    SGEMM_ELAUNCH = 6,       /* the kernel launch itself failed */
    SGEMM_EDEVICE = 7,       /* no usable device, or the device is not sm_103 */
    SGEMM_EWORKSPACE = 8     /* workspace NULL, misaligned or smaller than required */
} sgemm_status;

/*
 * C = op(A) op(B), fp32 on the CUDA cores.
 * Defined by: "CUDA GEMM operator performance optimization", section 1.1
 * (GEMM), built as in sections 4-10 of that page (block, warp and thread
 * tiling, float4 access, transposed/swizzled shared-memory tiles, multi-stage
 * asynchronous copies); edge tiles are zero-padded as in the DD2360 workbook,
 * section 14.3.  Matrix-vector shapes (N == 1 or M == 1) go to bandwidth-bound
 * kernels instead (warp-per-output dot products or thread-per-output column
 * sums, DD2360 workbook section 15.2); their sums run in a different but
 * fixed order, so they are deterministic too.  Problems whose 128 x 128
 * output tiles cover at most half the SMs (e.g. 256 x 256 x 256: four tiles)
 * split K over the 2, 4, 8 or 16 CTAs of a thread-block cluster and add the
 * partial tiles on chip through distributed shared memory, in chunk order:
 * the split-K of the ChetanC28/cuda-kernels page without a workspace.  The
 * smallest of them (256^3, 384^3, 128 x 128 x 32768, ...) take 64 x 64 tiles
 * for this, which cuts the work on each CTA's critical path.
 */
int sgemm_f32(int64_t M, int64_t N, int64_t K,
              const float *A, int64_t lda,
              const float *B, int64_t ldb,
              float *C, int64_t ldc,
              int transA, int transB, void *stream);

/*
 * For z in [0, batch): C_z = op(A_z) op(B_z) with X_z = X + z*strideX
 * (strides in elements).  strideA and strideB may be 0 (broadcast one
 * operand).  strideC must keep the batches' C regions disjoint:
 * strideC >= (M-1)*ldc + N when batch > 1 (else SGEMM_EINVAL_BATCH).
 * Defined by: "CUDA GEMM operator performance optimization", section 1.2
 * (batched matmul, Q K^T in attention), each problem as in sgemm_f32.
 */
int sgemm_f32_strided_batched(int64_t M, int64_t N, int64_t K,
                              const float *A, int64_t lda, int64_t strideA,
                              const float *B, int64_t ldb, int64_t strideB,
                              float *C, int64_t ldc, int64_t strideC,
                              int64_t batch, int transA, int transB, void *stream);

/*
 * C = alpha * op(A) op(B) + beta * C + bias, fp32 on the CUDA cores: the
 * fully connected layer Y = XW + b ("CUDA GEMM operator performance
 * optimization", section 1.2) with BLAS-style scaling, fused into the store
 * of sgemm_f32's kernel (each output: alpha * acc, then fma with beta * C,
 * then + bias[j], fp32).
 *   bias   NULL, or a device array of N floats added to every row.
 *   beta   0 means C is not read (it may hold anything, NaN included).
 *   alpha  0 means A and B are not read; C = beta * C + bias.
 * Results meet |C - C_ref| <= 1e-5 * (|alpha| sum_k |a||b| + |beta||C| +
 * |bias|) + 1e-6 against the same expression formed exactly.
 * Arguments otherwise as sgemm_f32.
 */
int sgemm_f32_ex(int64_t M, int64_t N, int64_t K, float alpha,
                 const float *A, int64_t lda,
                 const float *B, int64_t ldb,
                 float beta, float *C, int64_t ldc,
                 const float *bias, int transA, int transB, void *stream);

/* Strided-batched form of sgemm_f32_ex; the same bias row for every batch. */
int sgemm_f32_ex_strided_batched(int64_t M, int64_t N, int64_t K, float alpha,
                                 const float *A, int64_t lda, int64_t strideA,
                                 const float *B, int64_t ldb, int64_t strideB,
                                 float beta, float *C, int64_t ldc, int64_t strideC,
                                 const float *bias, int64_t batch, int transA, int transB,
                                 void *stream);

/*
 * sgemm_f32 with K split into `splits` chunks for problems whose output tiles
 * cannot fill the GPU (e.g. 256 x 256 x 256 is four 128 x 128 tiles, and
 * 128 x 128 x 32768 is one).  Each chunk computes a partial product into the
 * workspace; one more pass sums the partials in chunk order into C, so the
 * result is deterministic (not bit-identical to sgemm_f32: the sum is grouped
 * differently), meets the same FP32 bound, and is exact on small integers.
 * Defined by: the split-K stage of the ChetanC28/cuda-kernels page
 * ("splitting the K dimension across blocks for small problems", 28.87x on a
 * 128 x 128 x 32768 product), each chunk as in sgemm_f32.
 *   splits     0: choose automatically (sgemm_f32_splitk_auto_splits), else
 *              1..4096; chunks are whole multiples of 32 in K, so fewer
 *              chunks than asked may be used.  One chunk = plain sgemm_f32
 *              (no workspace needed).
 *   workspace  caller-owned device memory of at least
 *              sgemm_f32_splitk_workspace_size(M, N, K, splits) bytes,
 *              256-byte aligned, not overlapping A, B or C, not used by other
 *              work while this call runs on `stream`.  SGEMM_EWORKSPACE if
 *              missing or too small.
 * Not batched.  Arguments otherwise as sgemm_f32.
 */
int sgemm_f32_splitk(int64_t M, int64_t N, int64_t K,
                     const float *A, int64_t lda,
                     const float *B, int64_t ldb,
                     float *C, int64_t ldc,
                     int transA, int transB, int splits,
                     void *workspace, uint64_t workspace_bytes, void *stream);

/*
 * sgemm_f32 using a caller workspace for two things the tile kernel gains
 * from.  Deterministic on a given device, not bit-identical to sgemm_f32,
 * meets the same FP32 bound and is exact on small integers.
 *   1. Operand turning.  In a large problem (2MNK >= 1.6e10) an operand
 *      contiguous along K (row-major A with N >= 1024, or B stored transposed
 *      with M >= 1024) is first copied, transposed, into the workspace.  The
 *      tile kernel then streams both operands with 16-byte cp.async instead
 *      of corner-turning one through registers, as it does for A stored
 *      transposed with row-major B, the fastest layout (3072^3: 61.3 against
 *      58.0 TFLOP/s).  The copy is exact and costs about 8 bytes per element.
 *   2. A stream-K schedule, for that layout, when the output tiles fill the
 *      SMs a non-whole number of times (3072^3: 288 tiles of 128 x 256 on 152
 *      SMs leaves 16 SMs idle through the second wave).  Whole waves of tiles
 *      are computed whole; the K slices of the remaining tiles are dealt out
 *      evenly over one CTA per SM, and the tiles shared between CTAs are
 *      finished by a second pass that adds their pieces in K order.
 * Defined by: the GEMM of "CUDA GEMM operator performance optimization",
 * section 1.1, with the transposed-operand layout of its section 7.3 and the
 * split-K stage of the ChetanC28/cuda-kernels page (K split across blocks,
 * partial sums reduced afterwards) applied to the tail of the tile schedule.
 *   workspace  caller-owned device memory of at least
 *              sgemm_f32_streamk_workspace_size(M, N, K, transA, transB)
 *              bytes, 256-byte aligned, not overlapping A, B or C, not used
 *              by other work while this call runs on `stream`.  Problems that
 *              neither step helps (small ones, matrix-vector shapes, K = 0)
 *              run as sgemm_f32 and need none: the size is then 0 and
 *              workspace may be NULL.  SGEMM_EWORKSPACE if required and
 *              missing or too small.
 * Not batched.  Arguments otherwise as sgemm_f32.
 */
int sgemm_f32_streamk(int64_t M, int64_t N, int64_t K,
                      const float *A, int64_t lda,
                      const float *B, int64_t ldb,
                      float *C, int64_t ldc,
                      int transA, int transB,
                      void *workspace, uint64_t workspace_bytes, void *stream);

/* Workspace bytes for sgemm_f32_streamk on the current device: the turned
 * copies (K x round_up(M, 4) and/or K x round_up(N, 4) floats) and, when the
 * stream-K schedule applies, two partial tiles per SM (about 40 MB on
 * GB300); 0 when the call needs none. */
uint64_t sgemm_f32_streamk_workspace_size(int64_t M, int64_t N, int64_t K, int transA, int transB);

/* Number of K chunks chosen for splits = 0: enough 128 x 128 tiles to put one
 * CTA on every SM of the current device, each chunk at least 32 deep (one K
 * slice), at most 64; 1 when the tiles already fill the device. */
int sgemm_f32_splitk_auto_splits(int64_t M, int64_t N, int64_t K);

/* Workspace bytes for sgemm_f32_splitk (splits = 0: the automatic choice):
 * chunks * M * round_up(N, 4) floats plus padding; 0 when one chunk is used. */
uint64_t sgemm_f32_splitk_workspace_size(int64_t M, int64_t N, int64_t K, int splits);

/*
 * C = op(A) op(B) on the tensor cores with FP32 accuracy: every input is split
 * as x = hi + lo with hi = x cut to TF32 (its 13 low mantissa bits cleared:
 * the value a TF32 MMA reads from the fp32 word x) and lo = x - hi rounded to
 * TF32 (nearest), and the product is formed as lo_a*hi_b + hi_a*lo_b +
 * hi_a*hi_b (three TF32 MMAs per K step, tcgen05 with the accumulator in
 * tensor memory, fp32 accumulation).  The dropped lo_a*lo_b term and the TF32
 * rounding of lo are each below 2^-20 of |a||b| per product, so results meet
 * the same elementwise bound as
 * sgemm_f32; small-integer inputs are exact.  Not bit-identical to
 * sgemm_f32 (different summation order), deterministic across calls on the
 * same device with the same workspace size.
 * Defined by: "CUDA GEMM operator performance optimization", section 1.1
 * (GEMM); the TF32 accuracy trade-off it removes is the FMA vs TF32 RRMSE
 * comparison (1.03e-6 vs 7.78e-4) on the ChetanC28/cuda-kernels page.
 *
 * Arguments as sgemm_f32, plus a caller-owned DEVICE workspace of
 * sgemm_f32_tf32x3_workspace_size(M, N, K, 1) bytes, 256-byte aligned, not
 * overlapping A, B or C, and not used by other work while this call's
 * kernels run on `stream` (it holds the split operands).  A workspace of only
 * the planes' bytes (2 * (M + N) * round_up(K, 32) floats, each operand's
 * part rounded up to 256 bytes) is accepted too: the call then computes
 * every output tile whole, instead of splitting in K the tiles of a last
 * wave that would leave at least half the SMs idle, and those tiles' sums
 * may differ in the last bit.
 * SGEMM_EWORKSPACE if it is NULL, misaligned or smaller than the planes.
 */
int sgemm_f32_tf32x3(int64_t M, int64_t N, int64_t K,
                     const float *A, int64_t lda,
                     const float *B, int64_t ldb,
                     float *C, int64_t ldc,
                     int transA, int transB,
                     void *workspace, uint64_t workspace_bytes, void *stream);

/* sgemm_f32_tf32x3 with the epilogue of sgemm_f32_ex (alpha, beta, bias). */
int sgemm_f32_tf32x3_ex(int64_t M, int64_t N, int64_t K, float alpha,
                        const float *A, int64_t lda,
                        const float *B, int64_t ldb,
                        float beta, float *C, int64_t ldc,
                        const float *bias, int transA, int transB,
                        void *workspace, uint64_t workspace_bytes, void *stream);

/* Strided-batched form of sgemm_f32_tf32x3 (arguments as
 * sgemm_f32_strided_batched plus the workspace, sized for `batch`). */
int sgemm_f32_tf32x3_strided_batched(int64_t M, int64_t N, int64_t K,
                                     const float *A, int64_t lda, int64_t strideA,
                                     const float *B, int64_t ldb, int64_t strideB,
                                     float *C, int64_t ldc, int64_t strideC,
                                     int64_t batch, int transA, int transB,
                                     void *workspace, uint64_t workspace_bytes, void *stream);

/* Workspace bytes for the tf32x3 entry points on the current device: the hi
 * and lo TF32 planes of op(A) and op(B), 2 * batch * (M + N) * round_up(K, 32)
 * floats plus padding (an operand stored K-contiguous with aligned rows, 16
 * bytes for K <= 256 and 128 bytes above, is read as its own hi term and uses
 * only its lo plane, but the size does not depend on the pointers), then, for
 * K > 256 when the last wave of output tiles leaves at least half the SMs
 * idle, the partial tiles of those tiles' K segments (at most one 128 x 256
 * fp32 tile per SM, 19.9 MB on GB300).  0 for empty problems or negative
 * sizes. */
uint64_t sgemm_f32_tf32x3_workspace_size(int64_t M, int64_t N, int64_t K, int64_t batch);

/*
 * C = op(A) op(B) as ONE TF32 product per term: inputs rounded to TF32
 * (10 explicit mantissa bits, round to nearest), products summed in fp32 on
 * the tensor cores.  The fast, reduced-precision mode: each product carries a
 * relative error up to about 2^-10, so results are NOT held to the FP32
 * bound of the other entry points; the tests hold them to
 * |C - C_ref| <= 2e-3 * sum_k |a||b| + 1e-6 and report the RRMSE.  Inputs
 * that are exact in TF32 (e.g. small integers) give exact results.
 * Defined by: the TF32 tensor-core stage of the ChetanC28/cuda-kernels page
 * (19.12 TFLOP/s and RRMSE 7.78e-4 against 1.03e-6 for FMA on an RTX 4000
 * Ada), re-built on tcgen05.
 * Arguments as sgemm_f32_tf32x3; workspace of
 * sgemm_f32_tf32_workspace_size(M, N, K, batch) bytes (half of the split
 * product's).
 */
int sgemm_f32_tf32(int64_t M, int64_t N, int64_t K,
                   const float *A, int64_t lda,
                   const float *B, int64_t ldb,
                   float *C, int64_t ldc,
                   int transA, int transB,
                   void *workspace, uint64_t workspace_bytes, void *stream);

int sgemm_f32_tf32_strided_batched(int64_t M, int64_t N, int64_t K,
                                   const float *A, int64_t lda, int64_t strideA,
                                   const float *B, int64_t ldb, int64_t strideB,
                                   float *C, int64_t ldc, int64_t strideC,
                                   int64_t batch, int transA, int transB,
                                   void *workspace, uint64_t workspace_bytes, void *stream);

/* Workspace bytes of the sgemm_f32_tf32 entry points: batch * (M + N) *
 * round_up(K, 32) floats plus padding.  0 for empty problems. */
uint64_t sgemm_f32_tf32_workspace_size(int64_t M, int64_t N, int64_t K, int64_t batch);

/*
 * sgemm_f32_tf32x3 for callers that cannot allocate device memory: some hosts
 * own every byte of device memory themselves and forbid allocation inside the
 * callback that runs the GEMM (plugin and enqueue interfaces of inference
 * runtimes, for instance), and some latency-critical loops cannot afford
 * cudaMalloc, which may synchronise the device.  This entry point takes no
 * workspace and allocates nothing: the split TF32 operands go into a scratch
 * array of sgemm_f32_tf32x3_noalloc_max_bytes() bytes (64 MiB) that the
 * library reserves on every GPU that loads it, for the life of the process.
 * There is no counterpart on the source pages; it exists for these callers.
 *
 * Arguments, layout, precision and results as sgemm_f32_tf32x3 (no batch)
 * with a workspace of the scratch's size.
 * Limit: 2 * (M + N) * round_up(K, 32) * 4 bytes (plus 256-byte alignment
 * padding) must fit in the scratch, e.g. M = N = K = 2048; larger problems
 * return SGEMM_EWORKSPACE with the sizes in sgemm_last_error().  Where the
 * partial tiles of split tail tiles fit as well, the call splits them as
 * sgemm_f32_tf32x3 does.
 * The first call in each CUDA context (per device, and again after
 * cudaDeviceReset or when another context is made current) looks up the
 * scratch's device address (cudaGetSymbolAddress); make that first call
 * before any stream capture in that context.  Every call on a device shares
 * the one scratch
 * array: calls whose kernels can overlap on the GPU (different streams
 * without ordering between them) race on it and give wrong results.  The
 * scratch keeps the last call's contents; no call relies on it being zero.
 */
int sgemm_f32_tf32x3_noalloc(int64_t M, int64_t N, int64_t K,
                             const float *A, int64_t lda,
                             const float *B, int64_t ldb,
                             float *C, int64_t ldc,
                             int transA, int transB, void *stream);

/* Size in bytes of the built-in scratch of sgemm_f32_tf32x3_noalloc. */
uint64_t sgemm_f32_tf32x3_noalloc_max_bytes(void);

/*
 * Reads (and with reset != 0 clears) the library's device status word on the
 * current device.  Bit 0 set: a tensor-core kernel gave up on a pipeline wait
 * that exceeded its time limit (about 2 s); that call's C is not valid.
 * Synchronises the device.  Returns an sgemm_status.
 */
int sgemm_device_status(unsigned int *flags, int reset);

/* Text for a status code (static storage). */
const char *sgemm_status_string(int status);

/* Detail of the last failed call on the calling host thread ("" if none).
 * The pointer stays valid until the next call on this thread. */
const char *sgemm_last_error(void);

/* Library version as 10000*major + 100*minor + patch. */
int sgemm_version(void);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_GB300_H */
