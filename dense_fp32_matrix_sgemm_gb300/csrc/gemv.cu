// Degenerate GEMM shapes: matrix times vector.  When N == 1 (op(B) is a
// column) or M == 1 (op(A) is a row) every element of the matrix operand is
// used once, so the product is bound by reading that matrix from HBM
// (arithmetic intensity about 0.5 FLOP/B), not by the FMA units; the tile
// kernel would waste 127 of every 128 columns of its tiles.  Two kernels,
// after the thread-per-row and warp-per-row matrix-vector kernels of the
// DD2360 workbook, section 15.2:
//   * dot:    one warp per output, the matrix row contiguous along K (16-byte
//             loads when aligned), a butterfly shuffle sum;
//   * colsum: one thread per output (four with 16-byte loads), the matrix
//             contiguous along the outputs, K split over 8 warps whose partial
//             sums are added in warp order through shared memory.
// Both sum in a fixed order: results are deterministic.  The epilogue of
// sgemm_f32_ex (alpha, beta, bias) is applied on the store.
#include <cstdint>

#include <cuda_runtime.h>

#include "gemm_args.h"

namespace sgemm {
namespace {

// Shared epilogue: y = alpha * acc + beta * y_old + bias.
__device__ __forceinline__ float epilogue(float acc, float *y, float alpha, float beta,
                                          const float *bias, int64_t bias_index, bool plain) {
    if (plain) return acc;
    const float old = beta != 0.f ? *y : 0.f;
    const float b = bias != nullptr ? bias[bias_index] : 0.f;
    return fmaf(beta, old, alpha * acc) + b;
}

struct GemvArgs {
    const float *X;    // matrix operand
    int64_t ldx, sX;   // dot: row stride (K-contiguous rows); colsum: stride between k rows
    const float *v;    // vector operand, element k at v[k * incv]
    int64_t incv, sV;
    float *y;          // output, element r at y[r * incy]
    int64_t incy, sY;
    int R, K, batch;   // R outputs per problem
    float alpha, beta;
    const float *bias;
    int64_t bias_inc;  // bias index = r * bias_inc (0: one bias value for all outputs)
};

template <bool VEC>
__global__ void gemv_dot_kernel(const GemvArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const bool plain = a.alpha == 1.f && a.beta == 0.f && a.bias == nullptr;
    for (int64_t w = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5);
         w < (int64_t)a.batch * a.R; w += warps) {
        const int64_t z = w / a.R, r = w - z * a.R;
        const float *x = a.X + z * a.sX + r * a.ldx;
        const float *v = a.v + z * a.sV;
        float acc = 0.f;
        if constexpr (VEC) {
            int k = 4 * lane;
#pragma unroll 4
            for (; k + 3 < a.K; k += 128) {
                const float4 xv = __ldg(reinterpret_cast<const float4 *>(x + k));
                const float4 vv = __ldg(reinterpret_cast<const float4 *>(v + k));
                acc = fmaf(xv.x, vv.x, acc);
                acc = fmaf(xv.y, vv.y, acc);
                acc = fmaf(xv.z, vv.z, acc);
                acc = fmaf(xv.w, vv.w, acc);
            }
            // the < 4 elements past the last whole float4 group
            for (k = (a.K & ~3) + lane; k < a.K; k += 32) acc = fmaf(__ldg(x + k), __ldg(v + k), acc);
        } else {
            for (int k = lane; k < a.K; k += 32) acc = fmaf(__ldg(x + k), __ldg(v + k * a.incv), acc);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) {
            float *y = a.y + z * a.sY + r * a.incy;
            *y = epilogue(acc, y, a.alpha, a.beta, a.bias, r * a.bias_inc, plain);
        }
    }
}

constexpr int kColsumSplit = 8;   // warps splitting K in one block

template <bool VEC>
__global__ void __launch_bounds__(32 * kColsumSplit)
gemv_colsum_kernel(const GemvArgs a) {
    constexpr int PER = VEC ? 4 : 1;                 // outputs per thread
    __shared__ float part[kColsumSplit][32 * PER];
    const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
    const int z = blockIdx.y;
    const int64_t r0 = (int64_t)blockIdx.x * 32 * PER + PER * lane;
    const float *X = a.X + (int64_t)z * a.sX;
    const float *v = a.v + (int64_t)z * a.sV;
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    // warp wp takes k = wp, wp + 8, ...
    if (r0 < a.R) {
#pragma unroll 4
        for (int k = wp; k < a.K; k += kColsumSplit) {
            const float vk = __ldg(v + k * a.incv);
            const float *row = X + (int64_t)k * a.ldx + r0;
            if constexpr (VEC) {
                if (r0 + 3 < a.R) {
                    const float4 xv = __ldg(reinterpret_cast<const float4 *>(row));
                    acc[0] = fmaf(xv.x, vk, acc[0]);
                    acc[1] = fmaf(xv.y, vk, acc[1]);
                    acc[2] = fmaf(xv.z, vk, acc[2]);
                    acc[3] = fmaf(xv.w, vk, acc[3]);
                } else {
#pragma unroll
                    for (int e = 0; e < PER; ++e)
                        if (r0 + e < a.R) acc[e] = fmaf(__ldg(row + e), vk, acc[e]);
                }
            } else {
                acc[0] = fmaf(__ldg(row), vk, acc[0]);
            }
        }
    }
#pragma unroll
    for (int e = 0; e < PER; ++e) part[wp][PER * lane + e] = acc[e];
    __syncthreads();
    if (wp == 0) {
        const bool plain = a.alpha == 1.f && a.beta == 0.f && a.bias == nullptr;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const int64_t r = r0 + e;
            if (r >= a.R) continue;
            float s = part[0][PER * lane + e];
#pragma unroll
            for (int w = 1; w < kColsumSplit; ++w) s += part[w][PER * lane + e];
            float *y = a.y + (int64_t)z * a.sY + r * a.incy;
            *y = epilogue(s, y, a.alpha, a.beta, a.bias, r * a.bias_inc, plain);
        }
    }
}

bool aligned16(const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

cudaError_t launch_dot(const GemvArgs &g, cudaStream_t s) {
    const bool vec = aligned16(g.X) && g.ldx % 4 == 0 && g.sX % 4 == 0 && g.incv == 1 &&
                     aligned16(g.v) && g.sV % 4 == 0;
    const int64_t warps = (int64_t)g.batch * g.R;
    const int64_t want = (warps + 7) / 8;
    const int blocks = (int)(want < 152 * 64 ? want : 152 * 64);
    if (vec)
        gemv_dot_kernel<true><<<blocks, 256, 0, s>>>(g);
    else
        gemv_dot_kernel<false><<<blocks, 256, 0, s>>>(g);
    return cudaGetLastError();
}

cudaError_t launch_colsum(const GemvArgs &g, cudaStream_t s) {
    const bool vec = aligned16(g.X) && g.ldx % 4 == 0 && g.sX % 4 == 0 && g.incy == 1;
    const int per = vec ? 4 : 1;
    if (g.batch > 65535) return cudaErrorInvalidValue;
    dim3 grid((unsigned)((g.R + 32 * per - 1) / (32 * per)), (unsigned)g.batch);
    if (vec)
        gemv_colsum_kernel<true><<<grid, 32 * kColsumSplit, 0, s>>>(g);
    else
        gemv_colsum_kernel<false><<<grid, 32 * kColsumSplit, 0, s>>>(g);
    return cudaGetLastError();
}

}  // namespace

bool gemv_shape(const GemmArgs &a) { return (a.N == 1 || a.M == 1) && a.batch <= 65535; }

cudaError_t launch_gemv(const GemmArgs &a, bool transA, bool transB, cudaStream_t s) {
    GemvArgs g;
    g.K = a.K;
    g.batch = a.batch;
    g.alpha = a.alpha;
    g.beta = a.beta;
    g.bias = a.bias;
    g.y = a.C;
    g.sY = a.strideC;
    if (a.N == 1) {
        // c_i = sum_k opA(i, k) * opB(k, 0): outputs along M, C[i * ldc]
        g.R = a.M;
        g.incy = a.ldc;
        g.bias_inc = 0;
        g.X = a.A;
        g.sX = a.strideA;
        g.ldx = a.lda;
        g.v = a.B;
        g.sV = a.strideB;
        g.incv = transB ? 1 : a.ldb;
        return transA ? launch_colsum(g, s) : launch_dot(g, s);
    }
    // M == 1: c_j = sum_k opA(0, k) * opB(k, j): outputs along N, C[j]
    g.R = a.N;
    g.incy = 1;
    g.bias_inc = 1;
    g.X = a.B;
    g.sX = a.strideB;
    g.ldx = a.ldb;
    g.v = a.A;
    g.sV = a.strideA;
    g.incv = transA ? a.lda : 1;
    return transB ? launch_dot(g, s) : launch_colsum(g, s);
}

}  // namespace sgemm
