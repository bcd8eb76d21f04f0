// Degenerate GEMM shapes: matrix times vector.  When N == 1 (op(B) is a
// column) or M == 1 (op(A) is a row) every element of the matrix operand is
// used once, so the product is bound by reading that matrix from HBM
// (arithmetic intensity about 0.5 FLOP/B), not by the FMA units; the tile
// kernel would waste 127 of every 128 columns of its tiles.  Two kernels,
// after the thread-per-row and warp-per-row matrix-vector kernels of the
// DD2360 workbook, section 15.2:
//   * dot:    one warp per two outputs, the matrix rows contiguous along K
//             (16-byte streaming loads that skip L1 when aligned, so the
//             vector stays cached), a butterfly shuffle sum per row;
//   * colsum: one thread per output (four with 16-byte loads), the matrix
//             contiguous along the outputs; K split over the CS CTAs of a
//             cluster (contiguous ranges) and, inside each, over 8 warps.  The
//             warps' partial sums are added in warp order through shared
//             memory, then the CTAs' in rank order through distributed shared
//             memory: a few hundred CTAs instead of one per 128 outputs, with
//             no workspace.
// Both sum in a fixed order: results are deterministic.  The epilogue of
// sgemm_f32_ex (alpha, beta, bias) is applied on the store.
#include <cstdint>

#include <cuda_runtime.h>

#include "device_utils.cuh"
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

// 16-byte load of matrix data that is read once: bypasses L1 so the vector,
// read by every warp, stays there.
__device__ __forceinline__ float4 ld_stream_f4(const float *p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

constexpr int kDotRows = 2;   // outputs per warp: two rows share each vector load

template <bool VEC>
__global__ void gemv_dot_kernel(const GemvArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const bool plain = a.alpha == 1.f && a.beta == 0.f && a.bias == nullptr;
    const int64_t pairs = ((int64_t)a.R + kDotRows - 1) / kDotRows;   // per problem
    for (int64_t w = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5);
         w < (int64_t)a.batch * pairs; w += warps) {
        const int64_t z = w / pairs, r0 = (w - z * pairs) * kDotRows;
        const int rows = (int)min((int64_t)kDotRows, (int64_t)a.R - r0);   // 1 or 2, warp-uniform
        const float *x0 = a.X + z * a.sX + r0 * a.ldx;
        const float *x1 = rows > 1 ? x0 + a.ldx : x0;   // row 1 absent: reread row 0, discard
        const float *v = a.v + z * a.sV;
        float acc0 = 0.f, acc1 = 0.f;
        if constexpr (VEC) {
            int k = 4 * lane;
#pragma unroll 4
            for (; k + 3 < a.K; k += 128) {
                const float4 vv = __ldg(reinterpret_cast<const float4 *>(v + k));
                const float4 p = ld_stream_f4(x0 + k);
                const float4 q = ld_stream_f4(x1 + k);
                acc0 = fmaf(p.x, vv.x, acc0);
                acc0 = fmaf(p.y, vv.y, acc0);
                acc0 = fmaf(p.z, vv.z, acc0);
                acc0 = fmaf(p.w, vv.w, acc0);
                acc1 = fmaf(q.x, vv.x, acc1);
                acc1 = fmaf(q.y, vv.y, acc1);
                acc1 = fmaf(q.z, vv.z, acc1);
                acc1 = fmaf(q.w, vv.w, acc1);
            }
            // the < 4 elements past the last whole float4 group
            for (k = (a.K & ~3) + lane; k < a.K; k += 32) {
                const float vk = __ldg(v + k);
                acc0 = fmaf(__ldg(x0 + k), vk, acc0);
                acc1 = fmaf(__ldg(x1 + k), vk, acc1);
            }
        } else {
            for (int k = lane; k < a.K; k += 32) {
                const float vk = __ldg(v + k * a.incv);
                acc0 = fmaf(__ldg(x0 + k), vk, acc0);
                acc1 = fmaf(__ldg(x1 + k), vk, acc1);
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            acc0 += __shfl_xor_sync(0xffffffffu, acc0, off);
            acc1 += __shfl_xor_sync(0xffffffffu, acc1, off);
        }
        if (lane == 0) {
            float *y = a.y + z * a.sY + r0 * a.incy;
            *y = epilogue(acc0, y, a.alpha, a.beta, a.bias, r0 * a.bias_inc, plain);
            if (rows > 1) {
                y += a.incy;
                *y = epilogue(acc1, y, a.alpha, a.beta, a.bias, (r0 + 1) * a.bias_inc, plain);
            }
        }
    }
}

// Column sums: two 16-byte loads per thread per k (a warp reads 1 KB of a
// matrix row), 16 or 32 warps splitting K inside a CTA, clusters of up to 8
// CTAs splitting it further.  Measured on 8192 x 8192: 512-byte segments
// reached 3.6 TB/s, 1 KB segments 5.6 TB/s.
constexpr int kColsumVecs = 2;
constexpr int kColsumUnroll = 4;

// NV: 16-byte loads per thread per k when VEC (4 * NV consecutive outputs per
// thread, so a warp reads 512 * NV contiguous bytes of each matrix row).
template <bool VEC, int NV, int SPLIT, int UNROLL>
__global__ void __launch_bounds__(32 * SPLIT)
gemv_colsum_kernel(const GemvArgs a) {
    constexpr int PER = VEC ? 4 * NV : 1;            // outputs per thread
    __shared__ __align__(16) float part[SPLIT][32 * PER];
    const int lane = threadIdx.x & 31, wp = threadIdx.x >> 5;
    const int z = blockIdx.y;
    const uint32_t q = cluster_rank(), cs = cluster_size();
    const int64_t r0 = (int64_t)(blockIdx.x / cs) * 32 * PER + PER * lane;
    // CTA q of the cluster takes k in [k_lo, k_hi)
    const int k_lo = (int)((int64_t)a.K * q / cs), k_hi = (int)((int64_t)a.K * (q + 1) / cs);
    const float *X = a.X + (int64_t)z * a.sX;
    const float *v = a.v + (int64_t)z * a.sV;
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    // warp wp takes k = k_lo + wp, k_lo + wp + SPLIT, ...
    if (r0 < a.R) {
#pragma unroll UNROLL
        for (int k = k_lo + wp; k < k_hi; k += SPLIT) {
            const float vk = __ldg(v + k * a.incv);
            const float *row = X + (int64_t)k * a.ldx + r0;
            if constexpr (VEC) {
                if (r0 + PER - 1 < a.R) {
#pragma unroll
                    for (int j = 0; j < NV; ++j) {
                        const float4 xv = ld_stream_f4(row + 4 * j);
                        acc[4 * j + 0] = fmaf(xv.x, vk, acc[4 * j + 0]);
                        acc[4 * j + 1] = fmaf(xv.y, vk, acc[4 * j + 1]);
                        acc[4 * j + 2] = fmaf(xv.z, vk, acc[4 * j + 2]);
                        acc[4 * j + 3] = fmaf(xv.w, vk, acc[4 * j + 3]);
                    }
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
    // this CTA's partial sums over its warps, in warp order, into part[0]
    if (wp == 0) {
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            float s = part[0][PER * lane + e];
#pragma unroll
            for (int w = 1; w < SPLIT; ++w) s += part[w][PER * lane + e];
            part[0][PER * lane + e] = s;
        }
    }
    cluster_sync();
    // CTA 0 adds the cluster's partials in rank order and stores
    if (q == 0 && wp == 0) {
        const bool plain = a.alpha == 1.f && a.beta == 0.f && a.bias == nullptr;
        const uint32_t at = smem_u32(&part[0][PER * lane]);
        float sum[PER];
        if constexpr (VEC) {
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                const float4 t = cluster_sum_f4(at + 16 * j, cs);
                sum[4 * j + 0] = t.x;
                sum[4 * j + 1] = t.y;
                sum[4 * j + 2] = t.z;
                sum[4 * j + 3] = t.w;
            }
        } else {
            sum[0] = cluster_sum_f32(at, cs);
        }
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const int64_t r = r0 + e;
            if (r >= a.R) continue;
            float *y = a.y + (int64_t)z * a.sY + r * a.incy;
            *y = epilogue(sum[e], y, a.alpha, a.beta, a.bias, r * a.bias_inc, plain);
        }
    }
    // no CTA leaves while CTA 0 still reads its shared memory
    cluster_sync_relaxed();
}

bool aligned16(const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

cudaError_t launch_dot(const GemvArgs &g, cudaStream_t s) {
    const bool vec = aligned16(g.X) && g.ldx % 4 == 0 && g.sX % 4 == 0 && g.incv == 1 &&
                     aligned16(g.v) && g.sV % 4 == 0;
    const int64_t warps = (int64_t)g.batch * ((g.R + kDotRows - 1) / kDotRows);
    const int64_t want = (warps + 7) / 8;
    const int blocks = (int)(want < 152 * 64 ? want : 152 * 64);
    if (vec)
        gemv_dot_kernel<true><<<blocks, 256, 0, s>>>(g);
    else
        gemv_dot_kernel<false><<<blocks, 256, 0, s>>>(g);
    return cudaGetLastError();
}

template <int NV, int SPLIT, int UNROLL>
cudaError_t launch_colsum_cfg(const GemvArgs &g, bool vec, cudaStream_t s) {
    const int per = vec ? 4 * NV : 1;
    if (g.batch > 65535) return cudaErrorInvalidValue;
    // clusters of 8 CTAs along K while every warp still gets 8 or more rows
    const int64_t col_blocks = ((int64_t)g.R + 32 * per - 1) / (32 * per);
    int cs = 8;
    while (cs > 1 && (int64_t)g.K < 8LL * SPLIT * cs) cs /= 2;
    cudaError_t e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(col_blocks * cs), (unsigned)g.batch);
    cfg.blockDim = dim3(32 * SPLIT);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (vec)
        e = cudaLaunchKernelEx(&cfg, gemv_colsum_kernel<true, NV, SPLIT, UNROLL>, g);
    else
        e = cudaLaunchKernelEx(&cfg, gemv_colsum_kernel<false, NV, SPLIT, UNROLL>, g);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// 16 warps per CTA when clusters of 8 put a CTA on at least three quarters of
// the SMs, else 32 (more loads in flight per SM on narrow problems; measured:
// 4096 outputs x 16384 prefer 16, 3072 x 8192 and 1000 x 8192 prefer 32).
cudaError_t launch_colsum(const GemvArgs &g, cudaStream_t s) {
    const bool vec = aligned16(g.X) && g.ldx % 4 == 0 && g.sX % 4 == 0 && g.incy == 1;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int per = vec ? 4 * kColsumVecs : 1;
    const int64_t col_blocks = ((int64_t)g.R + 32 * per - 1) / (32 * per);
    if (col_blocks * g.batch * 8 * 4 >= 3LL * sms)
        return launch_colsum_cfg<kColsumVecs, 16, kColsumUnroll>(g, vec, s);
    return launch_colsum_cfg<kColsumVecs, 32, kColsumUnroll>(g, vec, s);
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
