// Split-K for the SIMT kernel: small or skinny problems whose output tiles
// cannot fill the GPU (a 128 x 128 x 32768 product is one tile: one SM of 152)
// split K into chunks, each chunk a separate problem of the batched kernel
// writing a partial plane, then one pass sums the planes into C.  The sum
// runs over the chunks in a fixed order, so results are deterministic, and
// exact whenever every partial sum is (e.g. small integers).
// After the split-K stage of the ChetanC28/cuda-kernels page (splitting K
// across blocks and reducing afterwards, 28.87x on 128 x 128 x 32768).
#include <cstdint>

#include <cuda_runtime.h>

#include "gemm_args.h"

namespace sgemm {
namespace {

constexpr int kChunkAlign = 32;       // whole K slices of the SIMT kernel
// One 32-deep slice per chunk at least: on GB300 the reduction pass is cheap
// next to an idle SM (256 x 256 x 256: 8 chunks 12.4 us against 20.6 us for 2;
// 256 x 256 x 4096: 32 chunks 22.7 us against 31.8 us for 16).
constexpr int kMinChunk = 32;
constexpr int kMaxAutoSplits = 64;

int64_t padded_n(int64_t N) { return (N + 3) / 4 * 4; }

int64_t chunk_len(int64_t K, int splits) {
    return ((K + splits - 1) / splits + kChunkAlign - 1) / kChunkAlign * kChunkAlign;
}

// C[i][j] = sum over s = 0..S-1 of P[s][i][j], planes of M x Np floats: one
// thread per float4 of C, the planes added in ascending s (few planes).
__global__ void splitk_reduce_kernel(const float *__restrict__ P, int S, int M, int N, int64_t Np,
                                     float *__restrict__ C, int64_t ldc, int vec) {
    const int64_t plane = (int64_t)M * Np;
    const int64_t groups = Np / 4;
    const int64_t total = (int64_t)M * groups;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
         t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = t / groups;
        const int j = (int)(t - i * groups) * 4;
        const float *p = P + i * Np + j;
        float4 acc = *reinterpret_cast<const float4 *>(p);
        for (int s = 1; s < S; ++s) {
            const float4 v = *reinterpret_cast<const float4 *>(p + s * plane);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        float *c = C + i * ldc + j;
        const bool full = vec && j + 3 < N;
        if (full) {
            *reinterpret_cast<float4 *>(c) = acc;
        } else {
            if (j + 0 < N) c[0] = acc.x;
            if (j + 1 < N) c[1] = acc.y;
            if (j + 2 < N) c[2] = acc.z;
            if (j + 3 < N) c[3] = acc.w;
        }
    }
}

constexpr int kWideSlots = 8;   // threads sharing one float4 of C in the many-plane form

// The same sum for many planes (one tile split 64 ways: the single-thread
// form reads 64 planes in sequence from only 16 CTAs): 8 threads share each
// float4 of C, slot w adding planes w, w + 8, ... in ascending order, and slot
// 0 then adds the 8 slot sums in slot order.  A fixed order: deterministic.
__global__ void __launch_bounds__(256)
splitk_reduce_wide_kernel(const float *__restrict__ P, int S, int M, int N, int64_t Np,
                          float *__restrict__ C, int64_t ldc, int vec) {
    constexpr int G = 256 / kWideSlots;   // float4 groups of C per CTA
    __shared__ float4 part[256];
    const int g = threadIdx.x % G, w = threadIdx.x / G;
    const int64_t plane = (int64_t)M * Np;
    const int64_t e = ((int64_t)blockIdx.x * G + g) * 4;   // element index in a plane
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (e < plane) {
#pragma unroll 4
        for (int s = w; s < S; s += kWideSlots) {
            const float4 v = *reinterpret_cast<const float4 *>(P + s * plane + e);
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
    }
    part[threadIdx.x] = acc;
    __syncthreads();
    if (w != 0 || e >= plane) return;
    for (int k = 1; k < kWideSlots; ++k) {
        const float4 v = part[k * G + g];
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
    }
    const int64_t i = e / Np;
    const int j = (int)(e - i * Np);
    float *c = C + i * ldc + j;
    const bool full = vec && j + 3 < N;
    if (full) {
        *reinterpret_cast<float4 *>(c) = acc;
    } else {
        if (j + 0 < N) c[0] = acc.x;
        if (j + 1 < N) c[1] = acc.y;
        if (j + 2 < N) c[2] = acc.z;
        if (j + 3 < N) c[3] = acc.w;
    }
}

int sms_on_current_device() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
    return sms > 0 ? sms : 1;
}

}  // namespace

int splitk_auto_splits(int64_t M, int64_t N, int64_t K) {
    const int64_t tiles = ((M + 127) / 128) * ((N + 127) / 128);
    const int64_t sms = sms_on_current_device();
    if (tiles >= sms) return 1;
    int64_t s = sms / tiles;
    const int64_t by_k = K / kMinChunk;
    if (s > by_k) s = by_k;
    if (s > kMaxAutoSplits) s = kMaxAutoSplits;
    return s < 1 ? 1 : (int)s;
}

size_t splitk_workspace_bytes(int64_t M, int64_t N, int64_t K, int splits) {
    if (splits < 1) splits = 1;
    const int64_t chunk = chunk_len(K, splits);
    const int64_t used = (K + chunk - 1) / chunk;
    if (used <= 1) return 0;
    const size_t bytes = (size_t)used * (size_t)M * (size_t)padded_n(N) * sizeof(float);
    return (bytes + 255) / 256 * 256;
}

cudaError_t launch_simt_splitk(const GemmArgs &a, bool transA, bool transB, bool vec, int splits,
                               void *ws, cudaStream_t s) {
    const int64_t chunk = chunk_len(a.K, splits);
    const int used = (int)((a.K + chunk - 1) / chunk);
    const int64_t Np = padded_n(a.N);
    GemmArgs g = a;
    g.batch = used;
    g.kchunk = (int)chunk;
    g.strideA = transA ? chunk * a.lda : chunk;
    g.strideB = transB ? chunk : chunk * a.ldb;
    g.C = static_cast<float *>(ws);
    g.ldc = Np;
    g.strideC = (int64_t)a.M * Np;
    cudaError_t e = launch_simt(g, transA, transB, vec, s);
    if (e != cudaSuccess) return e;
    const int vec_c = (reinterpret_cast<uintptr_t>(a.C) % 16 == 0) && a.ldc % 4 == 0;
    const float *P = static_cast<const float *>(ws);
    if (used <= kWideSlots) {
        // measured: with 2-8 planes the single-thread form is fastest
        const int64_t total = (int64_t)a.M * (Np / 4);
        const int64_t want = (total + 255) / 256;
        const int blocks = (int)(want < 152 * 16 ? want : 152 * 16);
        splitk_reduce_kernel<<<blocks, 256, 0, s>>>(P, used, a.M, a.N, Np, a.C, a.ldc, vec_c);
    } else {
        const int64_t groups = ((int64_t)a.M * Np / 4 + 31) / 32;
        if (groups > 0x7fffffff) return cudaErrorInvalidValue;
        splitk_reduce_wide_kernel<<<(unsigned)groups, 256, 0, s>>>(P, used, a.M, a.N, Np, a.C,
                                                                   a.ldc, vec_c);
    }
    return cudaGetLastError();
}

}  // namespace sgemm
