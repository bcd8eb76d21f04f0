// Exact fp32 transpose used to turn a K-contiguous operand (row-major A, or
// B stored transposed) into an M/N-contiguous copy in a caller workspace, so
// the tile kernel streams both operands with 16-byte cp.async instead of
// corner-turning one through registers (sgemm_f32_streamk).  A padded
// shared tile makes both the read and the write coalesced.
#include <cstdint>

#include <cuda_runtime.h>

#include "gemm_args.h"

namespace sgemm {
namespace {

// Y[c * ldy + r] = X[r * ldx + c] for r < rows, c < cols.  Each CTA moves
// 64 x 32 blocks of X through a padded shared tile: 8 loads per thread in
// flight before the barrier (enough bytes in flight per SM to cover the HBM
// latency), rows of 128 bytes read and written by every warp.
__global__ void __launch_bounds__(256) transpose_kernel(const float *__restrict__ X, int64_t ldx,
                                                        int rows, int cols, float *__restrict__ Y,
                                                        int64_t ldy) {
    __shared__ float tile[64][33];
    // the tile kernel that reads the copy may start its set-up meanwhile
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8
    const int64_t tiles_c = (cols + 31) / 32, tiles_r = (rows + 63) / 64;
    for (int64_t t = blockIdx.x; t < tiles_c * tiles_r; t += gridDim.x) {
        const int r0 = (int)(t / tiles_c) * 64, c0 = (int)(t % tiles_c) * 32;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = r0 + ty + 8 * i, c = c0 + tx;
            v[i] = (r < rows && c < cols) ? X[(int64_t)r * ldx + c] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) tile[ty + 8 * i][tx] = v[i];
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            // Y row c0 + ty + 8 (i % 4), columns r0 + tx + 32 (i / 4)
            const int c = c0 + ty + 8 * (i & 3), r = r0 + tx + 32 * (i >> 2);
            if (r < rows && c < cols) Y[(int64_t)c * ldy + r] = tile[tx + 32 * (i >> 2)][ty + 8 * (i & 3)];
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_transpose(const float *X, int64_t ldx, int rows, int cols, float *Y, int64_t ldy,
                             cudaStream_t s) {
    const int64_t tiles = ((int64_t)(rows + 63) / 64) * ((cols + 31) / 32);
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess)
        (void)cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t wave = (int64_t)sms * 8;   // 8 CTAs of 256 threads per SM
    const int blocks = (int)(tiles < wave ? tiles : wave);
    transpose_kernel<<<blocks, 256, 0, s>>>(X, ldx, rows, cols, Y, ldy);
    return cudaGetLastError();
}

}  // namespace sgemm
