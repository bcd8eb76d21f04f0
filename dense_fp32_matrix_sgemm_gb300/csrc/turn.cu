// Exact fp32 transpose used to turn a K-contiguous operand (row-major A, or
// B stored transposed) into an M/N-contiguous copy in a caller workspace, so
// the tile kernel streams both operands with 16-byte cp.async instead of
// corner-turning one through registers (sgemm_f32_streamk).  A 32 x 33
// shared tile makes both the read and the write coalesced.
#include <cstdint>

#include <cuda_runtime.h>

#include "gemm_args.h"

namespace sgemm {
namespace {

// Y[c * ldy + r] = X[r * ldx + c] for r < rows, c < cols.
__global__ void __launch_bounds__(256) transpose_kernel(const float *__restrict__ X, int64_t ldx,
                                                        int rows, int cols, float *__restrict__ Y,
                                                        int64_t ldy) {
    __shared__ float tile[32][33];
    // the tile kernel that reads the copy may start its set-up meanwhile
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8
    const int64_t tiles_c = (cols + 31) / 32, tiles_r = (rows + 31) / 32;
    for (int64_t t = blockIdx.x; t < tiles_c * tiles_r; t += gridDim.x) {
        const int r0 = (int)(t / tiles_c) * 32, c0 = (int)(t % tiles_c) * 32;
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
            const int r = r0 + ty + i, c = c0 + tx;
            if (r < rows && c < cols) tile[ty + i][tx] = X[(int64_t)r * ldx + c];
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
            const int c = c0 + ty + i, r = r0 + tx;
            if (r < rows && c < cols) Y[(int64_t)c * ldy + r] = tile[tx][ty + i];
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_transpose(const float *X, int64_t ldx, int rows, int cols, float *Y, int64_t ldy,
                             cudaStream_t s) {
    const int64_t tiles = ((int64_t)(rows + 31) / 32) * ((cols + 31) / 32);
    const int blocks = (int)(tiles < 152 * 16 ? tiles : 152 * 16);
    transpose_kernel<<<blocks, 256, 0, s>>>(X, ldx, rows, cols, Y, ldy);
    return cudaGetLastError();
}

}  // namespace sgemm
