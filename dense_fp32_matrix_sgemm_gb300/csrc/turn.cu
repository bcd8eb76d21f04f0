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

// The same copy with 16-byte aligned rows (X, ldx, Y, ldy all allow it):
// 32 x 128 blocks of X, each thread loading four 16-byte row segments (4
// consecutive c) and storing four 16-byte segments of Y rows (4 consecutive
// r), through a shared tile of row stride 129 floats whose reads
// (tile[4q + e][c], q = thread % 8, c = thread / 8 + 32 i) fall in 32
// distinct banks.  A quad of Y past `rows` (inside ldy, which is a multiple
// of 4) gets zeros.
__global__ void __launch_bounds__(256) transpose_vec_kernel(const float *__restrict__ X,
                                                            int64_t ldx, int rows, int cols,
                                                            float *__restrict__ Y, int64_t ldy) {
    __shared__ float tile[32][129];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x;
    const int lc = 4 * (tid & 31), lr = tid >> 5;   // load: c quad, row (0..7)
    const int q = tid & 7, sc = tid >> 3;           // store: r quad, Y row (0..31)
    const int64_t tiles_c = (cols + 127) / 128, tiles_r = (rows + 31) / 32;
    for (int64_t t = blockIdx.x; t < tiles_c * tiles_r; t += gridDim.x) {
        const int r0 = (int)(t / tiles_c) * 32, c0 = (int)(t % tiles_c) * 128;
        float4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = r0 + lr + 8 * i, c = c0 + lc;
            v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < rows) {
                const float *src = X + (int64_t)r * ldx + c;
                if (c + 3 < cols) {
                    v[i] = *reinterpret_cast<const float4 *>(src);
                } else {
                    if (c + 0 < cols) v[i].x = src[0];
                    if (c + 1 < cols) v[i].y = src[1];
                    if (c + 2 < cols) v[i].z = src[2];
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float *trow = tile[lr + 8 * i] + lc;
            trow[0] = v[i].x;
            trow[1] = v[i].y;
            trow[2] = v[i].z;
            trow[3] = v[i].w;
        }
        __syncthreads();
        const int r = r0 + 4 * q;
        if (r < rows) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int cc = sc + 32 * i, c = c0 + cc;
                if (c < cols)
                    *reinterpret_cast<float4 *>(Y + (int64_t)c * ldy + r) =
                        make_float4(tile[4 * q][cc], tile[4 * q + 1][cc], tile[4 * q + 2][cc],
                                    tile[4 * q + 3][cc]);
            }
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_transpose(const float *X, int64_t ldx, int rows, int cols, float *Y, int64_t ldy,
                             cudaStream_t s) {
    const bool vec = reinterpret_cast<uintptr_t>(X) % 16 == 0 && ldx % 4 == 0 &&
                     reinterpret_cast<uintptr_t>(Y) % 16 == 0 && ldy % 4 == 0;
    const int64_t tiles = vec ? ((int64_t)(rows + 31) / 32) * ((cols + 127) / 128)
                              : ((int64_t)(rows + 63) / 64) * ((cols + 31) / 32);
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess)
        (void)cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t wave = (int64_t)sms * (vec ? 6 : 8);   // CTAs of 256 threads resident per SM
    const int blocks = (int)(tiles < wave ? tiles : wave);
    if (vec)
        transpose_vec_kernel<<<blocks, 256, 0, s>>>(X, ldx, rows, cols, Y, ldy);
    else
        transpose_kernel<<<blocks, 256, 0, s>>>(X, ldx, rows, cols, Y, ldy);
    return cudaGetLastError();
}

}  // namespace sgemm
