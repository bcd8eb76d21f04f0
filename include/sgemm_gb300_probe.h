/*
 * sgemm_gb300_probe.h -- measuring the FP32 and TF32 peaks that SGEMM's
 * throughput is compared with.
 *
 * The peak of a GPU's FP32 units is cores x 2 FLOP (one FMA) x clock
 * (DD2360 workbook, section 3, worked example on the T4's FP32 peak).  This
 * probe measures it instead of assuming it: every thread runs 16 independent
 * FMA chains held in registers, no memory traffic, on a grid of 8 CTAs of 256
 * threads per SM.  The caller times the launch (e.g. with CUDA events on
 * `stream`) and divides *flops_out by the time.
 */
#ifndef SGEMM_GB300_PROBE_H
#define SGEMM_GB300_PROBE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The library is built with hidden symbol visibility; only the entry points
 * declared here are exported. */
#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

/*
 * Launch the FP32 FMA probe on `stream` (cudaStream_t as void*).
 *   packed      0: scalar fma.rn.f32;  1: packed fma.rn.f32x2 (two FMAs per
 *               instruction, sm_100 and newer).
 *   iterations  loop trips per thread (> 0); each trip does 32 FMAs per thread.
 *   out         device buffer of at least sgemm_probe_out_elems() floats,
 *               owned by the caller; receives one value per thread (the
 *               chains converge to 1.0, a check that the work was done).
 *   flops_out   host pointer; receives the FLOPs of one launch (2 per FMA).
 * Returns an sgemm_status (SGEMM_EINVAL_* on bad arguments, SGEMM_ELAUNCH,
 * SGEMM_EDEVICE); asynchronous like every call of the library.
 */
int sgemm_probe_fp32_fma(int packed, int64_t iterations, float *out, double *flops_out,
                         void *stream);

/* Number of floats `out` must hold on the current device. */
int64_t sgemm_probe_out_elems(void);

/*
 * Launch the TF32 tensor-pipe probe on `stream`: one CTA per SM issues
 * `iterations` rounds of four tcgen05.mma.kind::tf32 M128 N256 K8 (the
 * tensor-core path's wide-tile MMA) on operand tiles held in shared memory,
 * accumulating in tensor memory, with no global traffic.  The caller times the
 * launch and divides *flops_out by the time: the measured TF32 peak that the
 * 3xTF32 path's tensor-pipe work is compared with.  The pages have no
 * counterpart; they quote TF32 throughput only for a whole GEMM.
 *   iterations  1 .. 2^20 (2^20 rounds take about 0.3 s).
 *   out         device buffer of at least sgemm_probe_out_elems() floats;
 *               receives one accumulator value per CTA (finite when the work
 *               was done).
 *   flops_out   host pointer; receives the FLOPs of one launch.
 * SGEMM_EDEVICE unless the current device is sm_103.  If the completion wait
 * runs out, bit 0 of the device status word is set (sgemm_device_status).
 */
int sgemm_probe_tf32_mma(int64_t iterations, float *out, double *flops_out, void *stream);

/*
 * Measurement knob for the block raster ("CUDA GEMM operator performance
 * optimization", section 2.3: the order in which output tiles are scheduled
 * decides how often L2 re-serves operand panels).  Every kernel walks its
 * 128-row tiles in groups of `group_m` tile rows, sweeping each group down a
 * column of tiles before moving right; the library's choice is 8.  This sets
 * group_m for the calls made after it on any thread (1 = row-major order,
 * a value at least the tile-row count = column-major order), 0 restores 8.
 * Results are bit-identical for every value: only the order in which tiles
 * run changes, never the arithmetic of an output.  It exists to measure the
 * L2 hit rate against the order; calls already enqueued are not affected.
 * Returns the previous value, or -1 (nothing changed) if group_m is outside
 * 0 .. 65536.
 */
int sgemm_set_raster_group(int group_m);

/*
 * Measurement knob for the accuracy of sgemm_f32_tf32x3* over long reductions
 * (no counterpart on the source pages; the accuracy it trades is the FMA vs
 * TF32 RRMSE comparison of the ChetanC28/cuda-kernels page).  Products with
 * K > 256 accumulate on the tensor cores in chunks of `chunk_k` of K and add
 * the chunk sums in round-to-nearest fp32; the tensor cores' own accumulation
 * rounds towards zero, so shorter chunks are more accurate and cost a little
 * more (3072^3: 64 -> RRMSE 5.6e-7, 128 -> 1.0e-6, 256 -> 1.9e-6).  The
 * library's choice is 128.  Sets chunk_k for the calls made after it on any
 * thread: a multiple of 32 from 32 to 2^30 (a value at least K puts the whole
 * reduction in one chunk), 0 restores 128.  Results stay deterministic and
 * exact on small integers for every value.  Returns the previous value, or -1
 * (nothing changed) for any other chunk_k.
 */
int sgemm_set_tf32x3_chunk_k(int chunk_k);

/*
 * Self-test of the library's failure path (no counterpart on the source
 * pages): launches one CTA that waits, with the bounded wait of the tensor-core
 * pipeline, on a barrier nothing ever arrives on.  After about `limit_cycles`
 * SM cycles (1e3 .. 4e9) the wait gives up, the CTA sets bit 0 of the device
 * status word (read it with sgemm_device_status) and exits normally; the CUDA
 * context stays usable.  Nothing faults, traps or hangs.
 */
int sgemm_selftest_wait_timeout(int64_t limit_cycles, void *stream);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_GB300_PROBE_H */
