/*
 * gemm_probe.h -- measured throughput ceilings for the roofline of the GEMM
 * library's kernels (part of libgemmpipe.so).
 *
 * Pipelined kernels are judged against the hardware's own limits ("CUDA
 * Kernel Study: Pipelining", NCU Profiling Comparison: compute and memory
 * throughput as a fraction of peak).  For the INT8 path (warp-level IMMA; the
 * GB300's tcgen05 has no integer kind) and the FP32 FFMA path no measured
 * peak is supplied with the machine, so this probe measures one: independent
 * chains of the one instruction the kernel's inner loop is built from, on
 * every SM, with no memory traffic.
 */
#ifndef GEMM_PROBE_H
#define GEMM_PROBE_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GP_PROBE_IMMA_S8 0  /* mma.sync.m16n8k32 s8 x s8 -> s32: 2*16*8*32 ops per warp instruction */
#define GP_PROBE_FFMA_F32 1 /* fmaf on fp32: 2 FLOP per thread instruction */

/*
 * gemm_probe_peak -- run the probe for `kind` on the current device and
 * stream (cudaStream_t as void*, NULL = default stream) and store the best
 * measured rate in *ops_per_s (operations per second: INT8 ops or FP32 FLOP).
 * Synchronous: returns after the probe kernels have finished (about 0.1 s).
 * Returns 0, GP_ERR_ARG (-1) for a bad kind or NULL output, or GP_ERR_CUDA (-4).
 * Allocates nothing.
 */
int gemm_probe_peak(int kind, double* ops_per_s, void* stream);

/*
 * HBM bandwidth ceilings for the kernels whose roof is memory: the GEMMs with
 * few K steps write C far more than they read (store-bound), the skinny ones
 * read A once (load-bound).  Each is measured with 16-byte accesses by a
 * grid-stride kernel over a caller-supplied device buffer, so that the
 * denominators come from this GPU rather than from a nominal figure.
 */
#define GP_PROBE_HBM_WRITE 2 /* stores only: bytes written per second over the whole buffer */
#define GP_PROBE_HBM_READ 3  /* loads only: bytes read per second over the whole buffer */
#define GP_PROBE_HBM_COPY 4  /* first half copied to the second: bytes read + bytes written per second */

/*
 * gemm_probe_hbm -- time the access pattern `kind` over the device buffer
 * `buf` of `bytes` bytes (owned by the caller, 16-byte aligned, at least
 * 1 MiB and a multiple of 32 bytes; its contents are overwritten by the
 * write and copy probes) on `stream` (cudaStream_t as void*, NULL = default
 * stream), five timed launches (each after an untimed one) for each of 2, 4
 * and 8 blocks of 512 threads per SM, and store the best rate in *bytes_per_s.  Use a
 * buffer far larger than the L2 (hundreds of MB or more) so that the rate is
 * that of HBM.  Synchronous.  Returns 0, GP_ERR_ARG (-1) for a bad kind, a
 * NULL pointer, a misaligned or too small buffer, or GP_ERR_CUDA (-4).
 * Allocates nothing.
 */
int gemm_probe_hbm(int kind, void* buf, size_t bytes, double* bytes_per_s, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_PROBE_H */
