/*
 * swe_probe.h -- measured denominators for the arithmetic rooflines of libswe.
 *
 * The kernels of the finite-volume step that are limited by arithmetic rather
 * than by memory (the fp64 steps, and the two-layer flux whose Roe matrix of
 * An MPI-CUDA implementation of an improved Roe method for two-layer shallow
 * water systems, Sec. 2.2, needs the roots of a quartic per edge) are measured
 * against the rate at which this GPU retires fused multiply-adds.  The papers
 * have no counterpart of this call: it measures that rate on the device it
 * runs on, so the fractions do not rest on a data-sheet figure.
 */
#ifndef SWE_PROBE_H
#define SWE_PROBE_H

#include "swe.h"

#ifdef __cplusplus
extern "C" {
#endif

#define SWE_PROBE_FFMA 0  /* FP32 fused multiply-add, one per instruction      */
#define SWE_PROBE_FFMA2 1 /* FP32 fused multiply-add on packed pairs (f32x2)   */
#define SWE_PROBE_DFMA 2  /* FP64 fused multiply-add                           */

/* Sustained FMA throughput of the current device, in floating-point
 * operations per second (one FMA = 2).  One full wave of blocks, each thread
 * running 8 independent FMA chains, is launched three times on `stream`
 * (cudaStream_t, NULL for the default stream): a short launch, then two sized
 * to last about target_ms; the last one is timed with CUDA events.
 *  kind         SWE_PROBE_FFMA, SWE_PROBE_FFMA2 or SWE_PROBE_DFMA
 *  target_ms    1 <= target_ms <= 1000
 *  flops_per_s  out: the measured rate (required)
 *  ms_out       out: duration of the timed launch in milliseconds (may be NULL)
 * Allocates and frees a few KB of device memory and synchronises the stream.
 * Changes no device setting; the rate is the one at the clocks the GPU runs
 * at during the call.  Errors: SWE_ERR_ARG, SWE_ERR_OOM, SWE_ERR_CUDA. */
swe_status swe_probe_fma_rate(int32_t kind, double target_ms, void *stream,
                              double *flops_per_s, double *ms_out);

#ifdef __cplusplus
}
#endif
#endif /* SWE_PROBE_H */
