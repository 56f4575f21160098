// swe_probe.cu -- throughput probe of the SMs' floating-point FMA pipes.
//
// The kernels of the scheme that are bound by arithmetic (the fp64 steps, the
// two-layer flux with its quartic roots) are reported against the rate at
// which this GPU retires fused multiply-adds.  This file measures that rate
// instead of taking it from a data sheet: every thread of a full-occupancy
// grid runs kChains independent FMA chains (no dependency between
// consecutive instructions of the unrolled loop, so the pipe, not latency,
// limits), timed with CUDA events on the caller's stream.  One FMA counts as
// two floating-point operations.
//
// Kinds: FP32 scalar FFMA, FP32 packed pairs (fma.rn.f32x2: two FMAs per
// instruction), FP64 DFMA.  The chains x <- x * m + c with 0 < m < 1 converge
// to a finite fixed point, so no value overflows or becomes subnormal.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/swe_probe.h"

namespace {

constexpr int kChains = 8;
constexpr int kUnroll = 8;
constexpr int kThreads = 256;

__device__ __forceinline__ float ffma_rn(float a, float b, float c) {
  float d;
  asm volatile("fma.rn.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ double dfma_rn(double a, double b, double c) {
  double d;
  asm volatile("fma.rn.f64 %0, %1, %2, %3;" : "=d"(d) : "d"(a), "d"(b), "d"(c));
  return d;
}

__global__ void __launch_bounds__(kThreads) probe_ffma_kernel(int64_t iters, float m, float c,
                                                              float* sink) {
  float x[kChains];
#pragma unroll
  for (int k = 0; k < kChains; ++k) x[k] = (float)(threadIdx.x + k) * 1e-3f;
  for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
      for (int k = 0; k < kChains; ++k) x[k] = ffma_rn(x[k], m, c);
  }
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < kChains; ++k) s += x[k];
  if (s == -1.0f) sink[blockIdx.x] = s;  // never true: keeps the chains live
}

__global__ void __launch_bounds__(kThreads) probe_ffma2_kernel(int64_t iters, float m, float c,
                                                               float* sink) {
  float2 x[kChains];
#pragma unroll
  for (int k = 0; k < kChains; ++k)
    x[k] = make_float2((float)(threadIdx.x + k) * 1e-3f, (float)(threadIdx.x - k) * 1e-3f);
  const float2 m2 = make_float2(m, m), c2 = make_float2(c, c);
  for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
      for (int k = 0; k < kChains; ++k) x[k] = __ffma2_rn(x[k], m2, c2);
  }
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < kChains; ++k) s += x[k].x + x[k].y;
  if (s == -1.0f) sink[blockIdx.x] = s;
}

__global__ void __launch_bounds__(kThreads) probe_dfma_kernel(int64_t iters, double m, double c,
                                                              float* sink) {
  double x[kChains];
#pragma unroll
  for (int k = 0; k < kChains; ++k) x[k] = (double)(threadIdx.x + k) * 1e-3;
  for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
#pragma unroll
      for (int k = 0; k < kChains; ++k) x[k] = dfma_rn(x[k], m, c);
  }
  double s = 0.0;
#pragma unroll
  for (int k = 0; k < kChains; ++k) s += x[k];
  if (s == -1.0) sink[blockIdx.x] = (float)s;
}

cudaError_t launch(int kind, int blocks, int64_t iters, float* sink, cudaStream_t st) {
  switch (kind) {
    case SWE_PROBE_FFMA:
      probe_ffma_kernel<<<blocks, kThreads, 0, st>>>(iters, 0.999f, 1e-3f, sink);
      break;
    case SWE_PROBE_FFMA2:
      probe_ffma2_kernel<<<blocks, kThreads, 0, st>>>(iters, 0.999f, 1e-3f, sink);
      break;
    default:
      probe_dfma_kernel<<<blocks, kThreads, 0, st>>>(iters, 0.999, 1e-3, sink);
      break;
  }
  return cudaGetLastError();
}

int occupancy(int kind, int* per_sm) {
  const void* f = kind == SWE_PROBE_FFMA    ? (const void*)probe_ffma_kernel
                  : kind == SWE_PROBE_FFMA2 ? (const void*)probe_ffma2_kernel
                                            : (const void*)probe_dfma_kernel;
  return (int)cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, f, kThreads, 0);
}

// flops of one launch: threads x iterations x unrolled chain steps x 2
// (x 2 again for packed pairs)
double flops_of(int kind, int blocks, int64_t iters) {
  const double per = 2.0 * kChains * kUnroll * (kind == SWE_PROBE_FFMA2 ? 2.0 : 1.0);
  return per * (double)blocks * kThreads * (double)iters;
}

}  // namespace

extern "C" swe_status swe_probe_fma_rate(int32_t kind, double target_ms, void* stream,
                                         double* flops_per_s, double* ms_out) {
  if (!flops_per_s) return SWE_ERR_ARG;
  if (kind != SWE_PROBE_FFMA && kind != SWE_PROBE_FFMA2 && kind != SWE_PROBE_DFMA)
    return SWE_ERR_ARG;
  if (!(target_ms >= 1.0 && target_ms <= 1000.0)) return SWE_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SWE_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SWE_ERR_CUDA;
  if (occupancy(kind, &per_sm) != 0 || per_sm < 1) return SWE_ERR_CUDA;
  const int blocks = sms * per_sm;  // one full wave
  float* sink = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  swe_status rc = SWE_OK;
  float ms = 0.f;
  if (cudaMalloc(&sink, sizeof(float) * (size_t)blocks) != cudaSuccess) {
    (void)cudaGetLastError();
    return SWE_ERR_OOM;
  }
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
    rc = SWE_ERR_CUDA;
    goto done;
  }
  {
    // a short launch first (warms the clocks and the module), then one sized
    // from it to last about target_ms
    int64_t iters = 256;
    for (int pass = 0; pass < 3 && rc == SWE_OK; ++pass) {
      if (cudaEventRecord(e0, st) != cudaSuccess || launch(kind, blocks, iters, sink, st) ||
          cudaEventRecord(e1, st) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess ||
          cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess) {
        rc = SWE_ERR_CUDA;
        break;
      }
      if (pass < 2) {
        const double scale = target_ms / (ms > 1e-3f ? (double)ms : 1e-3);
        double next = (double)iters * (scale < 64.0 ? scale : 64.0);
        if (next < 16.0) next = 16.0;
        if (next > 1e9) next = 1e9;
        iters = (int64_t)next;
      }
    }
    if (rc == SWE_OK) {
      *flops_per_s = flops_of(kind, blocks, iters) / ((double)ms * 1e-3);
      if (ms_out) *ms_out = ms;
    }
  }
done:
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  cudaFree(sink);
  if (rc != SWE_OK) (void)cudaGetLastError();
  return rc;
}
