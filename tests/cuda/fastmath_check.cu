// Compares the Newton-refined fp64 reciprocal and reciprocal square root of
// swe_fastmath.cuh with CUDA's own 1.0 / x and rsqrt(x) on the GPU over a
// sweep of positive arguments (decades 1e-300 .. 1e300 and a seeded random
// sample), printing the largest distance in units in the last place.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <cuda_runtime.h>

#include "../../finite_volume_shallow_gb300/csrc/swe_fastmath.cuh"

__global__ void check(const double* x, int n, unsigned long long* ulp_rcp,
                      unsigned long long* ulp_rsq) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const double v = x[i];
  const double a = swe::rcp_nr(v), b = 1.0 / v;
  const double c = swe::rsq_nr(v), d = rsqrt(v);
  long long da = __double_as_longlong(a) - __double_as_longlong(b);
  long long dc = __double_as_longlong(c) - __double_as_longlong(d);
  atomicMax(ulp_rcp, (unsigned long long)(da < 0 ? -da : da));
  atomicMax(ulp_rsq, (unsigned long long)(dc < 0 ? -dc : dc));
}

int main() {
  const int n = 1 << 20;
  double* h = new double[n];
  uint64_t s = 88172645463325252ull;
  for (int i = 0; i < n; ++i) {
    s ^= s << 13; s ^= s >> 7; s ^= s << 17;  // xorshift64
    const double u = (double)(s >> 11) * (1.0 / 9007199254740992.0);
    // log-uniform over [1e-300, 1e300], then the kernels' working range
    h[i] = i < n / 2 ? pow(10.0, -300.0 + 600.0 * u) : 0.01 + 100.0 * u;
  }
  double* d;
  unsigned long long* u;
  cudaMalloc(&d, n * sizeof(double));
  cudaMalloc(&u, 2 * sizeof(unsigned long long));
  cudaMemset(u, 0, 2 * sizeof(unsigned long long));
  cudaMemcpy(d, h, n * sizeof(double), cudaMemcpyHostToDevice);
  check<<<(n + 255) / 256, 256>>>(d, n, u, u + 1);
  unsigned long long r[2];
  cudaMemcpy(r, u, sizeof(r), cudaMemcpyDeviceToHost);
  cudaError_t e = cudaGetLastError();
  printf("%d %llu %llu\n", (int)e, r[0], r[1]);
  cudaFree(d);
  cudaFree(u);
  delete[] h;
  return e == cudaSuccess ? 0 : 1;
}
