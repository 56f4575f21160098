// swe_cart2.cu -- sm_103a kernels of the two-layer IR-Roe step on a
// Cartesian grid.
//
// Scheme: An MPI-CUDA implementation of an improved Roe method for two-layer
// shallow water systems, Sec. 2.1 (eq. (1): two superposed layers, 1 = upper,
// coupled through -g h1 dh2 and -r g h2 dh1) and Sec. 2.2 (eq. (4), steps 1-4
// with the 4x4 Roe matrix A_ij of the rotated system, CFL eq. (5)).
//
// Kernels:
//   cart2_flux_kernel    a 32 x 8 tile of cells and its one-cell halo in
//                        shared memory; every edge of the tile evaluated once
//                        (as in the tile scheme of A multi-GPU shallow-water
//                        simulation with transport of contaminants, Figure
//                        4); each cell sums its four edges into the residual
//                        R (global scratch) and max-reduces sum |Gamma| ||D||,
//                        which fixes dt of this step;
//   cart2_step_kernel    the same with the update of the previous step fused
//                        into the tile load: it reads W^{n-1}, R^{n-1} and
//                        the wave-speed maximum of W^{n-1}, forms W^n =
//                        W^{n-1} - (dt/dx) R^{n-1} for the tile and its halo,
//                        writes W^n of its own cells to the other buffer and
//                        evaluates the fluxes of W^n (W and R alternate
//                        between two buffers);
//   cart2_update_kernel  W -= (dt/dx) R (16-byte vectors over whole rows, the
//                        padding left as it is), checks, dt bookkeeping: a
//                        lone step, and the last step of a run.
// A run of n >= 2 steps is one flux launch, n - 1 fused launches and one
// update; every form applies the update with the same rounding (upd below),
// so a run and the same steps taken one at a time agree bit for bit.
//
// The edge flux itself (quartic roots, closed-form P^- d) is in swe_roe2.cuh.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "swe_internal.h"
#include "swe_roe2.cuh"

namespace swe {
namespace {

// per-cell quantities in shared memory
enum { C_H1, C_Q1X, C_Q1Y, C_H2, C_Q2X, C_Q2Y, C_H, C_S1, C_S2, C_RS1, C_RS2, NCQ };

constexpr int TX = kTile2X;

// Early exit of the outer Newton iteration (warp vote): always for fp64;
// for fp32 a compile-time choice (SWE_CART2_ADAPT32; on by default: 162 us
// per flux launch on the 2048^2 interface dam break against 167 us with the
// fixed count).
#ifndef SWE_CART2_ADAPT32
#define SWE_CART2_ADAPT32 1
#endif
template <typename T> constexpr bool kAdapt2 = sizeof(T) == 8 || SWE_CART2_ADAPT32 != 0;

// W^{n+1} = W^n - (dt/dx) R, one fused multiply-add
__device__ __forceinline__ float upd(float w, float k, float r) { return __fmaf_rn(-k, r, w); }
__device__ __forceinline__ double upd(double w, double k, double r) { return __fma_rn(-k, r, w); }

// dt of a finished flux pass from its wave-speed maximum (eq. (5)) as
// dt/dx = 2 cfl / max, computed by one thread per block; block (0, 0) also
// records dt, advances the clock and zeroes the slot(s) the next flux
// passes will reduce into.
template <typename T>
__device__ __forceinline__ T dt_of_step(const Update2Args<T>& A, T* k_sh) {
  if (threadIdx.x == 0 && threadIdx.y == 0) {
    const T tm = *reinterpret_cast<const T*>(A.tmax_in);
    const double dtdx = A.two_cfl / (double)tm;
    *k_sh = (T)dtdx;
    if (blockIdx.x == 0 && blockIdx.y == 0) {
      const double dt = dtdx * A.dx;
      A.dt_hist[A.step % kHistCap] = dt;
      *A.t_dev += dt;
      if (sizeof(T) == 4) *reinterpret_cast<unsigned*>(A.tmax_clear) = 0u;
      else *reinterpret_cast<unsigned long long*>(A.tmax_clear) = 0ull;
      if (A.tmax_clear2) {
        if (sizeof(T) == 4) *reinterpret_cast<unsigned*>(A.tmax_clear2) = 0u;
        else *reinterpret_cast<unsigned long long*>(A.tmax_clear2) = 0ull;
      }
    }
  }
  __syncthreads();
  return *k_sh;
}

template <typename T> struct Vec2;
template <> struct Vec2<float> { using type = float4; static constexpr int n = 4; };
template <> struct Vec2<double> { using type = double2; static constexpr int n = 2; };

template <typename T, int TY>
__device__ __forceinline__ Side2<T> side_of(const T (*c)[TY + 2][TX + 2], int lj, int li,
                                            bool xdir) {
  Side2<T> s;
  s.h[0] = c[C_H1][lj][li];
  s.h[1] = c[C_H2][lj][li];
  s.s[0] = c[C_S1][lj][li];
  s.s[1] = c[C_S2][lj][li];
  s.rs[0] = c[C_RS1][lj][li];
  s.rs[1] = c[C_RS2][lj][li];
  // normal / tangential discharge: x-edges (q_x, q_y); y-edges (q_y, q_x),
  // the tangential flux of a y-edge going to the x-momentum
  s.qn[0] = xdir ? c[C_Q1X][lj][li] : c[C_Q1Y][lj][li];
  s.qt[0] = xdir ? c[C_Q1Y][lj][li] : c[C_Q1X][lj][li];
  s.qn[1] = xdir ? c[C_Q2X][lj][li] : c[C_Q2Y][lj][li];
  s.qt[1] = xdir ? c[C_Q2Y][lj][li] : c[C_Q2X][lj][li];
  s.H = c[C_H][lj][li];
  return s;
}

// FUSED: the cart2_step_kernel form (U carries the previous step's update);
// otherwise U is unused.  EFIX: the entropy fix of edge2.
template <typename T, bool ANISO, bool FUSED, bool EFIX>
__device__ __forceinline__ void flux_tile(const Step2Args<T>& A, const Update2Args<T>& U) {
  constexpr int TY = Tile2Y<T>::v;
  __shared__ T cq[NCQ][TY + 2][TX + 2];
  __shared__ T ex[NEQ][TY][TX + 1];   // x-edge e joins local columns e and e + 1
  __shared__ T ey[NEQ][TY + 1][TX];   // y-edge e joins local rows e and e + 1
  __shared__ T k_sh;
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int t = ty * TX + tx;
  const int i0 = blockIdx.x * TX, j0 = blockIdx.y * TY;
  const int nx = A.nx, ny = A.ny;
  const T g = A.g, gh = T(0.5) * A.g, r = A.r;
  pdl_wait();
  const T k = FUSED ? dt_of_step<T>(U, &k_sh) : T(0);
  unsigned bad = 0;

  // tile + one-cell halo (the padded layout keeps every read in bounds)
  for (int idx = t; idx < (TX + 2) * (TY + 2); idx += TX * TY) {
    const int li = idx % (TX + 2), lj = idx / (TX + 2);
    const int64_t o = (int64_t)(j0 - 1 + lj + kPadY) * A.pitch + (i0 - 1 + li + kPadX);
    T w[6];
#pragma unroll
    for (int f = 0; f < 6; ++f) w[f] = A.w[f][o];
    if (FUSED) {
      // the previous step's update, on cells of the grid only (the padding
      // keeps its resting state); the tile's own cells are written out
      const int gi = i0 - 1 + li, gj = j0 - 1 + lj;
      if (gi >= 0 && gi < nx && gj >= 0 && gj < ny) {
#pragma unroll
        for (int f = 0; f < 6; ++f) w[f] = upd(w[f], k, U.R[f][o]);
        if (li >= 1 && li <= TX && lj >= 1 && lj <= TY) {
#pragma unroll
          for (int f = 0; f < 6; ++f) U.w[f][o] = w[f];
          const T sum = ((w[0] + w[1]) + (w[2] + w[3])) + (w[4] + w[5]);
          if (!(fabs(sum) <= M2<T>::big())) bad |= kErrNonfinite;
          if (!(w[0] > T(0)) || !(w[3] > T(0))) bad |= kErrDepth;
        }
      }
    }
    const T h1 = w[0], h2 = w[3];
    cq[C_H1][lj][li] = h1;
    cq[C_Q1X][lj][li] = w[1];
    cq[C_Q1Y][lj][li] = w[2];
    cq[C_H2][lj][li] = h2;
    cq[C_Q2X][lj][li] = w[4];
    cq[C_Q2Y][lj][li] = w[5];
    cq[C_H][lj][li] = A.H[o];
    const T r1 = M2<T>::rsq(h1), r2 = M2<T>::rsq(h2);
    cq[C_RS1][lj][li] = r1;
    cq[C_RS2][lj][li] = r2;
    cq[C_S1][lj][li] = h1 * r1;
    cq[C_S2][lj][li] = h2 * r2;
  }
  __syncthreads();

  bool hyper_ok = true;
  // x-edges: (TX + 1) per row; global column of the left cell i0 - 1 + e
  for (int k = t; k < (TX + 1) * TY; k += TX * TY) {
    const int e = k % (TX + 1), row = k / (TX + 1);
    const int gl = i0 - 1 + e;  // left cell's global column
    Side2<T> a = side_of<T, TY>(cq, row + 1, e, true);
    Side2<T> b = side_of<T, TY>(cq, row + 1, e + 1, true);
    const bool lw = gl == -1, rw = gl == nx - 1;
    if (lw) mirror2(a, b);
    if (rw) mirror2(b, a);
    T out[NEQ];
    hyper_ok &= edge2<T, kAdapt2<T>, EFIX>(a, b, g, gh, r, lw || rw, out);
#pragma unroll
    for (int q = 0; q < NEQ; ++q) ex[q][row][e] = out[q];
  }
  // y-edges: TY + 1 per column; global row of the lower cell j0 - 1 + e.
  // The thread index is rotated by one warp, so that the second pass of the
  // y-edges falls on the last warp, not on the one that took the x-edges'
  // second pass.
  for (int k = (t + TX * TY - 32) % (TX * TY); k < TX * (TY + 1); k += TX * TY) {
    const int col = k % TX, e = k / TX;
    const int gl = j0 - 1 + e;
    Side2<T> a = side_of<T, TY>(cq, e, col + 1, false);
    Side2<T> b = side_of<T, TY>(cq, e + 1, col + 1, false);
    const bool lw = gl == -1, rw = gl == ny - 1;
    if (lw) mirror2(a, b);
    if (rw) mirror2(b, a);
    T out[NEQ];
    hyper_ok &= edge2<T, kAdapt2<T>, EFIX>(a, b, g, gh, r, lw || rw, out);
#pragma unroll
    for (int q = 0; q < NEQ; ++q) ey[q][e][col] = out[q];
  }
  __syncthreads();

  // residual of this thread's cell: east and north edges as the left/lower
  // side, west and south as the right/upper side
  const int gi = i0 + tx, gj = j0 + ty;
  const bool own = gi < nx && gj < ny;
  const T rho = A.rho;
  auto ys = [&](T v) { return ANISO ? v * rho : v; };
  T R[6];
  R[0] = (ex[E_M1][ty][tx + 1] - ex[E_M1][ty][tx]) + ys(ey[E_M1][ty + 1][tx] - ey[E_M1][ty][tx]);
  R[1] = (ex[E_PM1][ty][tx + 1] + ex[E_PS1][ty][tx]) + ys(ey[E_T1][ty + 1][tx] - ey[E_T1][ty][tx]);
  R[2] = (ex[E_T1][ty][tx + 1] - ex[E_T1][ty][tx]) + ys(ey[E_PM1][ty + 1][tx] + ey[E_PS1][ty][tx]);
  R[3] = (ex[E_M2][ty][tx + 1] - ex[E_M2][ty][tx]) + ys(ey[E_M2][ty + 1][tx] - ey[E_M2][ty][tx]);
  R[4] = (ex[E_PM2][ty][tx + 1] + ex[E_PS2][ty][tx]) + ys(ey[E_T2][ty + 1][tx] - ey[E_T2][ty][tx]);
  R[5] = (ex[E_T2][ty][tx + 1] - ex[E_T2][ty][tx]) + ys(ey[E_PM2][ty + 1][tx] + ey[E_PS2][ty][tx]);
  const T Tsum = (ex[E_D][ty][tx] + ex[E_D][ty][tx + 1]) +
                 ys(ey[E_D][ty][tx] + ey[E_D][ty + 1][tx]);
  if (own) {
    const int64_t o = (int64_t)(gj + kPadY) * A.pitch + gi + kPadX;
#pragma unroll
    for (int f = 0; f < 6; ++f) A.R[f][o] = R[f];
  }
  // hyperbolicity of every edge of this block, and the block's max of T
  if (!__all_sync(kFull2, hyper_ok) && (tx & 31) == 0) atomicOr(A.err, kErrHyperbolic);
  if (FUSED && bad) atomicOr(A.err, bad);
  T m = own ? Tsum : T(0);
  pdl_trigger();
  block_max_publish<T, TX * TY / 32>(m, A.tmax_out);
}

// Resident blocks per SM the registers are held to: five 256-thread fp32
// tiles (48 registers) fit next to their 35 KB of shared memory each; fp64
// tiles are bounded by shared memory and the FP64 pipe; the entropy-fix
// variants (two more root solves per edge) are left to the compiler.
template <typename T, bool EFIX> struct MinBlocks2 { static constexpr int v = 1; };
template <> struct MinBlocks2<float, false> { static constexpr int v = 5; };

template <typename T, bool ANISO, bool EFIX>
__global__ void __launch_bounds__(kTile2X * Tile2Y<T>::v, MinBlocks2<T, EFIX>::v)
    cart2_flux_kernel(const Step2Args<T> A) {
  flux_tile<T, ANISO, false, EFIX>(A, Update2Args<T>{});
}

template <typename T, bool ANISO, bool EFIX>
__global__ void __launch_bounds__(kTile2X * Tile2Y<T>::v, MinBlocks2<T, EFIX>::v)
    cart2_step_kernel(const Step2Args<T> A, const Update2Args<T> U) {
  flux_tile<T, ANISO, true, EFIX>(A, U);
}

template <typename T>
__global__ void cart2_update_kernel(const Update2Args<T> A) {
  // dt / dx = 2 cfl / max T, once per block (a double division per thread
  // would cost more than the update on GB300's FP64 pipe)
  __shared__ T k_sh;
  pdl_wait();
  const T k = dt_of_step<T>(A, &k_sh);
  // whole rows in 16-byte vectors (the pitch is a multiple of 32); elements
  // of the padding keep their value exactly (even if k is not finite)
  using V = typename Vec2<T>::type;
  constexpr int VN = Vec2<T>::n;
  const int nvr = A.pitch / VN;
  const int v = blockIdx.x * blockDim.x + threadIdx.x;
  const int c0 = v * VN - kPadX;  // logical column of the vector's first element
  unsigned bad = 0;
  for (int gj = blockIdx.y * blockDim.y + threadIdx.y; v < nvr && gj < A.ny;
       gj += gridDim.y * blockDim.y) {
    const int64_t o = (int64_t)(gj + kPadY) * nvr + v;
    T w[6][VN];
#pragma unroll
    for (int f = 0; f < 6; ++f) {
      V wv = reinterpret_cast<const V*>(A.win[f])[o];
      const V rv = reinterpret_cast<const V*>(A.R[f])[o];
      T* wp = reinterpret_cast<T*>(&wv);
      const T* rp = reinterpret_cast<const T*>(&rv);
#pragma unroll
      for (int j = 0; j < VN; ++j) {
        const bool in = c0 + j >= 0 && c0 + j < A.nx;
        const T nw = upd(wp[j], k, rp[j]);
        wp[j] = in ? nw : wp[j];
        w[f][j] = wp[j];
      }
      reinterpret_cast<V*>(A.w[f])[o] = wv;
    }
#pragma unroll
    for (int j = 0; j < VN; ++j) {
      if (!(c0 + j >= 0 && c0 + j < A.nx)) continue;
      const T sum = ((w[0][j] + w[1][j]) + (w[2][j] + w[3][j])) + (w[4][j] + w[5][j]);
      if (!(fabs(sum) <= M2<T>::big())) bad |= kErrNonfinite;
      if (!(w[0][j] > T(0)) || !(w[3][j] > T(0))) bad |= kErrDepth;
    }
  }
  pdl_trigger();
  if (bad) atomicOr(A.err, bad);
}

// initial / restarted state: positivity and finiteness
template <typename T>
__global__ void cart2_check_kernel(const Fields6<T> w6, int nx, int ny, int pitch,
                                   unsigned* err) {
  const int gi = blockIdx.x * blockDim.x + threadIdx.x;
  unsigned bad = 0;
  for (int gj = blockIdx.y; gi < nx && gj < ny; gj += gridDim.y) {
    const int64_t o = (int64_t)(gj + kPadY) * pitch + gi + kPadX;
    T s = T(0);
    for (int f = 0; f < 6; ++f) s += w6.p[f][o];
    if (!isfinite(s)) bad |= kErrNonfinite;
    if (!(w6.p[0][o] > T(0)) || !(w6.p[3][o] > T(0))) bad |= kErrDepth;
  }
  if (bad) atomicOr(err, bad);
}

}  // namespace

template <typename T>
cudaError_t launch_flux2(const Step2Args<T>& f, cudaStream_t st) {
  constexpr int TY = Tile2Y<T>::v;
  dim3 block(TX, TY);
  dim3 grid((unsigned)((f.nx + TX - 1) / TX), (unsigned)((f.ny + TY - 1) / TY));
  if (f.efix)
    return f.rho == T(1) ? launch_pdl(cart2_flux_kernel<T, false, true>, grid, block, 0, st, f)
                         : launch_pdl(cart2_flux_kernel<T, true, true>, grid, block, 0, st, f);
  return f.rho == T(1) ? launch_pdl(cart2_flux_kernel<T, false, false>, grid, block, 0, st, f)
                       : launch_pdl(cart2_flux_kernel<T, true, false>, grid, block, 0, st, f);
}

template <typename T>
cudaError_t launch_fused2(const Step2Args<T>& f, const Update2Args<T>& u, cudaStream_t st) {
  constexpr int TY = Tile2Y<T>::v;
  dim3 block(TX, TY);
  dim3 grid((unsigned)((f.nx + TX - 1) / TX), (unsigned)((f.ny + TY - 1) / TY));
  if (f.efix)
    return f.rho == T(1)
               ? launch_pdl(cart2_step_kernel<T, false, true>, grid, block, 0, st, f, u)
               : launch_pdl(cart2_step_kernel<T, true, true>, grid, block, 0, st, f, u);
  return f.rho == T(1) ? launch_pdl(cart2_step_kernel<T, false, false>, grid, block, 0, st, f, u)
                       : launch_pdl(cart2_step_kernel<T, true, false>, grid, block, 0, st, f, u);
}

template <typename T>
cudaError_t launch_update2(const Update2Args<T>& u, cudaStream_t st) {
  constexpr int VN = Vec2<T>::n;
  dim3 ub(64, 4);
  dim3 ug((unsigned)((u.pitch / VN + 63) / 64), (unsigned)min((u.ny + 3) / 4, 1024));
  return launch_pdl(cart2_update_kernel<T>, ug, ub, 0, st, u);
}

template <typename T>
cudaError_t launch_check2(const Fields6<T>& w6, int nx, int ny, int pitch, unsigned* err,
                          cudaStream_t st) {
  dim3 grid((unsigned)((nx + 127) / 128), (unsigned)(ny < 1024 ? ny : 1024));
  cart2_check_kernel<T><<<grid, 128, 0, st>>>(w6, nx, ny, pitch, err);
  return cudaGetLastError();
}

template cudaError_t launch_flux2<float>(const Step2Args<float>&, cudaStream_t);
template cudaError_t launch_flux2<double>(const Step2Args<double>&, cudaStream_t);
template cudaError_t launch_fused2<float>(const Step2Args<float>&, const Update2Args<float>&,
                                          cudaStream_t);
template cudaError_t launch_fused2<double>(const Step2Args<double>&, const Update2Args<double>&,
                                           cudaStream_t);
template cudaError_t launch_update2<float>(const Update2Args<float>&, cudaStream_t);
template cudaError_t launch_update2<double>(const Update2Args<double>&, cudaStream_t);
template cudaError_t launch_check2<float>(const Fields6<float>&, int, int, int, unsigned*,
                                          cudaStream_t);
template cudaError_t launch_check2<double>(const Fields6<double>&, int, int, int, unsigned*,
                                           cudaStream_t);

}  // namespace swe
