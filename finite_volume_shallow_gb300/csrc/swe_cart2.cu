// swe_cart2.cu -- sm_103a kernels of the two-layer IR-Roe step on a
// Cartesian grid.
//
// Scheme: An MPI-CUDA implementation of an improved Roe method for two-layer
// shallow water systems, Sec. 2.1 (eq. (1): two superposed layers, 1 = upper,
// coupled through -g h1 dh2 and -r g h2 dh1) and Sec. 2.2 (eq. (4), steps 1-4
// with the 4x4 Roe matrix A_ij of the rotated system, CFL eq. (5)).
//
// Two launches per step:
//   cart2_flux_kernel    a 32 x 8 tile of cells and its one-cell halo in
//                        shared memory; every edge of the tile evaluated once
//                        (as in the tile scheme of A multi-GPU shallow-water
//                        simulation with transport of contaminants, Figure
//                        4); each cell sums its four edges into the residual
//                        R (global scratch) and max-reduces sum |Gamma| ||D||,
//                        which fixes dt of this step;
//   cart2_update_kernel  W -= (dt/dx) R in place, checks, dt bookkeeping.
//
// The eigenvalues of A_ij are the roots of the quartic
//   p(l) = Q1(l) Q2(l) - r c1^2 c2^2,   Q_k(l) = (l - u_k)^2 - c_k^2.
// The outer two are found by Newton from bounds where p > 0 (p is convex and
// monotone there, so the iterates approach the root from outside without
// overshooting); the inner pair comes from deflating p by the outer pair and
// is polished by Newton on p.  A complex inner pair (loss of hyperbolicity)
// sets an error bit.  With right eigenvectors K_k = (1, l_k, m_k, l_k m_k),
// m_k = Q1(l_k)/c1^2, the left eigenvectors of A_ij are proportional to
// (l - 2u1, 1, c1^2 (l - 2u2)/Q2, c1^2/Q2), which gives the coordinates of d
// in the eigenvector basis without a linear solve:
//   alpha_k = [Q2(l_k)((l_k - 2u1) d1 + d2) + c1^2 ((l_k - 2u2) d3 + d4)] / p'(l_k).
// Then P^- d = sum_k w_k alpha_k K_k with w_k = (1 - sgn l_k)/2.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "swe_internal.h"

namespace swe {
namespace {

constexpr unsigned kFull2 = 0xffffffffu;

template <typename T> struct M2;
template <> struct M2<float> {
  __device__ static __forceinline__ float rsq(float x) { return rsqrtf(x); }
  __device__ static __forceinline__ float rcp(float x) {  // MUFU approximation
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
  }
  __device__ static __forceinline__ float sq(float x) { return sqrtf(x); }
  __device__ static __forceinline__ float big() { return 3.402823466e38f; }
};
template <> struct M2<double> {
  __device__ static __forceinline__ double rsq(double x) { return rsqrt(x); }
  __device__ static __forceinline__ double rcp(double x) { return __drcp_rn(x); }
  __device__ static __forceinline__ double sq(double x) { return sqrt(x); }
  __device__ static __forceinline__ double big() { return 1.7976931348623157e308; }
};

// Newton iterations: the outer roots converge quadratically from a bound a
// fixed fraction of c away; the inner ones start from the deflated estimate.
template <typename T> struct Iters;
template <> struct Iters<float> { static constexpr int outer = 7, inner = 2; };
template <> struct Iters<double> { static constexpr int outer = 9, inner = 3; };

// per-cell quantities in shared memory
enum { C_H1, C_Q1X, C_Q1Y, C_H2, C_Q2X, C_Q2Y, C_H, C_S1, C_S2, C_RS1, C_RS2, NCQ };
// per-edge results in shared memory
enum { E_M1, E_PM1, E_PS1, E_T1, E_M2, E_PM2, E_PS2, E_T2, E_D, NEQ };

// One side of an edge in the frame of its normal: per layer the depth, its
// square root and inverse square root, the normal and tangential discharge.
template <typename T>
struct Side2 {
  T h[2], s[2], rs[2], qn[2], qt[2], H;
};

template <typename T>
__device__ __forceinline__ void mirror2(Side2<T>& g, const Side2<T>& a) {
  g = a;
  g.qn[0] = -a.qn[0];
  g.qn[1] = -a.qn[1];
}

template <typename T>
struct Quartic {
  T u1, u2, c1s, c2s, rc;
  __device__ __forceinline__ T q1(T l) const { return (l - u1) * (l - u1) - c1s; }
  __device__ __forceinline__ T q2(T l) const { return (l - u2) * (l - u2) - c2s; }
  __device__ __forceinline__ T p(T l) const { return q1(l) * q2(l) - rc; }
  __device__ __forceinline__ T dp(T l) const {
    return T(2) * ((l - u1) * q2(l) + (l - u2) * q1(l));
  }
};

// IR-Roe flux of one edge, two layers.  Writes the edge results; returns
// false when A_ij has a complex pair of eigenvalues.
template <typename T>
__device__ __forceinline__ bool edge2(const Side2<T>& a, const Side2<T>& b, T g, T gh, T r,
                                      bool wall, T* out) {
  // Roe averages per layer: sqrt(h)-weighted normal velocity, arithmetic
  // depth; c_k^2 = g hbar_k
  T un[2], cs[2], qu_a[2], qu_b[2], ut_a[2], ut_b[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const T va = a.qn[k] * a.rs[k], vb = b.qn[k] * b.rs[k];
    un[k] = (va + vb) * M2<T>::rcp(a.s[k] + b.s[k]);
    cs[k] = gh * (a.h[k] + b.h[k]);
    const T iha = a.rs[k] * a.rs[k], ihb = b.rs[k] * b.rs[k];
    qu_a[k] = a.qn[k] * a.qn[k] * iha;
    qu_b[k] = b.qn[k] * b.qn[k] * ihb;
    ut_a[k] = a.qt[k] * iha;
    ut_b[k] = b.qt[k] * ihb;
  }
  Quartic<T> q{un[0], un[1], cs[0], cs[1], r * cs[0] * cs[1]};
  const T c1 = M2<T>::sq(cs[0]), c2 = M2<T>::sq(cs[1]);
  // outer roots: from below / above, where p > 0, p convex and monotone
  T l1 = fmin(un[0] - T(1.5) * c1, un[1] - T(1.5) * c2);
  T l4 = fmax(un[0] + T(1.5) * c1, un[1] + T(1.5) * c2);
#pragma unroll
  for (int it = 0; it < Iters<T>::outer; ++it) {
    l1 -= q.p(l1) * M2<T>::rcp(q.dp(l1));
    l4 -= q.p(l4) * M2<T>::rcp(q.dp(l4));
  }
  // inner pair: p / ((l - l1)(l - l4)) = l^2 + bb l + cc
  const T p3 = T(-2) * (un[0] + un[1]);
  const T p2 = (un[0] * un[0] - cs[0]) + (un[1] * un[1] - cs[1]) + T(4) * un[0] * un[1];
  const T ss = l1 + l4, pp = l1 * l4;
  const T bb = p3 + ss;
  const T cc = p2 + ss * bb - pp;
  const T disc = bb * bb - T(4) * cc;
  const bool hyper = disc > T(0);
  const T sd = M2<T>::sq(hyper ? disc : T(0));
  T l2 = T(0.5) * (-bb - sd), l3 = T(0.5) * (-bb + sd);
#pragma unroll
  for (int it = 0; it < Iters<T>::inner; ++it) {
    l2 -= q.p(l2) * M2<T>::rcp(q.dp(l2));
    l3 -= q.p(l3) * M2<T>::rcp(q.dp(l3));
  }
  // fluctuation d = F_1(W_j) - F_1(W_i) - B_ij (W_j - W_i) - S_ij (H_j - H_i)
  // (pressure differences written g hbar_k (h_k,j - h_k,i))
  const T dh1 = b.h[0] - a.h[0], dh2 = b.h[1] - a.h[1], dH = b.H - a.H;
  const T d1 = b.qn[0] - a.qn[0];
  const T d2 = (qu_b[0] - qu_a[0]) + cs[0] * ((dh1 + dh2) - dH);
  const T d3 = b.qn[1] - a.qn[1];
  const T d4 = (qu_b[1] - qu_a[1]) + cs[1] * ((dh2 + r * dh1) - dH);
  // P^- d = sum_k w_k alpha_k K_k
  const T lam[4] = {l1, l2, l3, l4};
  const T ic1s = M2<T>::rcp(cs[0]);
  T pd0 = T(0), pd1 = T(0), pd2 = T(0), pd3 = T(0);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const T l = lam[k];
    const T w = (l < T(0)) ? T(1) : ((l > T(0)) ? T(0) : T(0.5));
    const T Q1 = q.q1(l), Q2 = q.q2(l);
    const T num = Q2 * ((l - T(2) * un[0]) * d1 + d2) + cs[0] * ((l - T(2) * un[1]) * d3 + d4);
    const T alpha = w * num * M2<T>::rcp(q.dp(l));
    const T mu = Q1 * ic1s;
    pd0 += alpha;
    pd1 += alpha * l;
    pd2 += alpha * mu;
    pd3 += alpha * l * mu;
  }
  T m1 = a.qn[0] + pd0;
  T m2 = a.qn[1] + pd2;
  if (wall) {  // a reflective wall passes no mass (algebraically 0)
    m1 = T(0);
    m2 = T(0);
  }
  out[E_M1] = m1;
  out[E_PM1] = pd1;
  out[E_PS1] = d2 - pd1;
  out[E_T1] = m1 * (m1 > T(0) ? ut_a[0] : ut_b[0]);
  out[E_M2] = m2;
  out[E_PM2] = pd3;
  out[E_PS2] = d4 - pd3;
  out[E_T2] = m2 * (m2 > T(0) ? ut_a[1] : ut_b[1]);
  out[E_D] = fmax(fabs(l1), fabs(l4));
  return hyper;
}

template <typename T>
__device__ __forceinline__ void atomic_max_pos2(void* slot, T v);
template <>
__device__ __forceinline__ void atomic_max_pos2<float>(void* slot, float v) {
  atomicMax(reinterpret_cast<unsigned int*>(slot), __float_as_uint(v));
}
template <>
__device__ __forceinline__ void atomic_max_pos2<double>(void* slot, double v) {
  atomicMax(reinterpret_cast<unsigned long long*>(slot),
            static_cast<unsigned long long>(__double_as_longlong(v)));
}
template <typename T>
__device__ __forceinline__ T nanmax2(T acc, T x) {
  return (x > acc || x != x) ? x : acc;
}

constexpr int TX = kTile2X;

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

template <typename T, bool ANISO>
__global__ void __launch_bounds__(kTile2X * Tile2Y<T>::v) cart2_flux_kernel(const Step2Args<T> A) {
  constexpr int TY = Tile2Y<T>::v;
  __shared__ T cq[NCQ][TY + 2][TX + 2];
  __shared__ T ex[NEQ][TY][TX + 1];   // x-edge e joins local columns e and e + 1
  __shared__ T ey[NEQ][TY + 1][TX];   // y-edge e joins local rows e and e + 1
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int t = ty * TX + tx;
  const int i0 = blockIdx.x * TX, j0 = blockIdx.y * TY;
  const int nx = A.nx, ny = A.ny;
  const T g = A.g, gh = T(0.5) * A.g, r = A.r;

  // tile + one-cell halo (the padded layout keeps every read in bounds)
  for (int idx = t; idx < (TX + 2) * (TY + 2); idx += TX * TY) {
    const int li = idx % (TX + 2), lj = idx / (TX + 2);
    const int64_t o = (int64_t)(j0 - 1 + lj + kPadY) * A.pitch + (i0 - 1 + li + kPadX);
    const T h1 = A.w[0][o], h2 = A.w[3][o];
    cq[C_H1][lj][li] = h1;
    cq[C_Q1X][lj][li] = A.w[1][o];
    cq[C_Q1Y][lj][li] = A.w[2][o];
    cq[C_H2][lj][li] = h2;
    cq[C_Q2X][lj][li] = A.w[4][o];
    cq[C_Q2Y][lj][li] = A.w[5][o];
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
    hyper_ok &= edge2<T>(a, b, g, gh, r, lw || rw, out);
#pragma unroll
    for (int q = 0; q < NEQ; ++q) ex[q][row][e] = out[q];
  }
  // y-edges: TY + 1 per column; global row of the lower cell j0 - 1 + e
  for (int k = t; k < TX * (TY + 1); k += TX * TY) {
    const int col = k % TX, e = k / TX;
    const int gl = j0 - 1 + e;
    Side2<T> a = side_of<T, TY>(cq, e, col + 1, false);
    Side2<T> b = side_of<T, TY>(cq, e + 1, col + 1, false);
    const bool lw = gl == -1, rw = gl == ny - 1;
    if (lw) mirror2(a, b);
    if (rw) mirror2(b, a);
    T out[NEQ];
    hyper_ok &= edge2<T>(a, b, g, gh, r, lw || rw, out);
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
  T m = own ? Tsum : T(0);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = nanmax2(m, __shfl_xor_sync(kFull2, m, o));
  if ((t & 31) == 0 && (m > T(0) || m != m)) atomic_max_pos2<T>(A.tmax_out, m);
}

template <typename T>
__global__ void cart2_update_kernel(const Update2Args<T> A) {
  const T tm = *reinterpret_cast<const T*>(A.tmax_in);
  const double dtdx = A.two_cfl / (double)tm;
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 && threadIdx.y == 0) {
    const double dt = dtdx * A.dx;
    A.dt_hist[A.step % kHistCap] = dt;
    *A.t_dev += dt;
    if (sizeof(T) == 4) *reinterpret_cast<unsigned*>(A.tmax_clear) = 0u;
    else *reinterpret_cast<unsigned long long*>(A.tmax_clear) = 0ull;
  }
  const T k = (T)dtdx;
  const int gi = blockIdx.x * blockDim.x + threadIdx.x;
  unsigned bad = 0;
  for (int gj = blockIdx.y * blockDim.y + threadIdx.y; gi < A.nx && gj < A.ny;
       gj += gridDim.y * blockDim.y) {
    const int64_t o = (int64_t)(gj + kPadY) * A.pitch + gi + kPadX;
    T w[6];
#pragma unroll
    for (int f = 0; f < 6; ++f) {
      w[f] = A.w[f][o] - k * A.R[f][o];
      A.w[f][o] = w[f];
    }
    const T sum = ((w[0] + w[1]) + (w[2] + w[3])) + (w[4] + w[5]);
    if (!(fabs(sum) <= M2<T>::big())) bad |= kErrNonfinite;
    if (!(w[0] > T(0)) || !(w[3] > T(0))) bad |= kErrDepth;
  }
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
cudaError_t launch_step2(const Step2Args<T>& f, const Update2Args<T>& u, cudaStream_t st) {
  constexpr int TY = Tile2Y<T>::v;
  dim3 block(TX, TY);
  dim3 grid((unsigned)((f.nx + TX - 1) / TX), (unsigned)((f.ny + TY - 1) / TY));
  if (f.rho == T(1)) cart2_flux_kernel<T, false><<<grid, block, 0, st>>>(f);
  else cart2_flux_kernel<T, true><<<grid, block, 0, st>>>(f);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 ub(64, 4);
  dim3 ug((unsigned)((u.nx + 63) / 64), (unsigned)min((u.ny + 3) / 4, 4096));
  cart2_update_kernel<T><<<ug, ub, 0, st>>>(u);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_check2(const Fields6<T>& w6, int nx, int ny, int pitch, unsigned* err,
                          cudaStream_t st) {
  dim3 grid((unsigned)((nx + 127) / 128), (unsigned)(ny < 1024 ? ny : 1024));
  cart2_check_kernel<T><<<grid, 128, 0, st>>>(w6, nx, ny, pitch, err);
  return cudaGetLastError();
}

template cudaError_t launch_step2<float>(const Step2Args<float>&, const Update2Args<float>&,
                                         cudaStream_t);
template cudaError_t launch_step2<double>(const Step2Args<double>&, const Update2Args<double>&,
                                          cudaStream_t);
template cudaError_t launch_check2<float>(const Fields6<float>&, int, int, int, unsigned*,
                                          cudaStream_t);
template cudaError_t launch_check2<double>(const Fields6<double>&, int, int, int, unsigned*,
                                           cudaStream_t);

}  // namespace swe
