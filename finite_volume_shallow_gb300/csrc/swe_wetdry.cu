// swe_wetdry.cu -- sm_103a kernels of the one-layer step with wet/dry fronts
// (swe_params.wet_dry = 1) on a Cartesian grid.
//
// Scheme: the IR-Roe step of An MPI-CUDA implementation of an improved Roe
// method for two-layer shallow water systems, Sec. 2.2 (eq. (4), steps 1-4,
// CFL eq. (5)) with one layer and a passive pollutant, in the flux form of
// eq. (4), plus a wet/dry treatment the pages do not give, made of two
// published techniques:
//  - Brufau, Vazquez-Cendon and Garcia-Navarro, "A numerical model for the
//    flooding and drying of irregular domains" (Int. J. Numer. Meth. Fluids
//    39, 2002): a cell with h <= h_dry is dry (no velocity, no
//    concentration); an edge between two dry cells passes nothing; an edge
//    between a wet cell and a dry cell whose bed is at or above the wet
//    free surface is a reflective wall for both; other wet/dry edges take
//    the Roe flux with the dry side at rest;
//  - Bollermann, Chen, Kurganov and Noelle, "A well-balanced reconstruction
//    of wet/dry fronts for the shallow water equations" (J. Sci. Comput. 56,
//    2013): the draining time tau_i = h_i |V_i| / (mass leaving cell i per
//    unit time) limits every term of an edge to min(1, tau_d / dt), d the
//    cell its mass flux leaves, so that no depth turns negative.
//
// Two kernels per step:
//   wd_speed_kernel  one thread per cell: sum_e L ||D_e|| over its four edges
//                    of W^n with the rules above, each edge evaluated once per
//                    block (its block maximum published with one atomic: dt
//                    of this step, eq. (5));
//   wd_tile_kernel   one block per 32 x 16 tile: the tile and a two-cell ring
//                    of W^n into shared memory; every edge that the tile and
//                    its one-cell ring need, once per block (mass flux m
//                    a -> b, each side's normal momentum flux in flux form
//                    -- a: Phi^-[1]; b: Phi^-[1] + g hbar (H_b - H_a) --,
//                    tangential momentum and pollutant fluxes); the draining
//                    time of the tile's cells and of the ring (a tile edge's
//                    donor may lie in the ring); then each cell of the tile:
//                    the limit of its four edges, the update of eq. (4) into
//                    the other state buffer, clean-up of dry cells, checks;
//                    block (0, 0) keeps the clock.  Edges on a tile's border
//                    are evaluated by both tiles with the same code and
//                    inputs, so every cell sees one value per edge.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "swe_fastmath.cuh"
#include "swe_internal.h"

namespace swe {
namespace {

constexpr unsigned kFullWd = 0xffffffffu;

template <typename T> struct Wm;
template <> struct Wm<float> {  // MUFU approximations (a few ulp)
  __device__ static __forceinline__ float rcp(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
  }
  __device__ static __forceinline__ float sqrt_(float x) {
    float r;
    asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
  }
};
template <> struct Wm<double> {  // Newton-refined reciprocal, CUDA's square root
  __device__ static __forceinline__ double rcp(double x) { return rcp_nr(x); }
  __device__ static __forceinline__ double sqrt_(double x) { return sqrt(x); }
};

// One side of an edge in the frame of its normal.
template <typename T>
struct SideW {
  T h, qn, qt, hC, H;
};

// d, db: ||D|| of the edge as each side counts it in eq. (5) (they differ
// only where the edge is a wall for one side and passes nothing to the other)
template <typename T>
struct EdgeW {
  T m, fa, fb, t, c, d, db;
};

// IR-Roe flux of one edge (a -> b), both sides taking part.  A dry side
// (h <= h_dry) is at rest and carries no concentration.  EFIX: the
// Harten-Hyman entropy fix as viscosity per wave on the state jump.
template <typename T, bool EFIX>
__device__ __forceinline__ EdgeW<T> roe_edge(const SideW<T>& a, const SideW<T>& b, T g, T hdry) {
  const bool dry_a = a.h <= hdry, dry_b = b.h <= hdry;
  const T qna = dry_a ? T(0) : a.qn, qnb = dry_b ? T(0) : b.qn;
  const T sa = Wm<T>::sqrt_(a.h), sb = Wm<T>::sqrt_(b.h);
  const T ia = dry_a ? T(0) : Wm<T>::rcp(a.h), ib = dry_b ? T(0) : Wm<T>::rcp(b.h);
  const T ua = qna * ia, ub = qnb * ib;  // normal velocities
  // Roe averages: sqrt(h)-weighted velocity, arithmetic depth
  const T un = (sa * ua + sb * ub) * Wm<T>::rcp(sa + sb);
  const T hbar = T(0.5) * (a.h + b.h);
  const T c = Wm<T>::sqrt_(g * hbar);
  const T l1 = un - c, l2 = un + c;
  // fluctuation d = F(W_b) - F(W_a) - (0, g hbar (H_b - H_a))
  const T fa1 = qna * ua + T(0.5) * g * a.h * a.h;
  const T fb1 = qnb * ub + T(0.5) * g * b.h * b.h;
  const T d0 = qnb - qna;
  const T d1 = (fb1 - fa1) - g * hbar * (b.H - a.H);
  // alpha = K^-1 d with K = [[1, 1], [l1, l2]], det = 2c; P^- d = sum_k w_k alpha_k K_k
  const T i2c = Wm<T>::rcp(c + c);
  const T al1 = (l2 * d0 - d1) * i2c, al2 = (d1 - l1 * d0) * i2c;
  const T w1 = l1 < T(0) ? T(1) : (l1 > T(0) ? T(0) : T(0.5));
  const T w2 = l2 < T(0) ? T(1) : (l2 > T(0) ? T(0) : T(0.5));
  T p0 = w1 * al1 + w2 * al2;
  T p1 = w1 * al1 * l1 + w2 * al2 * l2;
  if (EFIX) {
    const T ca = Wm<T>::sqrt_(g * a.h), cb = Wm<T>::sqrt_(g * b.h);
    const T dh = b.h - a.h;
    const T be1 = (l2 * dh - d0) * i2c, be2 = (d0 - l1 * dh) * i2c;
    const T del1 = fmax(T(0), fmax(l1 - (ua - ca), (ub - cb) - l1));
    const T del2 = fmax(T(0), fmax(l2 - (ua + ca), (ub + cb) - l2));
    T n1 = T(0), n2 = T(0);
    if (fabs(l1) < del1) n1 = T(0.5) * (fabs(l1) - (l1 * l1 + del1 * del1) * Wm<T>::rcp(del1 + del1)) * be1;
    if (fabs(l2) < del2) n2 = T(0.5) * (fabs(l2) - (l2 * l2 + del2 * del2) * Wm<T>::rcp(del2 + del2)) * be2;
    p0 += n1 + n2;
    p1 += n1 * l1 + n2 * l2;
  }
  EdgeW<T> e;
  e.m = qna + p0;
  e.fa = fa1 + p1;
  e.fb = e.fa + g * hbar * (b.H - a.H);
  const bool up = e.m > T(0);
  const T ut = up ? (dry_a ? T(0) : a.qt * ia) : (dry_b ? T(0) : b.qt * ib);
  const T cc = up ? (dry_a ? T(0) : a.hC * ia) : (dry_b ? T(0) : b.hC * ib);
  e.t = e.m * ut;
  e.c = e.m * cc;
  e.d = fabs(un) + c;
  e.db = e.d;
  return e;
}

// A reflective wall seen from side s (mirror ghost: same state, normal
// discharge negated): only the normal momentum flux of s and ||D|| remain;
// the mass, tangential and pollutant fluxes are algebraically zero.
template <typename T, bool EFIX>
__device__ __forceinline__ EdgeW<T> wall_of(const SideW<T>& s, T g, T hdry) {
  SideW<T> gst = s;
  gst.qn = -s.qn;
  EdgeW<T> e = roe_edge<T, EFIX>(s, gst, g, hdry);
  e.m = e.t = e.c = T(0);
  return e;
}

// Every case of an edge a -> b (a_wall / b_wall: that side is outside the
// domain and takes the other's mirror).  The result is in the frame a -> b:
// a adds L (m, fa, t, c), b subtracts L (m, fb, t, c) -- fb being b's own
// outward normal momentum flux (along b -> a), like Phi^+ of a Roe edge.
template <typename T, bool EFIX>
__device__ __forceinline__ EdgeW<T> edge_any(const SideW<T>& a, const SideW<T>& b, bool a_wall,
                                            bool b_wall, T g, T hdry) {
  EdgeW<T> z;
  z.m = z.fa = z.fb = z.t = z.c = z.d = z.db = T(0);
  if (b_wall) {  // domain wall on b's side: a's own wall flux
    EdgeW<T> w = wall_of<T, EFIX>(a, g, hdry);
    if (a.h <= hdry) w = z;
    w.fb = w.db = T(0);
    return w;
  }
  if (a_wall) {  // b's own wall flux; b subtracts fb along a -> b
    SideW<T> br = b;
    br.qn = -b.qn;  // b's frame: outward normal points back towards a
    EdgeW<T> w = wall_of<T, EFIX>(br, g, hdry);
    if (b.h <= hdry) w = z;
    z.fb = w.fa;
    z.db = w.d;
    return z;
  }
  const bool dry_a = a.h <= hdry, dry_b = b.h <= hdry;
  if (dry_a && dry_b) return z;
  if (dry_b && -b.H >= a.h - a.H) {  // dry bank at or above a's surface
    EdgeW<T> w = wall_of<T, EFIX>(a, g, hdry);
    w.fb = w.db = T(0);
    return w;
  }
  if (dry_a && -a.H >= b.h - b.H) {
    SideW<T> br = b;
    br.qn = -b.qn;
    EdgeW<T> w = wall_of<T, EFIX>(br, g, hdry);
    z.fb = w.fa;
    z.db = w.d;
    return z;
  }
  return roe_edge<T, EFIX>(a, b, g, hdry);
}

// Both sides' ||D|| of an edge a -> b under the same rules as edge_any
// (the Roe speed |u| + c; sqrt(g h) for the wet side of a wall; 0 for a
// side that receives nothing).
template <typename T>
__device__ __forceinline__ void edge_speeds(const SideW<T>& a, const SideW<T>& b, bool a_wall,
                                            bool b_wall, T g, T hdry, T& da, T& db) {
  auto wall_d = [&](const SideW<T>& w) { return w.h <= hdry ? T(0) : Wm<T>::sqrt_(g * w.h); };
  da = db = T(0);
  if (b_wall) { da = wall_d(a); return; }
  if (a_wall) { db = wall_d(b); return; }
  const bool dry_a = a.h <= hdry, dry_b = b.h <= hdry;
  if (dry_a && dry_b) return;
  if (dry_b && -b.H >= a.h - a.H) { da = wall_d(a); return; }
  if (dry_a && -a.H >= b.h - b.H) { db = wall_d(b); return; }
  const T sa = Wm<T>::sqrt_(a.h), sb = Wm<T>::sqrt_(b.h);
  const T ua = dry_a ? T(0) : a.qn * Wm<T>::rcp(a.h), ub = dry_b ? T(0) : b.qn * Wm<T>::rcp(b.h);
  const T un = (sa * ua + sb * ub) * Wm<T>::rcp(sa + sb);
  da = db = fabs(un) + Wm<T>::sqrt_(g * (T(0.5) * (a.h + b.h)));
}

template <typename T>
struct WdArgs {
  const T* win[4];  // W^n: h, qx, qy, hC (padded layout)
  T* wout[4];       // W^{n+1}
  const T* H;
  int nx, ny, pitch;
  T g, hdry, dx, dy;
  double two_cfl, area;
  void* tmax;       // max over cells of sum L ||D|| of W^n (starts at 0)
  void* tmax_clear; // the slot the next step reduces into
  double* dt_hist;
  double* t_dev;
  int64_t step;
  unsigned* err;
};

template <typename T>
__device__ __forceinline__ T nanmax_wd(T acc, T x) {
  return (x > acc || x != x) ? x : acc;
}
__device__ __forceinline__ void atomic_max_wd(void* slot, float v) {
  atomicMax(reinterpret_cast<unsigned int*>(slot), __float_as_uint(v));
}
__device__ __forceinline__ void atomic_max_wd(void* slot, double v) {
  atomicMax(reinterpret_cast<unsigned long long*>(slot),
            static_cast<unsigned long long>(__double_as_longlong(v)));
}

template <typename T>
__global__ void __launch_bounds__(256) wd_speed_kernel(const WdArgs<T> A) {
  // 32 x 8 threads, one per cell.  Each thread evaluates the east and north
  // edges of its cell (the cell is side a) and hands side b's speed to the
  // neighbour through shared memory; the block's first column and first row
  // evaluate their west and south edges themselves.  Every edge is thus
  // evaluated once inside a block (the two sides can differ: a bank is a
  // wall for one of them only).
  __shared__ T part[8];
  __shared__ T east_b[8][33], north_b[8][32];
  pdl_wait();
  const int tx = threadIdx.x, ty = threadIdx.y;
  const int i = blockIdx.x * blockDim.x + tx;
  const int j = blockIdx.y * blockDim.y + ty;
  const int nx = A.nx, ny = A.ny;
  const bool in = i < nx && j < ny;
  T s = T(0), dEa = T(0), dNa = T(0), dW = T(0), dS = T(0), dEb = T(0), dNb = T(0);
  if (in) {
    // the cell and the neighbours it needs (a missing one: the cell itself,
    // unused behind the wall), h, q_x, q_y and H of each read once
    const int64_t o = (int64_t)(j + kPadY) * A.pitch + i + kPadX;
    auto side = [&](int64_t at, bool xdir) {
      SideW<T> c;
      c.h = A.win[0][at];
      c.qn = xdir ? A.win[1][at] : A.win[2][at];
      c.qt = T(0);
      c.hC = T(0);
      c.H = A.H[at];
      return c;
    };
    const SideW<T> cx = side(o, true), cy = side(o, false);
    T unused;
    // East, North (the cell is a), West, South (the cell is b)
    edge_speeds(cx, side(i + 1 < nx ? o + 1 : o, true), false, i + 1 >= nx, A.g, A.hdry, dEa,
                dEb);
    edge_speeds(cy, side(j + 1 < ny ? o + A.pitch : o, false), false, j + 1 >= ny, A.g, A.hdry,
                dNa, dNb);
    if (tx == 0)
      edge_speeds(side(i > 0 ? o - 1 : o, true), cx, i == 0, false, A.g, A.hdry, unused, dW);
    if (ty == 0)
      edge_speeds(side(j > 0 ? o - A.pitch : o, false), cy, j == 0, false, A.g, A.hdry, unused,
                  dS);
  }
  east_b[ty][tx] = dEb;
  north_b[ty][tx] = dNb;
  __syncthreads();
  if (in) {
    if (tx > 0) dW = east_b[ty][tx - 1];
    if (ty > 0) dS = north_b[ty - 1][tx];
    s = (A.dy * dEa + A.dx * dNa) + (A.dy * dW + A.dx * dS);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s = nanmax_wd(s, __shfl_xor_sync(kFullWd, s, o));
  const int t = threadIdx.y * blockDim.x + threadIdx.x;
  if ((t & 31) == 0) part[t >> 5] = s;
  __syncthreads();
  if (t < 32) {
    s = t < (int)(blockDim.x * blockDim.y / 32) ? part[t] : T(0);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = nanmax_wd(s, __shfl_xor_sync(kFullWd, s, o));
    if (t == 0 && (s > T(0) || s != s)) atomic_max_wd(A.tmax, s);
  }
  pdl_trigger();
}

// tile of TX x TY cells; shared memory holds the cells of the tile and a
// two-cell ring, the x- and y-edges of the tile and a one-cell ring, and the
// draining times of the tile and a one-cell ring
constexpr int kWdTX = 32, kWdTY = 16;
constexpr int kCX = kWdTX + 4, kCY = kWdTY + 4;  // cells (x0 - 2 + i, y0 - 2 + j)
constexpr int kXX = kWdTX + 3, kXY = kWdTY + 2;  // x-edge (ii, jj): cells (x0-2+ii | x0-1+ii), row y0-1+jj
constexpr int kYX = kWdTX + 2, kYY = kWdTY + 3;  // y-edge (ii, jj): column x0-1+ii, rows (y0-2+jj | y0-1+jj)
constexpr int kRX = kWdTX + 2, kRY = kWdTY + 2;  // ring cells (x0 - 1 + i, y0 - 1 + j)
enum { TE_M, TE_FA, TE_FB, TE_T, TE_C, TE_N };

template <typename T>
struct WdSmem {
  T c[5][kCY][kCX];         // h, qx, qy, hC, H
  T ex[TE_N][kXY][kXX];
  T ey[TE_N][kYY][kYX];
  T tau[kRY][kRX];
  T kdt;
  int bad_dt;
};

template <typename T>
__device__ __forceinline__ SideW<T> sm_side(const WdSmem<T>& S, int j, int i, bool xdir) {
  SideW<T> s;
  s.h = S.c[0][j][i];
  s.qn = xdir ? S.c[1][j][i] : S.c[2][j][i];
  s.qt = xdir ? S.c[2][j][i] : S.c[1][j][i];
  s.hC = S.c[3][j][i];
  s.H = S.c[4][j][i];
  return s;
}

template <typename T, bool EFIX>
__global__ void __launch_bounds__(kWdTX * kWdTY) wd_tile_kernel(const WdArgs<T> A) {
  extern __shared__ __align__(16) unsigned char wd_smem[];
  WdSmem<T>& S = *reinterpret_cast<WdSmem<T>*>(wd_smem);
  const int nx = A.nx, ny = A.ny;
  const int x0 = blockIdx.x * kWdTX, y0 = blockIdx.y * kWdTY;
  const int t = threadIdx.y * kWdTX + threadIdx.x;
  constexpr int NT = kWdTX * kWdTY;
  pdl_wait();
  if (t == 0) {
    const T tm = *reinterpret_cast<const T*>(A.tmax);
    // dt = min_i 2 cfl |V_i| / sum L ||D|| (eq. (5)); no wet edge at all
    // (every cell dry) leaves no finite dt
    const double dt = A.two_cfl * A.area / (double)tm;
    S.bad_dt = !(tm > T(0)) || !isfinite(dt);
    S.kdt = (T)dt;
    if (blockIdx.x == 0 && blockIdx.y == 0) {
      A.dt_hist[A.step % kHistCap] = dt;
      *A.t_dev += dt;
      if (sizeof(T) == 4) *reinterpret_cast<unsigned*>(A.tmax_clear) = 0u;
      else *reinterpret_cast<unsigned long long*>(A.tmax_clear) = 0ull;
      if (S.bad_dt) atomicOr(A.err, kErrNonfinite);
    }
  }
  // cells of the tile and a two-cell ring; outside the grid the nearest
  // grid cell (never used as such: edges to it are walls)
  for (int k = t; k < kCX * kCY; k += NT) {
    const int i = k % kCX, j = k / kCX;
    const int gx = min(max(x0 - 2 + i, 0), nx - 1), gy = min(max(y0 - 2 + j, 0), ny - 1);
    const int64_t o = (int64_t)(gy + kPadY) * A.pitch + gx + kPadX;
#pragma unroll
    for (int f = 0; f < 4; ++f) S.c[f][j][i] = A.win[f][o];
    S.c[4][j][i] = A.H[o];
  }
  __syncthreads();
  // edges of the tile and its one-cell ring
  auto inside = [&](int gx, int gy) { return gx >= 0 && gx < nx && gy >= 0 && gy < ny; };
  for (int k = t; k < kXX * kXY + kYX * kYY; k += NT) {
    EdgeW<T> e;
    if (k < kXX * kXY) {
      const int ii = k % kXX, jj = k / kXX;
      const int gy = y0 - 1 + jj, ga = x0 - 2 + ii;
      const bool ia = inside(ga, gy), ib = inside(ga + 1, gy);
      e.m = e.fa = e.fb = e.t = e.c = T(0);
      if (ia || ib)
        e = edge_any<T, EFIX>(sm_side(S, jj + 1, ii, true), sm_side(S, jj + 1, ii + 1, true),
                              !ia, !ib, A.g, A.hdry);
      S.ex[TE_M][jj][ii] = e.m;
      S.ex[TE_FA][jj][ii] = e.fa;
      S.ex[TE_FB][jj][ii] = e.fb;
      S.ex[TE_T][jj][ii] = e.t;
      S.ex[TE_C][jj][ii] = e.c;
    } else {
      const int kk = k - kXX * kXY;
      const int ii = kk % kYX, jj = kk / kYX;
      const int gx = x0 - 1 + ii, ga = y0 - 2 + jj;
      const bool ia = inside(gx, ga), ib = inside(gx, ga + 1);
      e.m = e.fa = e.fb = e.t = e.c = T(0);
      if (ia || ib)
        e = edge_any<T, EFIX>(sm_side(S, jj, ii + 1, false), sm_side(S, jj + 1, ii + 1, false),
                              !ia, !ib, A.g, A.hdry);
      S.ey[TE_M][jj][ii] = e.m;
      S.ey[TE_FA][jj][ii] = e.fa;
      S.ey[TE_FB][jj][ii] = e.fb;
      S.ey[TE_T][jj][ii] = e.t;
      S.ey[TE_C][jj][ii] = e.c;
    }
  }
  __syncthreads();
  // draining time of the tile's cells and the ring: h |V| / mass leaving per
  // unit time (East, North, West, South: (E + N) + (W + S))
  const T ly = A.dy, lx = A.dx;
  for (int k = t; k < kRX * kRY; k += NT) {
    const int i = k % kRX, j = k / kRX;
    const T oE = fmax(ly * S.ex[TE_M][j][i + 1], T(0));
    const T oN = fmax(lx * S.ey[TE_M][j + 1][i], T(0));
    const T oW = fmax(-(ly * S.ex[TE_M][j][i]), T(0));
    const T oS = fmax(-(lx * S.ey[TE_M][j][i]), T(0));
    const T M = (oE + oN) + (oW + oS);
    S.tau[j][i] = M > T(0) ? S.c[0][j + 1][i + 1] * (T)A.area / M : T(INFINITY);
  }
  __syncthreads();
  // the update of the tile's own cell
  const int ti = threadIdx.x, tj = threadIdx.y;
  const int gx = x0 + ti, gy = y0 + tj;
  unsigned bad = 0;
  if (gx < nx && gy < ny && !S.bad_dt) {
    const T dt = S.kdt;
    const int ri = ti + 1, rj = tj + 1;  // ring coordinates of the cell
    const T r0 = fmin(T(1), S.tau[rj][ri] / dt);
    auto theta = [&](T m_out, bool nb_in, int ni, int nj) -> T {
      if (m_out > T(0)) return r0;
      if (m_out < T(0) && nb_in) return fmin(T(1), S.tau[nj][ni] / dt);
      return T(1);
    };
    const T mE = ly * S.ex[TE_M][rj][ri + 1], mN = lx * S.ey[TE_M][rj + 1][ri];
    const T mW = ly * S.ex[TE_M][rj][ri], mS = lx * S.ey[TE_M][rj][ri];
    const T tE = theta(mE, gx + 1 < nx, ri + 1, rj), tN = theta(mN, gy + 1 < ny, ri, rj + 1);
    const T tW = theta(-mW, gx > 0, ri - 1, rj), tS = theta(-mS, gy > 0, ri, rj - 1);
    T fE[4], fN[4], fW[4], fS[4];
    fE[0] = tE * mE;
    fE[1] = tE * (ly * S.ex[TE_FA][rj][ri + 1]);
    fE[2] = tE * (ly * S.ex[TE_T][rj][ri + 1]);
    fE[3] = tE * (ly * S.ex[TE_C][rj][ri + 1]);
    fN[0] = tN * mN;
    fN[1] = tN * (lx * S.ey[TE_T][rj + 1][ri]);
    fN[2] = tN * (lx * S.ey[TE_FA][rj + 1][ri]);
    fN[3] = tN * (lx * S.ey[TE_C][rj + 1][ri]);
    fW[0] = -(tW * mW);
    fW[1] = -(tW * (ly * S.ex[TE_FB][rj][ri]));
    fW[2] = -(tW * (ly * S.ex[TE_T][rj][ri]));
    fW[3] = -(tW * (ly * S.ex[TE_C][rj][ri]));
    fS[0] = -(tS * mS);
    fS[1] = -(tS * (lx * S.ey[TE_T][rj][ri]));
    fS[2] = -(tS * (lx * S.ey[TE_FB][rj][ri]));
    fS[3] = -(tS * (lx * S.ey[TE_C][rj][ri]));
    const T kk = dt / (T)A.area;
    T w[4];
#pragma unroll
    for (int f = 0; f < 4; ++f) w[f] = S.c[f][tj + 2][ti + 2] - kk * ((fE[f] + fN[f]) + (fW[f] + fS[f]));
    // clean-up: a depth below zero is rounding; a dry cell keeps no discharge
    if (w[0] < T(0)) w[0] = T(0);
    if (w[0] <= A.hdry) w[1] = w[2] = T(0);
    const T sum = (w[0] + w[1]) + (w[2] + w[3]);
    if (!isfinite(sum)) bad |= kErrNonfinite;
    const int64_t o = (int64_t)(gy + kPadY) * A.pitch + gx + kPadX;
#pragma unroll
    for (int f = 0; f < 4; ++f) A.wout[f][o] = w[f];
  }
  if (bad) atomicOr(A.err, bad);
  pdl_trigger();
}

// initial / restarted state: finite, depths >= 0
template <typename T>
__global__ void wd_check_kernel(const T* h, const T* qx, const T* qy, const T* hC, int nx, int ny,
                                int pitch, unsigned* err) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  unsigned bad = 0;
  for (int j = blockIdx.y; i < nx && j < ny; j += gridDim.y) {
    const int64_t o = (int64_t)(j + kPadY) * pitch + i + kPadX;
    if (!(isfinite(h[o]) && isfinite(qx[o]) && isfinite(qy[o]) && isfinite(hC[o])))
      bad |= kErrNonfinite;
    else if (!(h[o] >= T(0)))
      bad |= kErrDepth;
  }
  if (bad) atomicOr(err, bad);
}

}  // namespace

template <typename T>
cudaError_t launch_wd_step(const WdStepArgs& a, cudaStream_t st, const cudaEvent_t* marks) {
  WdArgs<T> A;
  for (int f = 0; f < 4; ++f) {
    A.win[f] = (const T*)a.win[f];
    A.wout[f] = (T*)a.wout[f];
  }
  A.H = (const T*)a.H;
  A.nx = a.nx;
  A.ny = a.ny;
  A.pitch = a.pitch;
  A.g = (T)a.g;
  A.hdry = (T)a.h_dry;
  A.dx = (T)a.dx;
  A.dy = (T)a.dy;
  A.two_cfl = a.two_cfl;
  A.area = a.dx * a.dy;
  A.tmax = a.tmax_slot;
  A.tmax_clear = a.tmax_clear;
  A.dt_hist = a.dt_hist;
  A.t_dev = a.t_dev;
  A.step = a.step;
  A.err = a.err;
  const dim3 blk(kWdTX, kWdTY), sblk(32, 8);
  const dim3 grid((unsigned)((a.nx + kWdTX - 1) / kWdTX), (unsigned)((a.ny + kWdTY - 1) / kWdTY));
  const dim3 sgrid((unsigned)((a.nx + 31) / 32), (unsigned)((a.ny + 7) / 8));
  const size_t smem = sizeof(WdSmem<T>);
  cudaError_t e;
  if (marks && (e = cudaEventRecord(marks[0], st)) != cudaSuccess) return e;
  if ((e = launch_pdl(wd_speed_kernel<T>, sgrid, sblk, 0, st, A)) != cudaSuccess) return e;
  if (marks && (e = cudaEventRecord(marks[1], st)) != cudaSuccess) return e;
  e = a.efix ? launch_pdl(wd_tile_kernel<T, true>, grid, blk, smem, st, A)
             : launch_pdl(wd_tile_kernel<T, false>, grid, blk, smem, st, A);
  if (e != cudaSuccess) return e;
  if (marks && (e = cudaEventRecord(marks[2], st)) != cudaSuccess) return e;
  return cudaSuccess;
}

template <typename T>
cudaError_t wd_prepare() {
  // the tile's shared memory exceeds the default 48 KB in fp64: allow it on
  // the current device (function attributes are per device)
  const int smem = (int)sizeof(WdSmem<T>);
  cudaError_t e = cudaFuncSetAttribute(wd_tile_kernel<T, true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(wd_tile_kernel<T, false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

template <typename T>
cudaError_t launch_wd_check(const T* const* w, int nx, int ny, int pitch, unsigned* err,
                            cudaStream_t st) {
  dim3 grid((unsigned)((nx + 127) / 128), (unsigned)(ny < 1024 ? ny : 1024));
  wd_check_kernel<T><<<grid, 128, 0, st>>>(w[0], w[1], w[2], w[3], nx, ny, pitch, err);
  return cudaGetLastError();
}

template cudaError_t launch_wd_step<float>(const WdStepArgs&, cudaStream_t, const cudaEvent_t*);
template cudaError_t launch_wd_step<double>(const WdStepArgs&, cudaStream_t, const cudaEvent_t*);
template cudaError_t wd_prepare<float>();
template cudaError_t wd_prepare<double>();
template cudaError_t launch_wd_check<float>(const float* const*, int, int, int, unsigned*,
                                            cudaStream_t);
template cudaError_t launch_wd_check<double>(const double* const*, int, int, int, unsigned*,
                                             cudaStream_t);

}  // namespace swe
