// swe_cart2.cu -- sm_103a kernels of the two-layer IR-Roe step on a
// Cartesian grid.
//
// Scheme: An MPI-CUDA implementation of an improved Roe method for two-layer
// shallow water systems, Sec. 2.1 (eq. (1): two superposed layers, 1 = upper,
// coupled through -g h1 dh2 and -r g h2 dh1) and Sec. 2.2 (eq. (4), steps 1-4
// with the 4x4 Roe matrix A_ij of the rotated system, CFL eq. (5)).
//
// Kernels:
//   cart2_march_kernel   one warp per (column band, row segment) marches up
//                        its rows; each lane evaluates the x-edge east of its
//                        cell and the y-edge below it (as one FP32x2
//                        evaluation in fp32), so every edge is computed once
//                        except at band and segment borders, and the edge
//                        results pass between cells by warp shuffles and
//                        registers (the idea of A multi-GPU shallow-water
//                        simulation with transport of contaminants, Figure 4,
//                        at warp level).  Each cell sums its four edges into
//                        the residual R and max-reduces sum |Gamma| ||D||,
//                        which fixes dt of this step.  FUSED: the update of
//                        the previous step is applied to every cell as it is
//                        loaded (W^n = W^{n-1} - (dt/dx) R^{n-1}, W and R
//                        alternate between two buffers) and W^n of the own
//                        cells is written;
//   cart2_update_kernel  W -= (dt/dx) R (16-byte vectors over whole rows, the
//                        padding left as it is), checks, dt bookkeeping: a
//                        lone step, and the last step of a run.
// A run of n >= 2 steps is one plain march, n - 1 fused marches and one
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

// ---- the row march -----------------------------------------------------------
// One warp per (column band, row segment).  Lane l of band b holds column
// x = kBand2 * b - 1 + l: lanes 1..30 own their columns, lanes 0 and 31 are
// the one-cell halo.  The warp marches up rows y0 - 1 .. y1 of its segment;
// at row r each lane evaluates, in one FP32x2 evaluation in fp32 (one after
// the other in fp64 and with the entropy fix), the x-edge east of its cell
// and the y-edge below it.  The west x-edge's results come from the lane on
// the left by shuffle; the residual of row r - 1 is complete once the
// y-edge above it is known (row r), and is written then.

// one cell of a row: per layer depth, discharge (x, y), sqrt(h), 1/sqrt(h);
// the bottom depth
template <typename T>
struct Cell2 {
  T h[2], qx[2], qy[2], s[2], rs[2], H;
};

template <typename T>
__device__ __forceinline__ void derive(Cell2<T>& c) {
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    c.rs[k] = M2<T>::rsq(c.h[k]);
    c.s[k] = c.h[k] * c.rs[k];
  }
}

// the cell seen from an x-edge (normal (1, 0)) or a y-edge (normal (0, 1));
// `mirror`: the reflective wall's ghost (normal discharge negated)
template <typename T>
__device__ __forceinline__ Side2<T> side2(const Cell2<T>& c, bool xdir, bool mirror) {
  Side2<T> s;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    s.h[k] = c.h[k];
    s.s[k] = c.s[k];
    s.rs[k] = c.rs[k];
    const T n = xdir ? c.qx[k] : c.qy[k];
    s.qn[k] = mirror ? -n : n;
    s.qt[k] = xdir ? c.qy[k] : c.qx[k];
  }
  s.H = c.H;
  return s;
}

template <typename T>
__device__ __forceinline__ Cell2<T> shfl_down_cell(const Cell2<T>& c) {
  Cell2<T> o;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    o.h[k] = __shfl_down_sync(kFull2, c.h[k], 1);
    o.qx[k] = __shfl_down_sync(kFull2, c.qx[k], 1);
    o.qy[k] = __shfl_down_sync(kFull2, c.qy[k], 1);
    o.s[k] = __shfl_down_sync(kFull2, c.s[k], 1);
    o.rs[k] = __shfl_down_sync(kFull2, c.rs[k], 1);
  }
  o.H = __shfl_down_sync(kFull2, c.H, 1);
  return o;
}

// Both edges of a lane: ox for (a_x, b_x), oy for (a_y, b_y); returns bit 0
// (bit 1) when the x-edge's (y-edge's) Roe matrix has real eigenvalues.
template <typename T, bool EFIX>
__device__ __forceinline__ unsigned edge_pair(const Side2<T>& ax, const Side2<T>& bx, bool wx,
                                              const Side2<T>& ay, const Side2<T>& by, bool wy,
                                              T g, T gh, T r, T ox[NEQ], T oy[NEQ]) {
  unsigned ok = edge2<T, kAdapt2<T>, EFIX>(ax, bx, g, gh, r, wx, ox) ? 1u : 0u;
  ok |= edge2<T, kAdapt2<T>, EFIX>(ay, by, g, gh, r, wy, oy) ? 2u : 0u;
  return ok;
}
__device__ __forceinline__ Side2P pack2(const Side2<float>& x, const Side2<float>& y) {
  Side2P p;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    p.h[k] = f2(x.h[k], y.h[k]);
    p.s[k] = f2(x.s[k], y.s[k]);
    p.rs[k] = f2(x.rs[k], y.rs[k]);
    p.qn[k] = f2(x.qn[k], y.qn[k]);
    p.qt[k] = f2(x.qt[k], y.qt[k]);
  }
  p.H = f2(x.H, y.H);
  return p;
}
// fp32: both edges in one evaluation on the FP32x2 pipe
template <bool EFIX>
__device__ __forceinline__ unsigned edge_pair_f32(const Side2<float>& ax, const Side2<float>& bx,
                                                  bool wx, const Side2<float>& ay,
                                                  const Side2<float>& by, bool wy, float g,
                                                  float gh, float r, float ox[NEQ],
                                                  float oy[NEQ]) {
  float2 o[NEQ];
  const unsigned ok = edge2p<EFIX>(pack2(ax, ay), pack2(bx, by), g, gh, r, wx, wy, o);
#pragma unroll
  for (int q = 0; q < NEQ; ++q) {
    ox[q] = o[q].x;
    oy[q] = o[q].y;
  }
  return ok;
}
template <>
__device__ __forceinline__ unsigned edge_pair<float, false>(
    const Side2<float>& ax, const Side2<float>& bx, bool wx, const Side2<float>& ay,
    const Side2<float>& by, bool wy, float g, float gh, float r, float ox[NEQ], float oy[NEQ]) {
  return edge_pair_f32<false>(ax, bx, wx, ay, by, wy, g, gh, r, ox, oy);
}
// (fp32 with the entropy fix: edge_pair_shared below)

// Entropy fix, fp32: the sides' own speeds (roots of side_quartic2p) are
// the same for every edge of a cell in one frame, so each lane solves its
// cell's quartics once per row, in the x- and the y-frame at once, and the
// edges take them from there: the x-edge's side b from the east lane, the
// y-edge's side a from the row below.  A wall's mirror ghost (its normal
// discharge negated) has exactly the negated roots in reverse order, every
// step of the root finding being symmetric under that sign change.
struct OwnRoots {
  float2 l[4];  // .x: the cell in the x-frame, .y: in the y-frame
  unsigned hyper;
};
__device__ __forceinline__ OwnRoots own_roots(const Cell2<float>& c, float g, float r) {
  OwnRoots o;
  o.hyper = roots2p(side_quartic2p(pack2(side2(c, true, false), side2(c, false, false)), g, r),
                    o.l);
  return o;
}
__device__ __forceinline__ unsigned edge_pair_shared(
    const Side2<float>& ax, const Side2<float>& bx, bool lw, bool rw, const Side2<float>& ay,
    const Side2<float>& by, bool bw, bool tw, const OwnRoots& cur, const float below[4],
    unsigned below_hyper, float g, float gh, float r, float ox[NEQ], float oy[NEQ]) {
  float east[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) east[k] = __shfl_down_sync(kFull2, cur.l[k].x, 1);
  const unsigned east_hyper = __shfl_down_sync(kFull2, cur.hyper & 1u, 1);
  float2 la[4], lb[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    la[k] = f2(lw ? -cur.l[3 - k].x : cur.l[k].x, bw ? -below[3 - k] : below[k]);
    lb[k] = f2(rw ? -cur.l[3 - k].x : east[k], tw ? -cur.l[3 - k].y : cur.l[k].y);
  }
  const unsigned hx = (cur.hyper & 1u) & (rw ? cur.hyper & 1u : east_hyper);
  const unsigned hy = below_hyper & ((cur.hyper >> 1) & 1u);
  float2 o[NEQ];
  const unsigned ok = edge2p<true>(pack2(ax, ay), pack2(bx, by), g, gh, r, lw || rw, bw || tw,
                                   o, la, lb, hx | (hy << 1));
#pragma unroll
  for (int q = 0; q < NEQ; ++q) {
    ox[q] = o[q].x;
    oy[q] = o[q].y;
  }
  return ok;
}

// what a cell takes from the x-edge on its west (it is side b) and from the
// y-edge below it: mass fluxes, P^+ d of the normal momentum, tangential
// fluxes, ||D|| (the order of the shuffled and carried arrays)
enum { B_M1, B_PS1, B_T1, B_M2, B_PS2, B_T2, B_D, NB };

// Resident blocks per SM the registers are held to (four-warp blocks).
#ifndef SWE_MARCH2_MIN_BLOCKS
#define SWE_MARCH2_MIN_BLOCKS 4
#endif
template <typename T, bool EFIX> struct MinBlocks2 { static constexpr int v = 1; };
template <> struct MinBlocks2<float, false> { static constexpr int v = SWE_MARCH2_MIN_BLOCKS; };
// With the entropy fix (fp32 evaluates both edges with the packed fix form,
// about 200 registers unbounded): three blocks at 168 registers, a few bytes
// spilled, ran 0.234 ms per step on the 2048^2 interface dam break against
// 0.258 ms at two blocks unspilled.
#ifndef SWE_MARCH2_MIN_BLOCKS_EFIX
#define SWE_MARCH2_MIN_BLOCKS_EFIX 3
#endif
template <> struct MinBlocks2<float, true> { static constexpr int v = SWE_MARCH2_MIN_BLOCKS_EFIX; };

// FUSED: the pass also applies the previous step's update to every cell it
// loads (W^n = W^{n-1} - (dt/dx) R^{n-1}) and writes W^n of its own cells.
template <typename T, bool ANISO, bool FUSED, bool EFIX>
__global__ void __launch_bounds__(kMarch2Warps * 32, MinBlocks2<T, EFIX>::v)
    cart2_march_kernel(const Step2Args<T> A, const Update2Args<T> U) {
  __shared__ T k_sh;
  pdl_wait();
  const T kdt = FUSED ? dt_of_step<T>(U, &k_sh) : T(0);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nx = A.nx, ny = A.ny, nb = A.nbands, ns = A.nsegs;
  const int unit = blockIdx.x * kMarch2Warps + warp;
  T tmax = T(0);
  unsigned bad = 0, hyp_ok = 1u;
  if (unit < nb * ns) {
    const int band = unit % nb, seg = unit / nb;
    const int y0 = (int)((int64_t)seg * ny / ns), y1 = (int)((int64_t)(seg + 1) * ny / ns);
    const int x = kBand2 * band - 1 + lane;
    const bool own_x = lane >= 1 && lane <= kBand2 && x < nx;
    const bool need_ex = lane <= kBand2 && x >= -1 && x <= nx - 1;  // x-edges used
    const T g = A.g, gh = T(0.5) * A.g, r = A.r, rho = A.rho;
    auto ys = [&](T v) { return ANISO ? v * rho : v; };
    // Every lane and row outside the grid reads the nearest cell of the grid
    // instead (column -1 reads column 0, column nx reads nx - 1, rows -1 and
    // ny read rows 0 and ny - 1): a wall's mirror ghost is then that copy
    // with its normal discharge negated.
    const int xc = min(max(x, 0), nx - 1);
    auto row_of = [&](int rr) -> int64_t {
      const int rc = min(max(rr, 0), ny - 1);
      return (int64_t)(rc + kPadY) * A.pitch + xc + kPadX;
    };
    int64_t o = row_of(y0 - 1);
    // row y0 - 1 into registers
    T w[6], R[6], Hn;
    auto load = [&](int64_t at, T* wv, T* rv, T& hv) {
#pragma unroll
      for (int f = 0; f < 6; ++f) wv[f] = A.w[f][at];
      if (FUSED) {
#pragma unroll
        for (int f = 0; f < 6; ++f) rv[f] = U.R[f][at];
      }
      hv = A.H[at];
    };
    load(o, w, R, Hn);
    Cell2<T> prev;
    constexpr bool SHARED = EFIX && sizeof(T) == 4;  // fp32 fix: own roots shared
    float below[4] = {0.f, 0.f, 0.f, 0.f};           // y-frame roots of row r - 1
    unsigned below_hyper = 1u;
    T xr[6], xd = T(0), yb[NB];  // row r - 1: x-part of its residual, its south edge
#pragma unroll
    for (int f = 0; f < 6; ++f) xr[f] = T(0);
#pragma unroll
    for (int q = 0; q < NB; ++q) yb[q] = T(0);
    for (int rr = y0 - 1; rr <= y1; ++rr) {
      // ---- the row: previous step's update (fused), next row's loads -----
      Cell2<T> cur;
      {
        T wc[6];
#pragma unroll
        for (int f = 0; f < 6; ++f) wc[f] = w[f];
        if (FUSED) {
#pragma unroll
          for (int f = 0; f < 6; ++f) wc[f] = upd(wc[f], kdt, R[f]);
          if (own_x && rr >= y0 && rr < y1) {
#pragma unroll
            for (int f = 0; f < 6; ++f) U.w[f][o] = wc[f];
            const T sum = ((wc[0] + wc[1]) + (wc[2] + wc[3])) + (wc[4] + wc[5]);
            if (!(fabs(sum) <= M2<T>::big())) bad |= kErrNonfinite;
            if (!(wc[0] > T(0)) || !(wc[3] > T(0))) bad |= kErrDepth;
          }
        }
        cur.h[0] = wc[0]; cur.qx[0] = wc[1]; cur.qy[0] = wc[2];
        cur.h[1] = wc[3]; cur.qx[1] = wc[4]; cur.qy[1] = wc[5];
        cur.H = Hn;
      }
      const int64_t on = row_of(rr + 1);
      if (rr < y1) load(on, w, R, Hn);
      derive(cur);
      OwnRoots own;
      if constexpr (SHARED) own = own_roots(cur, g, r);
      if (rr >= y0) {
        // ---- the x-edge east of the cell, the y-edge below it ---------------
        const Cell2<T> right = shfl_down_cell(cur);
        const bool lw = x == -1, rw = x == nx - 1;
        const bool bw = rr == 0, tw = rr == ny;
        const Side2<T> ax = side2(cur, true, lw);
        const Side2<T> bx = side2(right, true, rw);
        const Side2<T> ay = side2(prev, false, bw);
        const Side2<T> by = side2(cur, false, tw);
        T ox[NEQ], oy[NEQ];
        unsigned ok;
        if constexpr (SHARED)
          ok = edge_pair_shared(ax, bx, lw, rw, ay, by, bw, tw, own, below, below_hyper, g, gh, r,
                                ox, oy);
        else
          ok = edge_pair<T, EFIX>(ax, bx, lw || rw, ay, by, bw || tw, g, gh, r, ox, oy);
        const bool row_x = rr < y1;  // this row's x-edges are used
        if (row_x && need_ex && !(ok & 1u)) hyp_ok = 0u;
        if (own_x && !(ok & 2u)) hyp_ok = 0u;
        // ---- row r - 1 is complete: its north edge is this y-edge ---------
        if (rr - 1 >= y0 && own_x) {
          T Rn[6];
          Rn[0] = xr[0] + ys(oy[E_M1] - yb[B_M1]);
          Rn[1] = xr[1] + ys(oy[E_T1] - yb[B_T1]);
          Rn[2] = xr[2] + ys(oy[E_PM1] + yb[B_PS1]);
          Rn[3] = xr[3] + ys(oy[E_M2] - yb[B_M2]);
          Rn[4] = xr[4] + ys(oy[E_T2] - yb[B_T2]);
          Rn[5] = xr[5] + ys(oy[E_PM2] + yb[B_PS2]);
          const T ts = xd + ys(yb[B_D] + oy[E_D]);
          const int64_t ob = row_of(rr - 1);  // an owned row: inside the grid
#pragma unroll
          for (int f = 0; f < 6; ++f) A.R[f][ob] = Rn[f];
          tmax = nanmax2(tmax, ts);
        }
        // ---- this row's x-part, from the east edge and (shuffled) the west
        {
          T wv[NB];
          wv[B_M1] = __shfl_up_sync(kFull2, ox[E_M1], 1);
          wv[B_PS1] = __shfl_up_sync(kFull2, ox[E_PS1], 1);
          wv[B_T1] = __shfl_up_sync(kFull2, ox[E_T1], 1);
          wv[B_M2] = __shfl_up_sync(kFull2, ox[E_M2], 1);
          wv[B_PS2] = __shfl_up_sync(kFull2, ox[E_PS2], 1);
          wv[B_T2] = __shfl_up_sync(kFull2, ox[E_T2], 1);
          wv[B_D] = __shfl_up_sync(kFull2, ox[E_D], 1);
          xr[0] = ox[E_M1] - wv[B_M1];
          xr[1] = ox[E_PM1] + wv[B_PS1];
          xr[2] = ox[E_T1] - wv[B_T1];
          xr[3] = ox[E_M2] - wv[B_M2];
          xr[4] = ox[E_PM2] + wv[B_PS2];
          xr[5] = ox[E_T2] - wv[B_T2];
          xd = wv[B_D] + ox[E_D];
          yb[B_M1] = oy[E_M1];
          yb[B_PS1] = oy[E_PS1];
          yb[B_T1] = oy[E_T1];
          yb[B_M2] = oy[E_M2];
          yb[B_PS2] = oy[E_PS2];
          yb[B_T2] = oy[E_T2];
          yb[B_D] = oy[E_D];
        }
      }
      prev = cur;
      if constexpr (SHARED) {
#pragma unroll
        for (int k = 0; k < 4; ++k) below[k] = own.l[k].y;
        below_hyper = (own.hyper >> 1) & 1u;
      }
      o = on;
    }
  }
  // hyperbolicity and the checks of this warp, the block's max of sum L ||D||
  if (!__all_sync(kFull2, hyp_ok != 0u) && lane == 0) atomicOr(A.err, kErrHyperbolic);
  if (FUSED && bad) atomicOr(A.err, bad);
  pdl_trigger();
  block_max_publish<T, kMarch2Warps>(tmax, A.tmax_out);
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
cudaError_t march2_occupancy(int* blocks_per_sm, bool efix) {
  return efix ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                    blocks_per_sm, cart2_march_kernel<T, false, true, true>, kMarch2Warps * 32, 0)
              : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                    blocks_per_sm, cart2_march_kernel<T, false, true, false>, kMarch2Warps * 32,
                    0);
}

template <typename T, bool FUSED>
cudaError_t launch_march2(const Step2Args<T>& f, const Update2Args<T>& u, cudaStream_t st) {
  const int units = f.nbands * f.nsegs;
  const dim3 grid((unsigned)((units + kMarch2Warps - 1) / kMarch2Warps));
  const dim3 block(kMarch2Warps * 32);
  const bool aniso = f.rho != T(1);
  if (f.efix)
    return aniso ? launch_pdl(cart2_march_kernel<T, true, FUSED, true>, grid, block, 0, st, f, u)
                 : launch_pdl(cart2_march_kernel<T, false, FUSED, true>, grid, block, 0, st, f, u);
  return aniso ? launch_pdl(cart2_march_kernel<T, true, FUSED, false>, grid, block, 0, st, f, u)
               : launch_pdl(cart2_march_kernel<T, false, FUSED, false>, grid, block, 0, st, f, u);
}

template <typename T>
cudaError_t launch_flux2(const Step2Args<T>& f, cudaStream_t st) {
  return launch_march2<T, false>(f, Update2Args<T>{}, st);
}

template <typename T>
cudaError_t launch_fused2(const Step2Args<T>& f, const Update2Args<T>& u, cudaStream_t st) {
  return launch_march2<T, true>(f, u, st);
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

template cudaError_t march2_occupancy<float>(int*, bool);
template cudaError_t march2_occupancy<double>(int*, bool);
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
