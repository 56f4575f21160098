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
// Three kernels per step (the draining time of a cell needs all of its
// edges, and each edge's limit the draining time of its donor):
//   wd_edge_kernel    one thread per grid vertex (i, j): the x-edge on the
//                     left of cell (i, j) and the y-edge below it, each edge
//                     once: mass flux m (a -> b), each side's normal momentum
//                     flux (a: Phi^-[1]; b: Phi^-[1] + g hbar (H_b - H_a)),
//                     tangential momentum flux, pollutant flux, ||D|| as
//                     each side counts it;
//   wd_cell_kernel    one thread per cell: sum_e L ||D_e|| (its block maximum
//                     published with one atomic: dt of this step, eq. (5))
//                     and the draining time tau_i;
//   wd_update_kernel  one thread per cell: dt, the limit of each of its four
//                     edges, the update of eq. (4) in place, clean-up of dry
//                     cells, checks, the clock.
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

// per-edge record (structure of arrays): field q of an edge at q * stride + e
enum { WD_M, WD_FA, WD_FB, WD_T, WD_C, WD_DA, WD_DB, WD_NE };

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

template <typename T>
struct WdArgs {
  T* w[4];          // h, qx, qy, hC (padded layout), updated in place
  const T* H;
  int nx, ny, pitch;
  T g, hdry, dx, dy;
  T* ex;            // x-edge records: (nx + 1) * ny per field, edge (ie, j) at j * (nx + 1) + ie
  T* ey;            // y-edge records: nx * (ny + 1) per field, edge (i, je) at je * nx + i
  int64_t xs, ys;   // field strides of ex and ey
  T* tau;           // draining time per cell (j * nx + i)
  double two_cfl, area;
  void* tmax_out;   // wd_cell_kernel: max over cells of sum L ||D|| (starts at 0)
  const void* tmax_in;
  void* tmax_clear;
  double* dt_hist;
  double* t_dev;
  int64_t step;
  unsigned* err;
  int efix;
};

template <typename T>
__device__ __forceinline__ SideW<T> load_side(const WdArgs<T>& A, int i, int j, bool xdir) {
  const int64_t o = (int64_t)(j + kPadY) * A.pitch + i + kPadX;
  SideW<T> s;
  s.h = A.w[0][o];
  s.qn = xdir ? A.w[1][o] : A.w[2][o];
  s.qt = xdir ? A.w[2][o] : A.w[1][o];
  s.hC = A.w[3][o];
  s.H = A.H[o];
  return s;
}

template <typename T, bool EFIX>
__global__ void __launch_bounds__(256) wd_edge_kernel(const WdArgs<T> A) {
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;  // 0..nx
  const int j = blockIdx.y * blockDim.y + threadIdx.y;  // 0..ny
  const int nx = A.nx, ny = A.ny;
  if (i <= nx && j < ny) {  // x-edge between cells (i - 1, j) and (i, j)
    const bool aw = i == 0, bw = i == nx;
    const SideW<T> a = load_side(A, aw ? i : i - 1, j, true);
    const SideW<T> b = load_side(A, bw ? i - 1 : i, j, true);
    const EdgeW<T> e = edge_any<T, EFIX>(a, b, aw, bw, A.g, A.hdry);
    const int64_t k = (int64_t)j * (nx + 1) + i;
    A.ex[WD_M * A.xs + k] = e.m;
    A.ex[WD_FA * A.xs + k] = e.fa;
    A.ex[WD_FB * A.xs + k] = e.fb;
    A.ex[WD_T * A.xs + k] = e.t;
    A.ex[WD_C * A.xs + k] = e.c;
    A.ex[WD_DA * A.xs + k] = e.d;
    A.ex[WD_DB * A.xs + k] = e.db;
  }
  if (i < nx && j <= ny) {  // y-edge between cells (i, j - 1) and (i, j)
    const bool aw = j == 0, bw = j == ny;
    const SideW<T> a = load_side(A, i, aw ? j : j - 1, false);
    const SideW<T> b = load_side(A, i, bw ? j - 1 : j, false);
    // (the sides carry q_x as their tangential discharge, so e.t is the
    // x-momentum flux m u_x^* itself)
    const EdgeW<T> e = edge_any<T, EFIX>(a, b, aw, bw, A.g, A.hdry);
    const int64_t k = (int64_t)j * nx + i;
    A.ey[WD_M * A.ys + k] = e.m;
    A.ey[WD_FA * A.ys + k] = e.fa;
    A.ey[WD_FB * A.ys + k] = e.fb;
    A.ey[WD_T * A.ys + k] = e.t;
    A.ey[WD_C * A.ys + k] = e.c;
    A.ey[WD_DA * A.ys + k] = e.d;
    A.ey[WD_DB * A.ys + k] = e.db;
  }
  pdl_trigger();
}

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
__global__ void __launch_bounds__(256) wd_cell_kernel(const WdArgs<T> A) {
  __shared__ T part[8];
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int j = blockIdx.y * blockDim.y + threadIdx.y;
  const int nx = A.nx, ny = A.ny;
  T s = T(0);
  if (i < nx && j < ny) {
    const int64_t kw = (int64_t)j * (nx + 1) + i, ks = (int64_t)j * nx + i;
    const T ly = A.dy, lx = A.dx;
    // sum L ||D|| over East, North, West, South: (E + N) + (W + S)
    const T dE = ly * A.ex[WD_DA * A.xs + kw + 1], dN = lx * A.ey[WD_DA * A.ys + ks + nx];
    const T dW = ly * A.ex[WD_DB * A.xs + kw], dS = lx * A.ey[WD_DB * A.ys + ks];
    s = (dE + dN) + (dW + dS);
    // mass leaving the cell per unit time
    const T oE = fmax(ly * A.ex[WD_M * A.xs + kw + 1], T(0));
    const T oN = fmax(lx * A.ey[WD_M * A.ys + ks + nx], T(0));
    const T oW = fmax(-(ly * A.ex[WD_M * A.xs + kw]), T(0));
    const T oS = fmax(-(lx * A.ey[WD_M * A.ys + ks]), T(0));
    const T M = (oE + oN) + (oW + oS);
    const T h = A.w[0][(int64_t)(j + kPadY) * A.pitch + i + kPadX];
    A.tau[ks] = M > T(0) ? h * (T)A.area / M : T(INFINITY);
  }
  // block maximum (NaN wins), one atomic per block
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s = nanmax_wd(s, __shfl_xor_sync(kFullWd, s, o));
  const int t = threadIdx.y * blockDim.x + threadIdx.x;
  if ((t & 31) == 0) part[t >> 5] = s;
  __syncthreads();
  if (t < 32) {
    s = t < (int)(blockDim.x * blockDim.y / 32) ? part[t] : T(0);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = nanmax_wd(s, __shfl_xor_sync(kFullWd, s, o));
    if (t == 0 && (s > T(0) || s != s)) atomic_max_wd(A.tmax_out, s);
  }
  pdl_trigger();
}

template <typename T>
__global__ void __launch_bounds__(256) wd_update_kernel(const WdArgs<T> A) {
  __shared__ T k_sh;
  __shared__ int bad_dt;
  pdl_wait();
  const int t = threadIdx.y * blockDim.x + threadIdx.x;
  if (t == 0) {
    const T tm = *reinterpret_cast<const T*>(A.tmax_in);
    // dt = min_i 2 cfl |V_i| / sum L ||D|| (eq. (5)); no wet edge at all
    // (every cell dry) leaves no finite dt
    const double dt = A.two_cfl * A.area / (double)tm;
    bad_dt = !(tm > T(0)) || !isfinite(dt);
    k_sh = (T)dt;
    if (blockIdx.x == 0 && blockIdx.y == 0) {
      A.dt_hist[A.step % kHistCap] = dt;
      *A.t_dev += dt;
      if (sizeof(T) == 4) *reinterpret_cast<unsigned*>(A.tmax_clear) = 0u;
      else *reinterpret_cast<unsigned long long*>(A.tmax_clear) = 0ull;
      if (bad_dt) atomicOr(A.err, kErrNonfinite);
    }
  }
  __syncthreads();
  const T dt = k_sh;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int j = blockIdx.y * blockDim.y + threadIdx.y;
  const int nx = A.nx, ny = A.ny;
  unsigned bad = 0;
  if (i < nx && j < ny && !bad_dt) {
    const int64_t kw = (int64_t)j * (nx + 1) + i, ks = (int64_t)j * nx + i;
    const T ri = fmin(T(1), A.tau[ks] / dt);
    // limit of an edge: the ratio of the cell its mass flux leaves
    auto theta = [&](T m_out, bool nb_ok, int64_t nb) -> T {
      if (m_out > T(0)) return ri;
      if (m_out < T(0) && nb_ok) return fmin(T(1), A.tau[nb] / dt);
      return T(1);
    };
    const T* ex = A.ex;
    const T* ey = A.ey;
    const T ly = A.dy, lx = A.dx;
    // East (the cell is a), North (a), West (b), South (b)
    const T mE = ly * ex[WD_M * A.xs + kw + 1], mN = lx * ey[WD_M * A.ys + ks + nx];
    const T mW = ly * ex[WD_M * A.xs + kw], mS = lx * ey[WD_M * A.ys + ks];
    const T tE = theta(mE, i + 1 < nx, ks + 1), tN = theta(mN, j + 1 < ny, ks + nx);
    const T tW = theta(-mW, i > 0, ks - 1), tS = theta(-mS, j > 0, ks - nx);
    T fE[4], fN[4], fW[4], fS[4];
    fE[0] = tE * mE;
    fE[1] = tE * (ly * ex[WD_FA * A.xs + kw + 1]);
    fE[2] = tE * (ly * ex[WD_T * A.xs + kw + 1]);
    fE[3] = tE * (ly * ex[WD_C * A.xs + kw + 1]);
    fN[0] = tN * mN;
    fN[1] = tN * (lx * ey[WD_T * A.ys + ks + nx]);
    fN[2] = tN * (lx * ey[WD_FA * A.ys + ks + nx]);
    fN[3] = tN * (lx * ey[WD_C * A.ys + ks + nx]);
    fW[0] = -(tW * mW);
    fW[1] = -(tW * (ly * ex[WD_FB * A.xs + kw]));
    fW[2] = -(tW * (ly * ex[WD_T * A.xs + kw]));
    fW[3] = -(tW * (ly * ex[WD_C * A.xs + kw]));
    fS[0] = -(tS * mS);
    fS[1] = -(tS * (lx * ey[WD_T * A.ys + ks]));
    fS[2] = -(tS * (lx * ey[WD_FB * A.ys + ks]));
    fS[3] = -(tS * (lx * ey[WD_C * A.ys + ks]));
    const int64_t o = (int64_t)(j + kPadY) * A.pitch + i + kPadX;
    const T kk = dt / (T)A.area;
    T w[4];
#pragma unroll
    for (int f = 0; f < 4; ++f) w[f] = A.w[f][o] - kk * ((fE[f] + fN[f]) + (fW[f] + fS[f]));
    // clean-up: a depth below zero is rounding; a dry cell keeps no discharge
    if (w[0] < T(0)) w[0] = T(0);
    if (w[0] <= A.hdry) w[1] = w[2] = T(0);
    const T sum = (w[0] + w[1]) + (w[2] + w[3]);
    if (!isfinite(sum)) bad |= kErrNonfinite;
#pragma unroll
    for (int f = 0; f < 4; ++f) A.w[f][o] = w[f];
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
  for (int f = 0; f < 4; ++f) A.w[f] = (T*)a.w[f];
  A.H = (const T*)a.H;
  A.nx = a.nx;
  A.ny = a.ny;
  A.pitch = a.pitch;
  A.g = (T)a.g;
  A.hdry = (T)a.h_dry;
  A.dx = (T)a.dx;
  A.dy = (T)a.dy;
  A.ex = (T*)a.ex;
  A.ey = (T*)a.ey;
  A.xs = a.xs;
  A.ys = a.ys;
  A.tau = (T*)a.tau;
  A.two_cfl = a.two_cfl;
  A.area = a.dx * a.dy;
  A.tmax_out = a.tmax_slot;
  A.tmax_in = a.tmax_slot;
  A.tmax_clear = a.tmax_clear;
  A.dt_hist = a.dt_hist;
  A.t_dev = a.t_dev;
  A.step = a.step;
  A.err = a.err;
  A.efix = a.efix;
  const dim3 blk(32, 8);
  const dim3 ge((unsigned)((a.nx + 1 + 31) / 32), (unsigned)((a.ny + 1 + 7) / 8));
  const dim3 gc((unsigned)((a.nx + 31) / 32), (unsigned)((a.ny + 7) / 8));
  cudaError_t e;
  if (marks && (e = cudaEventRecord(marks[0], st)) != cudaSuccess) return e;
  e = a.efix ? launch_pdl(wd_edge_kernel<T, true>, ge, blk, 0, st, A)
             : launch_pdl(wd_edge_kernel<T, false>, ge, blk, 0, st, A);
  if (e != cudaSuccess) return e;
  if (marks && (e = cudaEventRecord(marks[1], st)) != cudaSuccess) return e;
  if ((e = launch_pdl(wd_cell_kernel<T>, gc, blk, 0, st, A)) != cudaSuccess) return e;
  if (marks && (e = cudaEventRecord(marks[2], st)) != cudaSuccess) return e;
  if ((e = launch_pdl(wd_update_kernel<T>, gc, blk, 0, st, A)) != cudaSuccess) return e;
  if (marks && (e = cudaEventRecord(marks[3], st)) != cudaSuccess) return e;
  return cudaSuccess;
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
template cudaError_t launch_wd_check<float>(const float* const*, int, int, int, unsigned*,
                                            cudaStream_t);
template cudaError_t launch_wd_check<double>(const double* const*, int, int, int, unsigned*,
                                             cudaStream_t);

}  // namespace swe
