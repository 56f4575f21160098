// swe_cart1.cu -- sm_103a kernels of the one-layer + pollutant Roe step on a
// Cartesian grid.
//
// Scheme: An MPI-CUDA implementation of an improved Roe method for two-layer
// shallow water systems, Sec. 2.2 -- update eq. (4), numerical flux steps 1-4
// (rotation, Roe matrix and P^-, passive tangential upwinding, back-rotation)
// and the CFL condition eq. (5) -- with one layer, plus the passive pollutant
// of A multi-GPU shallow-water simulation with transport of contaminants
// (abstract).  Every edge flux is computed once and handed to both of its
// cells, the idea of that paper's Figure 4, here at warp level.
//
// Fused step kernel (cart1_step_kernel).  One warp owns a vertical band of
// kOwn columns and a segment of rows, and marches up the rows.  Per row it
//   a1  streams the row of W^n = (h, qx, qy, hC) and H (plus two halo columns
//       on each side) into shared memory with cp.async.bulk, kStages rows
//       ahead, completion tracked by one mbarrier per stage;
//   a2  computes the x-edge fluxes of the row and the y-edge fluxes against
//       the row below, each edge once (neighbour lanes via shuffles);
//   a3  accumulates them per cell in registers;
//   a5  updates the row below (its residual is then complete) with the dt of
//       this step and writes it out (owned cells);
//   a4  computes the Roe wave speeds of the *new* state on the edges of its
//       owned cells and max-reduces sum |Gamma| ||D|| for the next step's dt.
// The next step's dt needs the new state one cell beyond the owned block, so
// each warp also updates a one-cell ring (halo of two cells of W^n).
//
// The flux is written in a form that is algebraically the paper's
// Phi^- = P^- d + F_1(W_eta,i):
//   mass, tangential momentum, pollutant: flux form, +f to the left/lower
//     cell and -f to the right/upper cell (exact antisymmetry);
//   normal momentum: fluctuation form, P^- d to the left cell and
//     d_1 - (P^- d)_1 = (P^+ d)_1 to the right one.  The sum over a closed
//     cell of |Gamma| F_eta(W_i) vanishes, so this equals eq. (4) up to
//     rounding, and water at rest over any bottom gives d = 0 exactly when the
//     surface is exactly flat.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <type_traits>

#include "swe_internal.h"

namespace swe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

template <typename T> struct Fm;
template <> struct Fm<float> {
  __device__ static __forceinline__ float rsq(float x) { return rsqrtf(x); }
  __device__ static __forceinline__ float rcp(float x) { return __frcp_rn(x); }
};
template <> struct Fm<double> {
  __device__ static __forceinline__ double rsq(double x) { return rsqrt(x); }
  __device__ static __forceinline__ double rcp(double x) { return __drcp_rn(x); }
};

// ---------------------------------------------------------------------------
// PTX helpers: shared-memory addresses, mbarrier, bulk async copy
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for a phase, giving up after `budget` SM clock cycles; false if the
// budget ran out.  The clock is read only once the first try has failed.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  long long budget) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long deadline = clock64() + budget;
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() > deadline) return false;
  }
  return true;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// About two seconds at the GB300's maximum SM clock.
constexpr long long kWaitCycles = 4000000000LL;

// ---------------------------------------------------------------------------
// vector moves of one lane's cells
template <typename T, int N>
__device__ __forceinline__ void lds_cells(const unsigned char* p, T (&a)[N]) {
  if constexpr (std::is_same<T, float>::value) {
    static_assert(N == 4, "four floats per lane");
    float4 v = *reinterpret_cast<const float4*>(p);
    a[0] = v.x; a[1] = v.y; a[2] = v.z; a[3] = v.w;
  } else {
    static_assert(N == 2, "two doubles per lane");
    double2 v = *reinterpret_cast<const double2*>(p);
    a[0] = v.x; a[1] = v.y;
  }
}
template <typename T, int N>
__device__ __forceinline__ void stg_cells(T* p, const T (&a)[N]) {
  if constexpr (std::is_same<T, float>::value) {
    *reinterpret_cast<float4*>(p) = make_float4(a[0], a[1], a[2], a[3]);
  } else {
    *reinterpret_cast<double2*>(p) = make_double2(a[0], a[1]);
  }
}

template <typename T>
__device__ __forceinline__ T shdn(T v) { return __shfl_down_sync(kFull, v, 1); }
template <typename T>
__device__ __forceinline__ T shup(T v) { return __shfl_up_sync(kFull, v, 1); }

// ---------------------------------------------------------------------------
// One side of an edge in the frame of the edge normal eta:
// depth h, s = sqrt(h), v = q_eta / sqrt(h), normal discharge q_eta,
// qu = q_eta^2 / h, tangential velocity ut, concentration C, bottom H.
template <typename T>
struct Side {
  T h, s, v, qn, qu, ut, C, H;
};
// Reflective wall: the ghost has the normal discharge negated.
template <typename T>
__device__ __forceinline__ Side<T> mirror(const Side<T>& a) {
  Side<T> m = a;
  m.v = -a.v;
  m.qn = -a.qn;
  return m;
}

// Contributions of one edge (left/lower cell a, right/upper cell b):
//   m   mass flux Phi^-[1] (to a: +m, to b: -m)
//   pm  (P^- d)[2]: normal-momentum fluctuation of a
//   dm  d[2] - (P^- d)[2]: normal-momentum fluctuation of b
//   t   tangential momentum flux m * u_t^* (to a: +t, to b: -t)
//   c   pollutant flux m * C^* (to a: +c, to b: -c)
template <typename T>
struct EdgeF {
  T m, pm, dm, t, c;
};

template <typename T>
__device__ __forceinline__ EdgeF<T> roe_edge(const Side<T>& a, const Side<T>& b, T gh) {
  // Roe averages: sqrt(h)-weighted normal velocity, arithmetic depth;
  // eigenvalues u -+ c of A_ij, c^2 = g hbar.
  const T un = (a.v + b.v) * Fm<T>::rcp(a.s + b.s);
  const T c2 = gh * (a.h + b.h);
  const T rc = Fm<T>::rsq(c2);
  const T c = c2 * rc;
  const T i2c = T(0.5) * rc;
  const T l1 = un - c;
  const T l2 = un + c;
  // d = F_1(W_j) - F_1(W_i) - S_ij (H_j - H_i); the pressure difference
  // g/2 (h_j^2 - h_i^2) is written g hbar (h_j - h_i).
  const T dH = b.H - a.H;
  const T d0 = b.qn - a.qn;
  const T d1 = (b.qu - a.qu) + c2 * ((b.h - a.h) - dH);
  // alpha = K^-1 d with K = [[1, 1], [l1, l2]]; P^- d = sum_k w_k alpha_k K_k,
  // w_k = (1 - sgn l_k) / 2 with sgn 0 = 0.
  const T a1 = (l2 * d0 - d1) * i2c;
  const T a2 = (d1 - l1 * d0) * i2c;
  const T w1 = (l1 < T(0)) ? T(1) : ((l1 > T(0)) ? T(0) : T(0.5));
  const T w2 = (l2 < T(0)) ? T(1) : ((l2 > T(0)) ? T(0) : T(0.5));
  const T b1 = w1 * a1;
  const T b2 = w2 * a2;
  EdgeF<T> f;
  f.m = (a.qn + b1) + b2;
  f.pm = b1 * l1 + b2 * l2;
  f.dm = d1 - f.pm;
  const bool up = f.m > T(0);
  f.t = f.m * (up ? a.ut : b.ut);
  f.c = f.m * (up ? a.C : b.C);
  return f;
}

// ||D_ij||_inf = |u_eta| + c of the Roe matrix of an edge (eq. (5)).
template <typename T>
__device__ __forceinline__ T roe_speed(T ha, T sa, T va, T hb, T sb, T vb, T gh) {
  const T un = (va + vb) * Fm<T>::rcp(sa + sb);
  const T c2 = gh * (ha + hb);
  return fabs(un) + c2 * Fm<T>::rsq(c2);
}

// max that keeps a NaN once it has appeared
template <typename T>
__device__ __forceinline__ T nanmax(T acc, T x) {
  return (x > acc || x != x) ? x : acc;
}

template <typename T>
__device__ __forceinline__ void atomic_max_pos(void* slot, T v);
template <>
__device__ __forceinline__ void atomic_max_pos<float>(void* slot, float v) {
  atomicMax(reinterpret_cast<unsigned int*>(slot), __float_as_uint(v));
}
template <>
__device__ __forceinline__ void atomic_max_pos<double>(void* slot, double v) {
  atomicMax(reinterpret_cast<unsigned long long*>(slot),
            static_cast<unsigned long long>(__double_as_longlong(v)));
}

template <typename T>
__device__ __forceinline__ void warp_max_publish(T v, void* slot) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = nanmax(v, __shfl_xor_sync(kFull, v, o));
  if ((threadIdx.x & 31) == 0 && v > T(0)) atomic_max_pos<T>(slot, v);
  else if ((threadIdx.x & 31) == 0 && v != v) atomic_max_pos<T>(slot, v);
}

// ---------------------------------------------------------------------------
// The fused step.  See the file comment.
template <typename T, bool ANISO, bool WALLX>
__device__ __forceinline__ void march(const StepArgs<T>& A, unsigned char* wsm, uint64_t* mbar,
                                      int band, int y0, int y1, T kdt) {
  constexpr int CPT = Cpt<T>::v;
  constexpr int WIN = 32 * CPT;
  constexpr int OWN = WIN - 4;
  constexpr uint32_t ROWB = WIN * sizeof(T);
  constexpr uint32_t STAGEB = 5 * ROWB;
  const int lane = threadIdx.x & 31;
  const int nx = A.nx, ny = A.ny;
  const T gh = A.ghalf;
  const int xb = band * OWN - 2 + lane * CPT;  // logical column of cell 0
  const int nrows = y1 - y0 + 4;               // rows y0-2 .. y1+1
  const int64_t col0 = (int64_t)band * OWN;    // physical column of the window

  unsigned own = 0;  // bit k: cell k of this lane is owned by this warp
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    const int x = xb + k;
    if (x >= band * OWN && x < band * OWN + OWN && x < nx) own |= 1u << k;
  }
  const bool own_all = own == (1u << CPT) - 1u;

  const T* src[5] = {A.win[0], A.win[1], A.win[2], A.win[3], A.H};
  auto issue = [&](int k) {
    const int st = k % kStages;
    const int r = y0 - 2 + k;
    const int64_t off = (int64_t)(r + kPadY) * A.pitch + col0;
    const uint32_t bar = smem_u32(&mbar[st]);
    mbar_expect_tx(bar, STAGEB);
#pragma unroll
    for (int f = 0; f < 5; ++f)
      bulk_g2s(smem_u32(wsm + st * STAGEB + f * ROWB), src[f] + off, ROWB, bar);
  };

  if (lane == 0) {
    for (int st = 0; st < kStages; ++st) mbar_init(smem_u32(&mbar[st]), 1);
    mbar_init_fence();
    for (int k = 0; k < kStages && k < nrows; ++k) issue(k);
  }
  __syncwarp();

  // W^n of the row below (r-1): what its y-edge with row r and its update need
  T ph[CPT], ps[CPT], pvy[CPT], pqy[CPT], pquy[CPT], pux[CPT], pC[CPT], pH[CPT];
  T pqx[CPT], phC[CPT];
  // residuals of rows r-1 (R1) and r (R0)
  T R1m[CPT], R1x[CPT], R1y[CPT], R1c[CPT];
  // new state of row r-2 and its partial wave-speed sum
  T n1h[CPT], n1s[CPT], n1vy[CPT], T1[CPT];
  T tmax = T(0);
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    ph[k] = ps[k] = pvy[k] = pqy[k] = pquy[k] = pux[k] = pC[k] = pH[k] = pqx[k] = phC[k] = T(0);
    R1m[k] = R1x[k] = R1y[k] = R1c[k] = T(0);
    n1h[k] = n1s[k] = n1vy[k] = T1[k] = T(0);
  }

  for (int k = 0; k < nrows; ++k) {
    const int r = y0 - 2 + k;
    const int st = k % kStages;
    // ---- a1: wait for the row, read it, release the stage --------------
    bool ok = mbar_wait_bounded(smem_u32(&mbar[st]), (uint32_t)((k / kStages) & 1), kWaitCycles);
    if (!__all_sync(kFull, ok)) {
      // give up: report, then wait (bounded) for the copies still in flight
      if (lane == 0) atomicOr(A.err, kErrTimeout);
      for (int q = k; q < nrows && q < k + kStages; ++q)
        (void)mbar_wait_bounded(smem_u32(&mbar[q % kStages]), (uint32_t)((q / kStages) & 1),
                                kWaitCycles);
      return;
    }
    T ch[CPT], cqx[CPT], cqy[CPT], chC[CPT], cH[CPT];
    const unsigned char* rowp = wsm + st * STAGEB + lane * CPT * sizeof(T);
    lds_cells<T, CPT>(rowp + 0 * ROWB, ch);
    lds_cells<T, CPT>(rowp + 1 * ROWB, cqx);
    lds_cells<T, CPT>(rowp + 2 * ROWB, cqy);
    lds_cells<T, CPT>(rowp + 3 * ROWB, chC);
    lds_cells<T, CPT>(rowp + 4 * ROWB, cH);
    __syncwarp();
    if (lane == 0 && k + kStages < nrows) {
      fence_proxy_async();
      issue(k + kStages);
    }
    // derived quantities of row r
    T cs[CPT], cvx[CPT], cvy[CPT], cux[CPT], cuy[CPT], cC[CPT], cqux[CPT], cquy[CPT];
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
      const T rs = Fm<T>::rsq(ch[i]);
      const T ih = rs * rs;
      cs[i] = ch[i] * rs;
      cvx[i] = cqx[i] * rs;
      cvy[i] = cqy[i] * rs;
      cux[i] = cqx[i] * ih;
      cuy[i] = cqy[i] * ih;
      cC[i] = chC[i] * ih;
      cqux[i] = cqx[i] * cux[i];
      cquy[i] = cqy[i] * cuy[i];
    }
    T R0m[CPT], R0x[CPT], R0y[CPT], R0c[CPT];
#pragma unroll
    for (int i = 0; i < CPT; ++i) R0m[i] = R0x[i] = R0y[i] = R0c[i] = T(0);

    // ---- a2/a3: x-edges of row r (needed for rows y0-1 .. y1) ------------
    if (r >= y0 - 1 && r <= y1) {
      Side<T> nb;
      nb.h = shdn(ch[0]); nb.s = shdn(cs[0]); nb.v = shdn(cvx[0]); nb.qn = shdn(cqx[0]);
      nb.qu = shdn(cqux[0]); nb.ut = shdn(cuy[0]); nb.C = shdn(cC[0]); nb.H = shdn(cH[0]);
      T cm = T(0), cx = T(0), cy = T(0), cc = T(0);
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        Side<T> a{ch[i], cs[i], cvx[i], cqx[i], cqux[i], cuy[i], cC[i], cH[i]};
        Side<T> b;
        if (i + 1 < CPT) b = Side<T>{ch[i + 1], cs[i + 1], cvx[i + 1], cqx[i + 1], cqux[i + 1],
                                     cuy[i + 1], cC[i + 1], cH[i + 1]};
        else b = nb;
        bool wall = false;
        if (WALLX) {
          const int xl = xb + i;
          if (xl == -1) { a = mirror(b); wall = true; }
          else if (xl == nx - 1) { b = mirror(a); wall = true; }
        }
        EdgeF<T> f = roe_edge(a, b, gh);
        if (WALLX && wall) { f.m = T(0); f.t = T(0); f.c = T(0); }
        R0m[i] += f.m; R0x[i] += f.pm; R0y[i] += f.t; R0c[i] += f.c;
        if (i + 1 < CPT) {
          R0m[i + 1] -= f.m; R0x[i + 1] += f.dm; R0y[i + 1] -= f.t; R0c[i + 1] -= f.c;
        } else {
          cm = -f.m; cx = f.dm; cy = -f.t; cc = -f.c;
        }
      }
      R0m[0] += shup(cm); R0x[0] += shup(cx); R0y[0] += shup(cy); R0c[0] += shup(cc);
    }

    // ---- a2/a3: y-edges between rows r-1 and r --------------------------
    if (r >= y0 - 1) {
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        Side<T> a{ph[i], ps[i], pvy[i], pqy[i], pquy[i], pux[i], pC[i], pH[i]};
        Side<T> b{ch[i], cs[i], cvy[i], cqy[i], cquy[i], cux[i], cC[i], cH[i]};
        if (r == 0) a = mirror(b);
        else if (r == ny) b = mirror(a);
        EdgeF<T> f = roe_edge(a, b, gh);
        if (r == 0 || r == ny) { f.m = T(0); f.t = T(0); f.c = T(0); }
        if (ANISO) { f.m *= A.rho; f.pm *= A.rho; f.dm *= A.rho; f.t *= A.rho; f.c *= A.rho; }
        R1m[i] += f.m; R1y[i] += f.pm; R1x[i] += f.t; R1c[i] += f.c;
        R0m[i] -= f.m; R0y[i] += f.dm; R0x[i] -= f.t; R0c[i] -= f.c;
      }
    }

    // ---- a5: update row r-1; a4: wave speeds of the new state ------------
    if (r >= y0) {
      const int rr = r - 1;
      T nh[CPT], nqx[CPT], nqy[CPT], nhC[CPT];
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        nh[i] = ph[i] - kdt * R1m[i];
        nqx[i] = pqx[i] - kdt * R1x[i];
        nqy[i] = pqy[i] - kdt * R1y[i];
        nhC[i] = phC[i] - kdt * R1c[i];
      }
      const bool owned_row = rr >= y0 && rr < y1;
      if (owned_row) {
        unsigned bad = 0;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
          if (own & (1u << i)) {
            const bool fin = isfinite(nh[i]) && isfinite(nqx[i]) && isfinite(nqy[i]) &&
                             isfinite(nhC[i]);
            if (!fin) bad |= kErrNonfinite;
            else if (!(nh[i] > T(0))) bad |= kErrDepth;
          }
        }
        if (bad) atomicOr(A.err, bad);
        const int64_t off = (int64_t)(rr + kPadY) * A.pitch + col0 + lane * CPT;
        if (own_all) {
          stg_cells<T, CPT>(A.wout[0] + off, nh);
          stg_cells<T, CPT>(A.wout[1] + off, nqx);
          stg_cells<T, CPT>(A.wout[2] + off, nqy);
          stg_cells<T, CPT>(A.wout[3] + off, nhC);
        } else if (own) {
#pragma unroll
          for (int i = 0; i < CPT; ++i) {
            if (own & (1u << i)) {
              A.wout[0][off + i] = nh[i];
              A.wout[1][off + i] = nqx[i];
              A.wout[2][off + i] = nqy[i];
              A.wout[3][off + i] = nhC[i];
            }
          }
        }
      }
      T ns[CPT], nvx[CPT], nvy[CPT], Tn[CPT];
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        const T rs = Fm<T>::rsq(nh[i]);
        ns[i] = nh[i] * rs;
        nvx[i] = nqx[i] * rs;
        nvy[i] = nqy[i] * rs;
        Tn[i] = T(0);
      }
      if (owned_row) {  // x-edges of the new row
        const T bh = shdn(nh[0]), bs = shdn(ns[0]), bv = shdn(nvx[0]);
        T carry = T(0);
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
          T ha = nh[i], sa = ns[i], va = nvx[i];
          T hb, sb, vb;
          if (i + 1 < CPT) { hb = nh[i + 1]; sb = ns[i + 1]; vb = nvx[i + 1]; }
          else { hb = bh; sb = bs; vb = bv; }
          if (WALLX) {
            const int xl = xb + i;
            if (xl == -1) { ha = hb; sa = sb; va = -vb; }
            else if (xl == nx - 1) { hb = ha; sb = sa; vb = -va; }
          }
          const T D = roe_speed(ha, sa, va, hb, sb, vb, gh);
          Tn[i] += D;
          if (i + 1 < CPT) Tn[i + 1] += D;
          else carry = D;
        }
        Tn[0] += shup(carry);
      }
      if (r >= y0 + 1) {  // y-edges between the new rows rr-1 and rr
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
          T ha = n1h[i], sa = n1s[i], va = n1vy[i];
          T hb = nh[i], sb = ns[i], vb = nvy[i];
          if (rr == 0) { ha = hb; sa = sb; va = -vb; }
          else if (rr == ny) { hb = ha; sb = sa; vb = -va; }
          T D = roe_speed(ha, sa, va, hb, sb, vb, gh);
          if (ANISO) D *= A.rho;
          T1[i] += D;
          Tn[i] += D;
        }
        if (rr - 1 >= y0 && rr - 1 < y1) {
#pragma unroll
          for (int i = 0; i < CPT; ++i)
            if (own & (1u << i)) tmax = nanmax(tmax, T1[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        n1h[i] = nh[i]; n1s[i] = ns[i]; n1vy[i] = nvy[i]; T1[i] = Tn[i];
      }
    }

    // ---- shift the W^n rows ----------------------------------------------
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
      ph[i] = ch[i]; ps[i] = cs[i]; pvy[i] = cvy[i]; pqy[i] = cqy[i]; pquy[i] = cquy[i];
      pux[i] = cux[i]; pC[i] = cC[i]; pH[i] = cH[i]; pqx[i] = cqx[i]; phC[i] = chC[i];
      R1m[i] = R0m[i]; R1x[i] = R0x[i]; R1y[i] = R0y[i]; R1c[i] = R0c[i];
    }
  }
  warp_max_publish<T>(tmax, A.tmax_out);
}

template <typename T, bool ANISO>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    cart1_step_kernel(const StepArgs<T> A) {
  constexpr int CPT = Cpt<T>::v;
  constexpr int WIN = 32 * CPT;
  constexpr int OWN = WIN - 4;
  constexpr uint32_t STAGEB = 5 * WIN * sizeof(T);
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5;

  // dt of this step from the previous step's wave-speed maximum (eq. (5)):
  // dt / dx = 2 cfl / max_i (sum_x D + (dx/dy) sum_y D)
  const T tm = *reinterpret_cast<const T*>(A.tmax_in);
  const double dtdx = A.two_cfl / (double)tm;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const double dt = dtdx * A.dx;
    A.dt_hist[A.step % kHistCap] = dt;
    *A.t_dev += dt;
    if (sizeof(T) == 4) *reinterpret_cast<unsigned*>(A.tmax_clear) = 0u;
    else *reinterpret_cast<unsigned long long*>(A.tmax_clear) = 0ull;
  }
  const T kdt = (T)dtdx;

  const int unit = blockIdx.x * kWarpsPerBlock + warp;
  if (unit >= A.nbands * A.nsegs) return;
  const int band = unit % A.nbands;
  const int seg = unit / A.nbands;
  const int y0 = (int)((int64_t)seg * A.ny / A.nsegs);
  const int y1 = (int)((int64_t)(seg + 1) * A.ny / A.nsegs);
  unsigned char* wsm = smem + warp * (kStages * STAGEB);
  uint64_t* mbar =
      reinterpret_cast<uint64_t*>(smem + kWarpsPerBlock * kStages * STAGEB) + warp * kStages;
  // bands whose window reaches a vertical wall take the checked path
  const bool wallx = band == 0 || band * OWN + WIN - 2 > A.nx - 1;
  if (wallx) march<T, ANISO, true>(A, wsm, mbar, band, y0, y1, kdt);
  else march<T, ANISO, false>(A, wsm, mbar, band, y0, y1, kdt);
}

// ---------------------------------------------------------------------------
// dt of a state loaded from the host: per cell sum_x D + rho sum_y D over its
// four edges (mirror ghosts at walls), max-reduced into a slot; also checks
// h > 0 and finiteness.  The per-cell quantities, the wave-speed formula and
// the order of the four additions are those of the fused step kernel, so a
// restart from a saved state reproduces an uninterrupted run bit for bit.
template <typename T>
__device__ __forceinline__ void speed_inputs(T h, T qx, T qy, T& s, T& vx, T& vy) {
  const T rs = Fm<T>::rsq(h);
  s = h * rs;
  vx = qx * rs;
  vy = qy * rs;
}

template <typename T>
__global__ void cart1_dt0_kernel(const T* __restrict__ h, const T* __restrict__ qx,
                                 const T* __restrict__ qy, const T* __restrict__ hC,
                                 int nx, int ny, int pitch, T gh, T rho, void* tmax_out,
                                 unsigned* err) {
  T tmax = T(0);
  unsigned bad = 0;
  const int64_t n = (int64_t)nx * ny;
  for (int64_t c = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; c < n;
       c += (int64_t)gridDim.x * blockDim.x) {
    const int i = (int)(c % nx), j = (int)(c / nx);
    const int64_t o = (int64_t)(j + kPadY) * pitch + i + kPadX;
    const T h0 = h[o], x0 = qx[o], y0 = qy[o], c0 = hC[o];
    if (!(isfinite(h0) && isfinite(x0) && isfinite(y0) && isfinite(c0))) bad |= kErrNonfinite;
    else if (!(h0 > T(0))) bad |= kErrDepth;
    T s0, vx0, vy0;
    speed_inputs(h0, x0, y0, s0, vx0, vy0);
    T hn, sn, vxn, vyn;
    // west and east edges
    T hw = h0, sw = s0, vw = -vx0;
    if (i > 0) { speed_inputs(h[o - 1], qx[o - 1], qy[o - 1], sn, vxn, vyn); hw = h[o - 1]; sw = sn; vw = vxn; }
    T he = h0, se = s0, ve = -vx0;
    if (i < nx - 1) { speed_inputs(h[o + 1], qx[o + 1], qy[o + 1], sn, vxn, vyn); he = h[o + 1]; se = sn; ve = vxn; }
    // south and north edges
    T hs = h0, ss = s0, vs = -vy0;
    if (j > 0) { hn = h[o - pitch]; speed_inputs(hn, qx[o - pitch], qy[o - pitch], sn, vxn, vyn); hs = hn; ss = sn; vs = vyn; }
    T hN = h0, sN = s0, vN = -vy0;
    if (j < ny - 1) { hn = h[o + pitch]; speed_inputs(hn, qx[o + pitch], qy[o + pitch], sn, vxn, vyn); hN = hn; sN = sn; vN = vyn; }
    T sum = roe_speed(hw, sw, vw, h0, s0, vx0, gh) + roe_speed(h0, s0, vx0, he, se, ve, gh);
    sum += roe_speed(hs, ss, vs, h0, s0, vy0, gh) * rho;
    sum += roe_speed(h0, s0, vy0, hN, sN, vN, gh) * rho;
    tmax = nanmax(tmax, sum);
  }
  if (bad) atomicOr(err, bad);
  warp_max_publish<T>(tmax, tmax_out);
}

template <typename T>
__global__ void fill_kernel(T* p, int64_t n, T v) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    p[i] = v;
}

}  // namespace

template <typename T>
size_t step_smem_bytes() {
  return (size_t)kWarpsPerBlock * kStages * 5 * band_window<T>() * sizeof(T) +
         (size_t)kWarpsPerBlock * kStages * sizeof(uint64_t);
}

template <typename T>
cudaError_t step_occupancy(int* blocks_per_sm, size_t* smem_bytes) {
  const size_t smem = step_smem_bytes<T>();
  *smem_bytes = smem;
  cudaError_t e;
  e = cudaFuncSetAttribute(cart1_step_kernel<T, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(cart1_step_kernel<T, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, cart1_step_kernel<T, false>,
                                                       kWarpsPerBlock * 32, smem);
}

template <typename T>
cudaError_t launch_step(const StepArgs<T>& a, int blocks, cudaStream_t st) {
  const size_t smem = step_smem_bytes<T>();
  if (a.rho == T(1))
    cart1_step_kernel<T, false><<<blocks, kWarpsPerBlock * 32, smem, st>>>(a);
  else
    cart1_step_kernel<T, true><<<blocks, kWarpsPerBlock * 32, smem, st>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_dt0(const T* const* w, const T* H, int nx, int ny, int pitch, T ghalf, T rho,
                       void* tmax_out, unsigned* err, cudaStream_t st) {
  (void)H;
  const int64_t n = (int64_t)nx * ny;
  int blocks = (int)((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  cart1_dt0_kernel<T><<<blocks, 256, 0, st>>>(w[0], w[1], w[2], w[3], nx, ny, pitch, ghalf, rho,
                                               tmax_out, err);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_fill(T* base, int64_t count, T value, cudaStream_t st) {
  int64_t blocks = (count + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  fill_kernel<T><<<(int)blocks, 256, 0, st>>>(base, count, value);
  return cudaGetLastError();
}

template cudaError_t step_occupancy<float>(int*, size_t*);
template cudaError_t step_occupancy<double>(int*, size_t*);
template cudaError_t launch_step<float>(const StepArgs<float>&, int, cudaStream_t);
template cudaError_t launch_step<double>(const StepArgs<double>&, int, cudaStream_t);
template cudaError_t launch_dt0<float>(const float* const*, const float*, int, int, int, float,
                                       float, void*, unsigned*, cudaStream_t);
template cudaError_t launch_dt0<double>(const double* const*, const double*, int, int, int, double,
                                        double, void*, unsigned*, cudaStream_t);
template cudaError_t launch_fill<float>(float*, int64_t, float, cudaStream_t);
template cudaError_t launch_fill<double>(double*, int64_t, double, cudaStream_t);

}  // namespace swe
