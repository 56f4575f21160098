// swe_roe2.cuh -- the IR-Roe numerical flux of one edge of the two-layer
// system, shared by the Cartesian and the triangle-mesh kernels.
//
// An MPI-CUDA implementation of an improved Roe method for two-layer shallow
// water systems, Sec. 2.2 (steps 1-4 with the 4x4 Roe matrix A_ij of the
// system rotated to the edge normal, eq. (2)-(3)).  The eigenvalues of A_ij
// are the roots of the quartic
//   p(l) = Q1(l) Q2(l) - r c1^2 c2^2,   Q_k(l) = (l - u_k)^2 - c_k^2.
// The outer two are found by Newton from bounds where p > 0 (p is convex and
// monotone there, so the iterates approach the root from outside without
// overshooting); the inner pair comes from deflating p by the outer pair and
// is polished by Newton on p.  Beyond max_k (u_k + c_k) both Q_k are positive
// and increasing, so p is increasing and convex there; for r < 1 it is
// positive wherever Q1 Q2 >= c1^2 c2^2, which holds at
//   l = max_k (u_k + sqrt(2) c_k)   (each Q_k >= c_k^2) and at
//   l = max_k u_k + sqrt(c1^2 + c2^2)   (Q1 >= c2^2, Q2 >= c1^2),
// so the smaller of the two is a safe start for the largest root (mirrored
// for the smallest).  The second is within a fraction of a percent of the
// root when the layers move together, the first when one layer is thin.  A complex inner pair (loss of hyperbolicity)
// is reported to the caller.  With right eigenvectors K_k = (1, l_k, m_k,
// l_k m_k), m_k = Q1(l_k)/c1^2, the left eigenvectors of A_ij are
// proportional to (l - 2u1, 1, c1^2 (l - 2u2)/Q2, c1^2/Q2), which gives the
// coordinates of d in the eigenvector basis without a linear solve:
//   alpha_k = [Q2(l_k)((l_k - 2u1) d1 + d2) + c1^2 ((l_k - 2u2) d3 + d4)] / p'(l_k).
// Then P^- d = sum_k w_k alpha_k K_k with w_k = (1 - sgn l_k)/2.
#pragma once

#include <cuda_runtime.h>
#include <math.h>

#include "swe_fastmath.cuh"

namespace swe {
namespace {

constexpr unsigned kFull2 = 0xffffffffu;

__device__ __forceinline__ float sqrt_approx(float x) {  // MUFU approximation
  float r;
  asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// sq: a square root that enters the flux; sqa: one that only seeds an
// iteration (Newton start, deflated inner roots), where a single-precision
// approximation is enough in either type.
template <typename T> struct M2;
template <> struct M2<float> {  // MUFU approximations (a few ulp)
  __device__ static __forceinline__ float rsq(float x) { return rsqrtf(x); }
  __device__ static __forceinline__ float rcp(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
  }
  __device__ static __forceinline__ float sq(float x) { return sqrt_approx(x); }
  __device__ static __forceinline__ float sqa(float x) { return sqrt_approx(x); }
  __device__ static __forceinline__ float big() { return 3.402823466e38f; }
};
template <> struct M2<double> {  // Newton-refined reciprocal (swe_fastmath.cuh)
  __device__ static __forceinline__ double rsq(double x) { return rsqrt(x); }
  __device__ static __forceinline__ double rcp(double x) { return rcp_nr(x); }
  __device__ static __forceinline__ double sq(double x) { return sqrt(x); }
  __device__ static __forceinline__ double sqa(double x) { return (double)sqrt_approx((float)x); }
  __device__ static __forceinline__ double big() { return 1.7976931348623157e308; }
};

// Newton iterations: the outer roots converge quadratically from the safe
// start; the inner ones start from the deflated estimate.  An edge's outer
// iteration stops once it has taken a step below tol * max(c1, c2) (after
// that the error is of the order of the type's rounding), after 2
// iterations on typical states.  `outer` bounds it: at
// small density ratios the two largest roots of p sit close together when
// u1 + c1 ~ u2 + c2, and Newton first converges linearly there; checked
// against extended-precision roots over depths 0.1-10 m, layer velocities up
// to 3 m/s and r from 0.001 to 0.98, 9 iterations reach fp32 rounding and 11
// fp64 rounding.  (At r = 0 with u1 + c1 = u2 + c2 the root is double and the
// eigenvector basis of A_ij degenerates.)  The inner pair, deflated from
// converged outer roots, reaches the type's rounding after one Newton step
// in fp64 (same check); `inner` keeps one more.
template <typename T> struct Iters;
template <> struct Iters<float> {
  static constexpr int outer = 10, inner = 2;
  static constexpr float tol = 2.44140625e-4f;  // 2^-12
};
template <> struct Iters<double> {
  static constexpr int outer = 12, inner = 2;
  static constexpr double tol = 1.4901161193847656e-8;  // 2^-26
};

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

// The four roots of p, in increasing order; false when the inner pair is
// complex (loss of hyperbolicity).  ADAPT: stop the outer Newton iteration
// early (warp vote) instead of running the fixed count.
template <typename T, bool ADAPT>
__device__ __forceinline__ bool quartic_roots(const Quartic<T>& q, T lam[4]) {
  const T c1 = M2<T>::sqa(q.c1s), c2 = M2<T>::sqa(q.c2s);
  const T sc = M2<T>::sqa(q.c1s + q.c2s);
  // outer roots: from below / above, where p > 0, p convex and monotone
  // (the approximate square roots widened by 2^-12, far more than their
  // error, so the starts stay outside)
  const T kr2 = T(1.4142135623730951 * (1.0 + 1.0 / 4096)), ks = T(1.0 + 1.0 / 4096);
  T l1 = fmax(fmin(q.u1 - kr2 * c1, q.u2 - kr2 * c2), fmin(q.u1, q.u2) - ks * sc);
  T l4 = fmin(fmax(q.u1 + kr2 * c1, q.u2 + kr2 * c2), fmax(q.u1, q.u2) + ks * sc);
  const T tol = Iters<T>::tol * fmax(c1, c2);
  const unsigned act = ADAPT ? __activemask() : 0u;
  // ADAPT: an edge keeps its roots once its own step fell below tol (so the
  // result depends on the edge's state alone, not on the warp it shares);
  // the loop ends when every edge of the warp has
  bool done = false;
#pragma unroll
  for (int it = 0; it < Iters<T>::outer; ++it) {
    const T s1 = q.p(l1) * M2<T>::rcp(q.dp(l1));
    const T s4 = q.p(l4) * M2<T>::rcp(q.dp(l4));
    if (!done) {
      l1 -= s1;
      l4 -= s4;
    }
    if (ADAPT) {
      done |= it >= 1 && (fabs(s1) <= tol) & (fabs(s4) <= tol);
      if (__all_sync(act, done)) break;
    }
  }
  // inner pair: p / ((l - l1)(l - l4)) = l^2 + bb l + cc
  const T p3 = T(-2) * (q.u1 + q.u2);
  const T p2 = (q.u1 * q.u1 - q.c1s) + (q.u2 * q.u2 - q.c2s) + T(4) * q.u1 * q.u2;
  const T ss = l1 + l4, pp = l1 * l4;
  const T bb = p3 + ss;
  const T cc = p2 + ss * bb - pp;
  const T disc = bb * bb - T(4) * cc;
  const bool hyper = disc > T(0);
  const T sd = M2<T>::sqa(hyper ? disc : T(0));
  T l2 = T(0.5) * (-bb - sd), l3 = T(0.5) * (-bb + sd);
  // each step at most half the pair's separation: near a double inner root
  // p' vanishes and an unclamped step can jump past the other root (or be
  // 0/0); the clamp also keeps a non-finite step finite
  const T lim = T(0.5) * sd;
#pragma unroll
  for (int it = 0; it < Iters<T>::inner; ++it) {
    l2 -= fmin(fmax(q.p(l2) * M2<T>::rcp(q.dp(l2)), -lim), lim);
    l3 -= fmin(fmax(q.p(l3) * M2<T>::rcp(q.dp(l3)), -lim), lim);
  }
  lam[0] = l1;
  lam[1] = l2;
  lam[2] = l3;
  lam[3] = l4;
  return hyper;
}

// The quartic of a side's own Jacobian A(W) (the same system with the side's
// normal velocities and c_k^2 = g h_k): its roots are the speeds
// lambda_k(W) of the entropy fix.
template <typename T>
__device__ __forceinline__ Quartic<T> side_quartic(const Side2<T>& a, T g, T r) {
  const T c1s = g * a.h[0], c2s = g * a.h[1];
  return Quartic<T>{a.qn[0] * (a.rs[0] * a.rs[0]), a.qn[1] * (a.rs[1] * a.rs[1]), c1s, c2s,
                    r * c1s * c2s};
}

// IR-Roe flux of one edge, two layers.  Writes the edge results; returns
// false when A_ij has a complex pair of eigenvalues.  ADAPT: early exit of
// the Newton iterations (quartic_roots).  EFIX: the Harten-Hyman entropy fix
// ([P1] Sec. 2.2, after eq. (5)) as numerical viscosity along each of the
// four waves: delta_k = max(0, l_k - l_k(W_i), l_k(W_j) - l_k) with l_k(W)
// the k-th root of the side's own quartic; where |l_k| < delta_k, Phi^-
// gains (|l_k| - |l_k|_d) beta_k K_k / 2, |l_k|_d = (l_k^2 + delta_k^2) /
// (2 delta_k), beta = K^-1 (W_j - W_i) from the left eigenvectors; side b's
// fluctuation P^+ d loses the same term.  A side whose own system is not
// hyperbolic is reported like A_ij.
template <typename T, bool ADAPT = false, bool EFIX = false>
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
  T lam[4];
  bool hyper = quartic_roots<T, ADAPT>(q, lam);
  const T l1 = lam[0], l4 = lam[3];
  // fluctuation d = F_1(W_j) - F_1(W_i) - B_ij (W_j - W_i) - S_ij (H_j - H_i)
  // (pressure differences written g hbar_k (h_k,j - h_k,i))
  const T dh1 = b.h[0] - a.h[0], dh2 = b.h[1] - a.h[1], dH = b.H - a.H;
  const T d1 = b.qn[0] - a.qn[0];
  const T d2 = (qu_b[0] - qu_a[0]) + cs[0] * ((dh1 + dh2) - dH);
  const T d3 = b.qn[1] - a.qn[1];
  const T d4 = (qu_b[1] - qu_a[1]) + cs[1] * ((dh2 + r * dh1) - dH);
  // entropy fix: each side's own speeds
  T la[4], lb[4];
  if (EFIX) {
    hyper &= quartic_roots<T, ADAPT>(side_quartic(a, g, r), la);
    hyper &= quartic_roots<T, ADAPT>(side_quartic(b, g, r), lb);
  }
  // P^- d = sum_k w_k alpha_k K_k (+ the fix's nu_k K_k).  Where every edge
  // of the warp has l1 < l2 < 0 < l3 < l4 (subcritical in both wave
  // families) waves 3 and 4 have w = 0 and add exact zeros: the loop stops
  // after wave 2, bit for bit the same sum.
  const T ic1s = M2<T>::rcp(cs[0]);
  T pd0 = T(0), pd1 = T(0), pd2 = T(0), pd3 = T(0);
  bool two_waves = false;
  if (ADAPT && !EFIX) {
    const bool sub = (l1 < T(0)) & (lam[1] < T(0)) & (lam[2] > T(0)) & (l4 > T(0));
    two_waves = __all_sync(__activemask(), sub);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (k == 2 && two_waves) break;
    const T l = lam[k];
    const T w = (l < T(0)) ? T(1) : ((l > T(0)) ? T(0) : T(0.5));
    const T Q1 = q.q1(l), Q2 = q.q2(l);
    const T num = Q2 * ((l - T(2) * un[0]) * d1 + d2) + cs[0] * ((l - T(2) * un[1]) * d3 + d4);
    const T rdp = M2<T>::rcp(q.dp(l));
    T alpha = w * num * rdp;
    if (EFIX) {
      const T del = fmax(T(0), fmax(l - la[k], lb[k] - l));
      const T al = fabs(l);
      if (al < del) {
        // beta_k: the left eigenvector applied to the state jump
        const T nb = Q2 * ((l - T(2) * un[0]) * dh1 + d1) + cs[0] * ((l - T(2) * un[1]) * dh2 + d3);
        alpha += T(0.5) * (al - (l * l + del * del) * M2<T>::rcp(del + del)) * (nb * rdp);
      }
    }
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

// ---- two edges at once on the packed FP32x2 pipe (fp32) ------------------------
// The same arithmetic as edge2<float> (swe_roe2.cuh), written with
// FADD2 / FMUL2 / FFMA2 so that one instruction serves both edges; the
// square roots and reciprocals stay per component.
__device__ __forceinline__ float2 f2(float x, float y) { return make_float2(x, y); }
__device__ __forceinline__ float2 s2(float v) { return make_float2(v, v); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 sub2(float2 a, float2 b) { return __ffma2_rn(b, s2(-1.f), a); }
__device__ __forceinline__ float2 rcp2(float2 a) { return f2(M2<float>::rcp(a.x), M2<float>::rcp(a.y)); }
__device__ __forceinline__ float2 rsq2(float2 a) { return f2(M2<float>::rsq(a.x), M2<float>::rsq(a.y)); }
__device__ __forceinline__ float2 sqrt2(float2 a) { return f2(sqrt_approx(a.x), sqrt_approx(a.y)); }
__device__ __forceinline__ float2 min2(float2 a, float2 b) { return f2(fminf(a.x, b.x), fminf(a.y, b.y)); }
__device__ __forceinline__ float2 max2(float2 a, float2 b) { return f2(fmaxf(a.x, b.x), fmaxf(a.y, b.y)); }
__device__ __forceinline__ float sgnw1(float l) { return l < 0.f ? 1.f : (l > 0.f ? 0.f : 0.5f); }

struct Side2P {
  float2 h[2], s[2], rs[2], qn[2], qt[2], H;
};

struct QuarticP {
  float2 u1, u2, c1s, c2s, rc;
  __device__ __forceinline__ void qq(float2 l, float2& d1, float2& d2, float2& q1,
                                     float2& q2) const {
    d1 = sub2(l, u1);
    d2 = sub2(l, u2);
    q1 = fma2(d1, d1, f2(-c1s.x, -c1s.y));
    q2 = fma2(d2, d2, f2(-c2s.x, -c2s.y));
  }
  // the Newton step p / p' at l (p = q1 q2 - rc, p' = 2 (d1 q2 + d2 q1))
  __device__ __forceinline__ float2 step(float2 l) const {
    float2 d1, d2, q1, q2;
    qq(l, d1, d2, q1, q2);
    const float2 p = fma2(q1, q2, f2(-rc.x, -rc.y));
    const float2 dp = mul2(s2(2.f), fma2(d1, q2, mul2(d2, q1)));
    return mul2(p, rcp2(dp));
  }
};

// The four roots of two quartics at once, in increasing order: edge2's
// quartic_roots (the same safe starts, per-edge early exit of the outer
// Newton iteration, clamped inner steps) on the FP32x2 pipe.  Returns a mask:
// bit 0 (bit 1) when the first (second) quartic's inner pair is real.
__device__ __forceinline__ unsigned roots2p(const QuarticP& q, float2 lam[4]) {
  const float2 c1 = sqrt2(q.c1s), c2 = sqrt2(q.c2s);
  const float2 sc = sqrt2(add2(q.c1s, q.c2s));
  const float kr2 = 1.4142135623730951f * (1.f + 1.f / 4096), ks = 1.f + 1.f / 4096;
  // outer roots: the safe starts of edge2 (swe_roe2.cuh)
  float2 l1 = max2(min2(fma2(s2(-kr2), c1, q.u1), fma2(s2(-kr2), c2, q.u2)),
                   fma2(s2(-ks), sc, min2(q.u1, q.u2)));
  float2 l4 = min2(max2(fma2(s2(kr2), c1, q.u1), fma2(s2(kr2), c2, q.u2)),
                   fma2(s2(ks), sc, max2(q.u1, q.u2)));
  const float2 tol = mul2(s2(Iters<float>::tol), max2(c1, c2));
  const unsigned act = __activemask();
  bool done0 = false, done1 = false;  // per edge, as in edge2
#pragma unroll
  for (int it = 0; it < Iters<float>::outer; ++it) {
    const float2 t1 = q.step(l1), t4 = q.step(l4);
    const float2 n1 = sub2(l1, t1), n4 = sub2(l4, t4);
    l1 = f2(done0 ? l1.x : n1.x, done1 ? l1.y : n1.y);
    l4 = f2(done0 ? l4.x : n4.x, done1 ? l4.y : n4.y);
    done0 |= it >= 1 && (fabsf(t1.x) <= tol.x) & (fabsf(t4.x) <= tol.x);
    done1 |= it >= 1 && (fabsf(t1.y) <= tol.y) & (fabsf(t4.y) <= tol.y);
    if (__all_sync(act, done0 & done1)) break;
  }
  // inner pair: p / ((l - l1)(l - l4)) = l^2 + bb l + cc
  const float2 p3 = mul2(s2(-2.f), add2(q.u1, q.u2));
  const float2 p2 = add2(add2(fma2(q.u1, q.u1, f2(-q.c1s.x, -q.c1s.y)),
                              fma2(q.u2, q.u2, f2(-q.c2s.x, -q.c2s.y))),
                         mul2(mul2(s2(4.f), q.u1), q.u2));
  const float2 ss = add2(l1, l4), pp = mul2(l1, l4);
  const float2 bb = add2(p3, ss);
  const float2 cc = sub2(fma2(ss, bb, p2), pp);
  const float2 disc = fma2(bb, bb, mul2(s2(-4.f), cc));
  const unsigned hyper = (disc.x > 0.f ? 1u : 0u) | (disc.y > 0.f ? 2u : 0u);
  const float2 sd = sqrt2(max2(disc, s2(0.f)));
  float2 l2 = mul2(s2(0.5f), sub2(f2(-bb.x, -bb.y), sd));
  float2 l3 = mul2(s2(0.5f), sub2(sd, bb));
  const float2 lim = mul2(s2(0.5f), sd);  // steps clamped as in edge2
  const float2 nlim = f2(-lim.x, -lim.y);
#pragma unroll
  for (int it = 0; it < Iters<float>::inner; ++it) {
    l2 = sub2(l2, min2(max2(q.step(l2), nlim), lim));
    l3 = sub2(l3, min2(max2(q.step(l3), nlim), lim));
  }
  lam[0] = l1;
  lam[1] = l2;
  lam[2] = l3;
  lam[3] = l4;
  return hyper;
}

// A side's own quartic (side_quartic) for two edges at once.
__device__ __forceinline__ QuarticP side_quartic2p(const Side2P& a, float g, float r) {
  const float2 c1s = mul2(s2(g), a.h[0]), c2s = mul2(s2(g), a.h[1]);
  return QuarticP{mul2(a.qn[0], mul2(a.rs[0], a.rs[0])), mul2(a.qn[1], mul2(a.rs[1], a.rs[1])),
                  c1s, c2s, mul2(mul2(s2(r), c1s), c2s)};
}

// Flux of two edges at once; walls per component.  Returns a mask: bit 0
// (bit 1) set when the first (second) edge's A_ij (and, with EFIX, each
// side's own matrix) has real eigenvalues.  EFIX: the Harten-Hyman fix of
// edge2, per component; the sides' own speeds are solved here unless the
// caller passes them (la_in, lb_in: roots of side_quartic2p of a and b,
// with side_hyper the mask of those quartics whose inner pair is real).
template <bool EFIX = false>
__device__ __forceinline__ unsigned edge2p(const Side2P& a, const Side2P& b, float g, float gh,
                                           float r, bool w0, bool w1, float2* out,
                                           const float2* la_in = nullptr,
                                           const float2* lb_in = nullptr,
                                           unsigned side_hyper = 3u) {
  float2 un[2], cs[2], qu_a[2], qu_b[2], ut_a[2], ut_b[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float2 va = mul2(a.qn[k], a.rs[k]), vb = mul2(b.qn[k], b.rs[k]);
    un[k] = mul2(add2(va, vb), rcp2(add2(a.s[k], b.s[k])));
    cs[k] = mul2(s2(gh), add2(a.h[k], b.h[k]));
    const float2 iha = mul2(a.rs[k], a.rs[k]), ihb = mul2(b.rs[k], b.rs[k]);
    qu_a[k] = mul2(mul2(a.qn[k], a.qn[k]), iha);
    qu_b[k] = mul2(mul2(b.qn[k], b.qn[k]), ihb);
    ut_a[k] = mul2(a.qt[k], iha);
    ut_b[k] = mul2(b.qt[k], ihb);
  }
  const QuarticP q{un[0], un[1], cs[0], cs[1], mul2(mul2(s2(r), cs[0]), cs[1])};
  float2 lam[4];
  unsigned hyper = roots2p(q, lam);
  const float2 l1 = lam[0], l2 = lam[1], l3 = lam[2], l4 = lam[3];
  // fluctuation d (pressure differences written g hbar_k dh_k)
  const float2 dh1 = sub2(b.h[0], a.h[0]), dh2 = sub2(b.h[1], a.h[1]), dH = sub2(b.H, a.H);
  const float2 d1 = sub2(b.qn[0], a.qn[0]);
  const float2 d2 = fma2(cs[0], sub2(add2(dh1, dh2), dH), sub2(qu_b[0], qu_a[0]));
  const float2 d3 = sub2(b.qn[1], a.qn[1]);
  const float2 d4 = fma2(cs[1], sub2(fma2(s2(r), dh1, dh2), dH), sub2(qu_b[1], qu_a[1]));
  // P^- d = sum_k w_k alpha_k K_k (+ the fix's term); without the fix waves
  // 3 and 4 add exact zeros when every edge of the warp is subcritical in
  // both families (as in edge2)
  // entropy fix: each side's own speeds
  float2 la[4], lb[4];
  if (EFIX) {
    if (la_in) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        la[k] = la_in[k];
        lb[k] = lb_in[k];
      }
      hyper &= side_hyper;
    } else {
      hyper &= roots2p(side_quartic2p(a, g, r), la);
      hyper &= roots2p(side_quartic2p(b, g, r), lb);
    }
  }
  const float2 ic1s = rcp2(cs[0]);
  const float2 tu1 = mul2(s2(2.f), un[0]), tu2 = mul2(s2(2.f), un[1]);
  float2 pd0 = s2(0.f), pd1 = s2(0.f), pd2 = s2(0.f), pd3 = s2(0.f);
  bool two_waves = false;
  if (!EFIX) {
    const bool sub = (l1.x < 0.f) & (l1.y < 0.f) & (l2.x < 0.f) & (l2.y < 0.f) & (l3.x > 0.f) &
                     (l3.y > 0.f) & (l4.x > 0.f) & (l4.y > 0.f);
    two_waves = __all_sync(__activemask(), sub);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (k == 2 && two_waves) break;
    const float2 l = lam[k];
    const float2 w = f2(sgnw1(l.x), sgnw1(l.y));
    float2 e1, e2, Q1, Q2;
    q.qq(l, e1, e2, Q1, Q2);
    const float2 dp = mul2(s2(2.f), fma2(e1, Q2, mul2(e2, Q1)));
    const float2 num = fma2(Q2, fma2(sub2(l, tu1), d1, d2),
                            mul2(cs[0], fma2(sub2(l, tu2), d3, d4)));
    const float2 rdp = rcp2(dp);
    float2 alpha = mul2(mul2(w, num), rdp);
    if (EFIX) {
      const float2 del = max2(s2(0.f), max2(sub2(l, la[k]), sub2(lb[k], l)));
      if ((fabsf(l.x) < del.x) | (fabsf(l.y) < del.y)) {
        // beta_k: the left eigenvector applied to the state jump
        const float2 nb = fma2(Q2, fma2(sub2(l, tu1), dh1, d1),
                               mul2(cs[0], fma2(sub2(l, tu2), dh2, d3)));
        const float2 nbr = mul2(nb, rdp);
        if (fabsf(l.x) < del.x)
          alpha.x += 0.5f * (fabsf(l.x) - (l.x * l.x + del.x * del.x) *
                                              M2<float>::rcp(del.x + del.x)) * nbr.x;
        if (fabsf(l.y) < del.y)
          alpha.y += 0.5f * (fabsf(l.y) - (l.y * l.y + del.y * del.y) *
                                              M2<float>::rcp(del.y + del.y)) * nbr.y;
      }
    }
    const float2 mu = mul2(Q1, ic1s);
    pd0 = add2(pd0, alpha);
    pd1 = fma2(alpha, l, pd1);
    pd2 = fma2(alpha, mu, pd2);
    pd3 = fma2(mul2(alpha, l), mu, pd3);
  }
  float2 m1 = add2(a.qn[0], pd0);
  float2 m2 = add2(a.qn[1], pd2);
  if (w0) { m1.x = 0.f; m2.x = 0.f; }  // a reflective wall passes no mass
  if (w1) { m1.y = 0.f; m2.y = 0.f; }
  out[E_M1] = m1;
  out[E_PM1] = pd1;
  out[E_PS1] = sub2(d2, pd1);
  out[E_T1] = mul2(m1, f2(m1.x > 0.f ? ut_a[0].x : ut_b[0].x, m1.y > 0.f ? ut_a[0].y : ut_b[0].y));
  out[E_M2] = m2;
  out[E_PM2] = pd3;
  out[E_PS2] = sub2(d4, pd3);
  out[E_T2] = mul2(m2, f2(m2.x > 0.f ? ut_a[1].x : ut_b[1].x, m2.y > 0.f ? ut_a[1].y : ut_b[1].y));
  out[E_D] = max2(f2(fabsf(l1.x), fabsf(l1.y)), f2(fabsf(l4.x), fabsf(l4.y)));
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

// Block-wide maximum (NaN wins) published with one atomic per block: the
// atomics of a grid all go to one address, so one per warp would serialise
// tens of thousands of them in a single L2 slice.  Every thread of the block
// must call it (it synchronises the block).
template <typename T, int NWARPS>
__device__ __forceinline__ void block_max_publish(T m, void* slot) {
  __shared__ T part[NWARPS];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = nanmax2(m, __shfl_xor_sync(kFull2, m, o));
  const int t = threadIdx.x + blockDim.x * threadIdx.y;
  if ((t & 31) == 0) part[t >> 5] = m;
  __syncthreads();
  if (t < 32) {
    m = t < NWARPS ? part[t] : T(0);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = nanmax2(m, __shfl_xor_sync(kFull2, m, o));
    if (t == 0 && (m > T(0) || m != m)) atomic_max_pos2<T>(slot, m);
  }
}

}  // namespace
}  // namespace swe
