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

#include "swe_fastmath.cuh"
#include "swe_internal.h"

namespace swe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

template <typename T> struct Fm;
// fp32: the MUFU approximations (relative error of a few ulp; the fp32
// tolerances of the method are orders of magnitude looser).
template <> struct Fm<float> {
  __device__ static __forceinline__ float rsq(float x) {
    float r;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
  }
  __device__ static __forceinline__ float rcp(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
  }
};
// fp64: the reciprocal from a hardware seed refined by Newton-Raphson
// (swe_fastmath.cuh, about one ulp; cheaper than the correctly rounded
// routine on GB300's narrow FP64 pipe); CUDA's rsqrt, which measured cheaper
// than a refined seed here.
template <> struct Fm<double> {
  __device__ static __forceinline__ double rsq(double x) { return rsqrt(x); }
  __device__ static __forceinline__ double rcp(double x) { return rcp_nr(x); }
};

template <typename T> struct Lim;
template <> struct Lim<float> {
  __device__ static __forceinline__ float max() { return 3.402823466e38f; }
};
template <> struct Lim<double> {
  __device__ static __forceinline__ double max() { return 1.7976931348623157e308; }
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
// Predicated forms: every lane executes the instruction, `on` selects the
// lanes that act, so the stage refill has no divergent branch.
__device__ __forceinline__ void mbar_expect_tx_if(bool on, uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %0, 0;\n\t"
      "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%1], %2;\n\t}" ::"r"((uint32_t)on),
      "r"(bar), "r"(bytes)
      : "memory");
}
__device__ __forceinline__ void bulk_g2s_if(bool on, uint32_t dst, const void* src,
                                            uint32_t bytes, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %0, 0;\n\t"
      "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%1], [%2], %3, [%4];"
      "\n\t}" ::"r"((uint32_t)on),
      "r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// About two seconds at the GB300's maximum SM clock.
constexpr long long kWaitCycles = 4000000000LL;

// ---------------------------------------------------------------------------
// Scalar operations with explicit rounding (never contracted into FMAs), so
// the host-loaded dt pass reproduces the fused kernel's wave speeds exactly.
__device__ __forceinline__ float sadd(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ double sadd(double a, double b) { return __dadd_rn(a, b); }
__device__ __forceinline__ float smul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ double smul(double a, double b) { return __dmul_rn(a, b); }
__device__ __forceinline__ float sfma(float a, float b, float c) { return __fmaf_rn(a, b, c); }
__device__ __forceinline__ double sfma(double a, double b, double c) { return __fma_rn(a, b, c); }

// ---------------------------------------------------------------------------
// Pairs: the two cells of a lane.  fp32 pairs use the packed FP32x2 pipe
// (one FADD2/FMUL2/FFMA2 per operation on both cells); fp64 pairs are two
// scalar operations.
template <typename T> struct PairOf;
template <> struct PairOf<float> { using type = float2; };
template <> struct PairOf<double> { using type = double2; };
template <typename T> using Pr = typename PairOf<T>::type;

__device__ __forceinline__ float2 pr(float a, float b) { return make_float2(a, b); }
__device__ __forceinline__ double2 pr(double a, double b) { return make_double2(a, b); }
template <typename T> __device__ __forceinline__ Pr<T> psplat(T v) { return pr(v, v); }

__device__ __forceinline__ float2 padd(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 pmul(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 pfma(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 psub(float2 a, float2 b) {
  return __ffma2_rn(b, make_float2(-1.f, -1.f), a);
}
__device__ __forceinline__ double2 padd(double2 a, double2 b) {
  return pr(__dadd_rn(a.x, b.x), __dadd_rn(a.y, b.y));
}
__device__ __forceinline__ double2 pmul(double2 a, double2 b) {
  return pr(__dmul_rn(a.x, b.x), __dmul_rn(a.y, b.y));
}
__device__ __forceinline__ double2 pfma(double2 a, double2 b, double2 c) {
  return pr(__fma_rn(a.x, b.x, c.x), __fma_rn(a.y, b.y, c.y));
}
__device__ __forceinline__ double2 psub(double2 a, double2 b) {
  return pr(__dsub_rn(a.x, b.x), __dsub_rn(a.y, b.y));
}
template <typename P> __device__ __forceinline__ P pneg(P a) { return pr(-a.x, -a.y); }
template <typename P> __device__ __forceinline__ P pabs(P a) { return pr(fabs(a.x), fabs(a.y)); }
template <typename T> __device__ __forceinline__ Pr<T> prsq(Pr<T> a) {
  return pr(Fm<T>::rsq(a.x), Fm<T>::rsq(a.y));
}
template <typename T> __device__ __forceinline__ Pr<T> prcp(Pr<T> a) {
  return pr(Fm<T>::rcp(a.x), Fm<T>::rcp(a.y));
}
template <typename P> __device__ __forceinline__ P pshup(P a) {  // (left lane's y, own x)
  return pr(__shfl_up_sync(kFull, a.y, 1), a.x);
}

template <typename T>
__device__ __forceinline__ T shdn(T v) { return __shfl_down_sync(kFull, v, 1); }

template <typename T>
__device__ __forceinline__ Pr<T> lds_pair(const unsigned char* p) {
  return *reinterpret_cast<const Pr<T>*>(p);
}

// ---------------------------------------------------------------------------
// Two edges (one per component) seen in the frame of their normals eta:
// depth h, s = sqrt(h), v = q_eta / sqrt(h), normal discharge q_eta,
// qu = q_eta^2 / h, tangential velocity ut, concentration C, bottom H, and
// (read by the entropy fix only) the normal velocity u = q_eta / h.
template <typename T>
struct SideP {
  Pr<T> h, s, v, qn, qu, ut, C, H, u;
};
// Reflective wall: the ghost is the cell with its normal discharge negated.
template <typename T>
__device__ __forceinline__ SideP<T> mirror(const SideP<T>& a) {
  SideP<T> m = a;
  m.v = pneg(a.v);
  m.qn = pneg(a.qn);
  m.u = pneg(a.u);
  return m;
}
// the same, for one component only (k = 0: .x, 1: .y)
template <typename T>
__device__ __forceinline__ void mirror_into(SideP<T>& dst, const SideP<T>& src, int k) {
  if (k == 0) {
    dst.h.x = src.h.x; dst.s.x = src.s.x; dst.v.x = -src.v.x; dst.qn.x = -src.qn.x;
    dst.qu.x = src.qu.x; dst.ut.x = src.ut.x; dst.C.x = src.C.x; dst.H.x = src.H.x;
    dst.u.x = -src.u.x;
  } else {
    dst.h.y = src.h.y; dst.s.y = src.s.y; dst.v.y = -src.v.y; dst.qn.y = -src.qn.y;
    dst.qu.y = src.qu.y; dst.ut.y = src.ut.y; dst.C.y = src.C.y; dst.H.y = src.H.y;
    dst.u.y = -src.u.y;
  }
}

// Contributions of a pair of edges (left/lower cell a, right/upper cell b):
//   m     mass flux Phi^-[1]                 a: +m   b: -m
//   pm    (P^- d)[2], normal momentum        a: +pm
//   dsum  (P^- d)[2] - d[2]                  b: -dsum  (= (P^+ d)[2])
//   t     tangential momentum m u_t^*        a: +t   b: -t
//   c     pollutant m C^*                    a: +c   b: -c
template <typename T>
struct FluxP {
  Pr<T> m, pm, dsum, t, c;
};

template <typename T>
__device__ __forceinline__ T sgn_weight(T l) {  // (1 - sgn l) / 2, sgn 0 = 0
  return (l < T(0)) ? T(1) : ((l > T(0)) ? T(0) : T(0.5));
}

// First half of the flux of a pair of edges: Roe averages (sqrt(h)-weighted
// normal velocity, arithmetic depth), eigenvalues l1,2 = u -+ c of A_ij with
// c^2 = g hbar, the fluctuation d = F_1(W_j) - F_1(W_i) - S_ij (H_j - H_i)
// (the pressure difference g/2 (h_j^2 - h_i^2) written g hbar (h_j - h_i);
// d1n = -d[2]) and alpha_1 of alpha = K^-1 d, K = [[1, 1], [l1, l2]].
template <typename T>
struct RoeHead {
  Pr<T> l1, l2, d0, d1n, a1, i2c;
};
// Entropy fix (EFIX; [P1] Sec. 2.2 remarks that a Harten-Hyman fix can be
// adapted, without a formula): Harten's regularised |l|_d = |l| when
// |l| >= delta, (l^2 + delta^2) / (2 delta) otherwise, with delta_k =
// max(0, l_k - l_k(W_a), l_k(W_b) - l_k), l_k(W) = u_eta -/+ sqrt(g h) of the
// state itself; it adds 1/2 (|l_k| - |l_k|_d) beta_k K_k to Phi^-, with
// beta = K^-1 (W_b - W_a).  Zero wherever |l_k| >= delta_k.  The deltas
// are formed twice: once for the warp vote (is the fix inactive on every
// edge?) and again in the general tail, so that none stays live in between.
template <typename T>
__device__ __forceinline__ T hh_delta(T l, T lL, T lR) {
  return fmax(T(0), fmax(l - lL, lR - l));
}
template <typename T>
struct HHDelta {
  Pr<T> d1, d2;
};
template <typename T>
__device__ __forceinline__ HHDelta<T> hh_deltas(const RoeHead<T>& e, const SideP<T>& a,
                                                const SideP<T>& b, Pr<T> gh) {
  using P = Pr<T>;
  // sqrt(g h) of each side: sqrt(2 gh) s
  const P sg = psplat<T>(sqrt(T(2) * gh.x));
  const P ca = pmul(sg, a.s), cb = pmul(sg, b.s);
  const P lL1 = psub(a.u, ca), lR1 = psub(b.u, cb);
  const P lL2 = padd(a.u, ca), lR2 = padd(b.u, cb);
  return {pr(hh_delta(e.l1.x, lL1.x, lR1.x), hh_delta(e.l1.y, lL1.y, lR1.y)),
          pr(hh_delta(e.l2.x, lL2.x, lR2.x), hh_delta(e.l2.y, lL2.y, lR2.y))};
}
template <typename T>
__device__ __forceinline__ bool no_fix(const RoeHead<T>& e, const SideP<T>& a, const SideP<T>& b,
                                       Pr<T> gh) {
  const HHDelta<T> d = hh_deltas(e, a, b, gh);
  return (fabs(e.l1.x) >= d.d1.x) & (fabs(e.l1.y) >= d.d1.y) & (fabs(e.l2.x) >= d.d2.x) &
         (fabs(e.l2.y) >= d.d2.y);
}
// 1/2 (|l| - |l|_d) for one edge (0 where the fix is not active)
template <typename T>
__device__ __forceinline__ T hh_visc(T l, T del) {
  const T a = fabs(l);
  if (!(a < del)) return T(0);
  return T(0.5) * (a - (l * l + del * del) * Fm<T>::rcp(del + del));
}
template <typename T>
__device__ __forceinline__ RoeHead<T> roe_head(const SideP<T>& a, const SideP<T>& b, Pr<T> gh) {
  using P = Pr<T>;
  RoeHead<T> e;
  const P un = pmul(padd(a.v, b.v), prcp<T>(padd(a.s, b.s)));
  const P c2 = pmul(gh, padd(a.h, b.h));
  const P rc = prsq<T>(c2);
  const P c = pmul(c2, rc);
  e.i2c = pmul(psplat<T>(T(0.5)), rc);
  e.l1 = psub(un, c);
  e.l2 = padd(un, c);
  e.d0 = psub(b.qn, a.qn);
  e.d1n = pfma(c2, psub(psub(b.H, a.H), psub(b.h, a.h)), psub(a.qu, b.qu));
  e.a1 = pmul(pfma(e.l2, e.d0, e.d1n), e.i2c);
  return e;
}
template <typename T>
__device__ __forceinline__ bool subcritical(const RoeHead<T>& e) {
  return (e.l1.x < T(0)) & (e.l1.y < T(0)) & (e.l2.x > T(0)) & (e.l2.y > T(0));
}
// Second half: P^- d = sum_k w_k alpha_k K_k with w_k = (1 - sgn l_k) / 2.
// `fast` (every edge of the warp has l1 < 0 < l2) takes w = (1, 0), which is
// the general branch bit for bit.  Then the passive upwinding of the
// tangential velocity and of the concentration.
template <typename T, bool EFIX = false>
__device__ __forceinline__ FluxP<T> roe_tail(const RoeHead<T>& e, const SideP<T>& a,
                                             const SideP<T>& b, Pr<T> gh, bool fast) {
  using P = Pr<T>;
  FluxP<T> f;
  if (fast) {
    f.m = padd(a.qn, e.a1);
    f.pm = pmul(e.a1, e.l1);
  } else {
    const P a2n = pmul(pfma(e.l1, e.d0, e.d1n), e.i2c);  // -alpha_2
    const P b1 = pmul(pr(sgn_weight(e.l1.x), sgn_weight(e.l1.y)), e.a1);
    const P b2n = pmul(pr(sgn_weight(e.l2.x), sgn_weight(e.l2.y)), a2n);
    f.m = psub(padd(a.qn, b1), b2n);
    f.pm = psub(pmul(b1, e.l1), pmul(b2n, e.l2));
    if (EFIX) {
      // beta = K^-1 (W_b - W_a): (l2 dh - dq, dq - l1 dh) / (2c)
      const P dh = psub(b.h, a.h);
      const P be1 = pmul(psub(pmul(e.l2, dh), e.d0), e.i2c);
      const P be2 = pmul(psub(e.d0, pmul(e.l1, dh)), e.i2c);
      const HHDelta<T> d = hh_deltas(e, a, b, gh);
      const P n1 = pmul(pr(hh_visc(e.l1.x, d.d1.x), hh_visc(e.l1.y, d.d1.y)), be1);
      const P n2 = pmul(pr(hh_visc(e.l2.x, d.d2.x), hh_visc(e.l2.y, d.d2.y)), be2);
      f.m = padd(f.m, padd(n1, n2));
      f.pm = padd(f.pm, padd(pmul(n1, e.l1), pmul(n2, e.l2)));
    }
  }
  f.dsum = padd(e.d1n, f.pm);
  const P ut = pr(f.m.x > T(0) ? a.ut.x : b.ut.x, f.m.y > T(0) ? a.ut.y : b.ut.y);
  const P cc = pr(f.m.x > T(0) ? a.C.x : b.C.x, f.m.y > T(0) ? a.C.y : b.C.y);
  f.t = pmul(f.m, ut);
  f.c = pmul(f.m, cc);
  return f;
}
template <typename T, bool EFIX = false>
__device__ __forceinline__ FluxP<T> roe_pair(const SideP<T>& a, const SideP<T>& b, Pr<T> gh) {
  const RoeHead<T> e = roe_head<T>(a, b, gh);
  bool ok = subcritical(e);
  if (EFIX) ok &= no_fix(e, a, b, gh);
  return roe_tail<T, EFIX>(e, a, b, gh, __all_sync(kFull, ok));
}
// Two pairs at once (the x-edges and the y-edges of a row), one vote.
template <typename T, bool EFIX = false>
__device__ __forceinline__ void roe_two(const SideP<T>& ax, const SideP<T>& bx,
                                        const SideP<T>& ay, const SideP<T>& by, Pr<T> gh,
                                        FluxP<T>& fx, FluxP<T>& fy) {
  const RoeHead<T> ex = roe_head<T>(ax, bx, gh);
  const RoeHead<T> ey = roe_head<T>(ay, by, gh);
  bool ok = subcritical(ex) & subcritical(ey);
  if (EFIX) ok &= no_fix(ex, ax, bx, gh) & no_fix(ey, ay, by, gh);
  const bool fast = __all_sync(kFull, ok);
  fx = roe_tail<T, EFIX>(ex, ax, bx, gh, fast);
  fy = roe_tail<T, EFIX>(ey, ay, by, gh, fast);
}

// ||D_ij||_inf = |u_eta| + c of the Roe matrix of an edge (eq. (5)); the
// pair form and the scalar form round identically.
template <typename T>
__device__ __forceinline__ Pr<T> speed_pair(Pr<T> ha, Pr<T> sa, Pr<T> va, Pr<T> hb, Pr<T> sb,
                                            Pr<T> vb, Pr<T> gh) {
  const Pr<T> un = pmul(padd(va, vb), prcp<T>(padd(sa, sb)));
  const Pr<T> c2 = pmul(gh, padd(ha, hb));
  return pfma(c2, prsq<T>(c2), pabs(un));
}
template <typename T>
__device__ __forceinline__ T speed_scalar(T ha, T sa, T va, T hb, T sb, T vb, T gh) {
  const T un = smul(sadd(va, vb), Fm<T>::rcp(sadd(sa, sb)));
  const T c2 = smul(gh, sadd(ha, hb));
  return sfma(c2, Fm<T>::rsq(c2), fabs(un));
}

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
  if ((threadIdx.x & 31) == 0 && (v > T(0) || v != v)) atomic_max_pos<T>(slot, v);
}

// ---------------------------------------------------------------------------
// The fused step.  See the file comment.

// W^n of one row of a lane (two cells) with the quantities its edges need,
// and the residual the row accumulates (R.x, R.y: x and y momentum).
template <typename T>
struct RowN {
  Pr<T> h, qx, qy, hC, H;
  Pr<T> s, vx, vy, ux, uy, C, qux, quy;
  Pr<T> Rm, Rx, Ry, Rc;
};
// W^{n+1} of one row: what the y-edge wave speeds need, and the row's
// partial wave-speed sum.
template <typename T>
struct RowW {
  Pr<T> h, s, vy, D;
};

template <typename T>
__device__ __forceinline__ SideP<T> side_x(const RowN<T>& q) {
  return SideP<T>{q.h, q.s, q.vx, q.qx, q.qux, q.uy, q.C, q.H, q.ux};
}
template <typename T>
__device__ __forceinline__ SideP<T> side_y(const RowN<T>& q) {
  return SideP<T>{q.h, q.s, q.vy, q.qy, q.quy, q.ux, q.C, q.H, q.uy};
}

// Everything a warp keeps while it marches.
template <typename T>
struct Ctx {
  const StepArgs<T>* A;
  unsigned char* wsm;
  uint64_t* mbar;
  int y0, y1, nrows, xb, lane;
  int64_t col0;
  unsigned own;  // bit 0 / 1: cell 0 / 1 of this lane is owned by this warp
  bool partial;  // some lane of the warp owns one cell only (warp-uniform)
  Pr<T> gh, rho, nkdt;
  T tmax;
  unsigned flags;
  Pr<T> nanacc;      // sum of (field sum * 0) over owned cells: 0 or NaN
  T hmin;            // minimum new depth over owned cells
  T* out[4];         // output fields at this lane's first cell of row 0
  const T* src;      // lanes 0-9: field (lane % 5) of row (lane / 5) of stage 0
  uint32_t dst_off;  // its offset inside a stage
  int64_t src_step;  // elements between the same lane's rows of two stages
};

template <typename T> constexpr uint32_t row_bytes() { return 64 * sizeof(T); }
template <typename T> constexpr uint32_t stage_bytes() { return 2 * 5 * row_bytes<T>(); }

// Stage s holds rows 2s and 2s+1 of the march: 5 fields each, copied by up
// to ten lanes at once, completion on the stage's mbarrier.
template <typename T>
__device__ __forceinline__ void issue_stage(const Ctx<T>& c, int s) {
  const int nr = min(2, c.nrows - 2 * s);
  const int st = s % kStages;
  const uint32_t bar = smem_u32(&c.mbar[st]);
  mbar_expect_tx_if(c.lane == 0, bar, (uint32_t)nr * 5u * row_bytes<T>());
  __syncwarp();
  bulk_g2s_if(c.lane < 5 * nr, smem_u32(c.wsm + st * stage_bytes<T>() + c.dst_off),
              c.src + s * c.src_step, row_bytes<T>(), bar);
}

// x-edges of a row: edge pair (cell0|cell1, cell1|next lane's cell0).
// Vertical walls (WALLX bands) take the mirror state; w0/w1 mark them.
template <typename T, bool WALLX, bool EFIX>
__device__ __forceinline__ void xsides(const Ctx<T>& c, const RowN<T>& q, SideP<T>& a,
                                       SideP<T>& b, bool& w0, bool& w1) {
  a = side_x(q);
  b.u = EFIX ? pr(q.ux.y, shdn(q.ux.x)) : a.u;
  b.h = pr(q.h.y, shdn(q.h.x));
  b.s = pr(q.s.y, shdn(q.s.x));
  b.v = pr(q.vx.y, shdn(q.vx.x));
  b.qn = pr(q.qx.y, shdn(q.qx.x));
  b.qu = pr(q.qux.y, shdn(q.qux.x));
  b.ut = pr(q.uy.y, shdn(q.uy.x));
  b.C = pr(q.C.y, shdn(q.C.x));
  b.H = pr(q.H.y, shdn(q.H.x));
  w0 = false;
  w1 = false;
  if (WALLX) {
    const int nx = c.A->nx;
    if (c.xb == -1) { mirror_into(a, b, 0); w0 = true; }
    else if (c.xb == nx - 1) { mirror_into(b, a, 0); w0 = true; }
    if (c.xb + 1 == -1) { mirror_into(a, b, 1); w1 = true; }
    else if (c.xb + 1 == nx - 1) { mirror_into(b, a, 1); w1 = true; }
  }
}
template <typename T, bool WALLX, bool INIT>
__device__ __forceinline__ void xaccum(RowN<T>& q, FluxP<T> f, bool w0, bool w1) {
  if (WALLX) {
    if (w0) { f.m.x = T(0); f.t.x = T(0); f.c.x = T(0); }
    if (w1) { f.m.y = T(0); f.t.y = T(0); f.c.y = T(0); }
  }
  if (INIT) {
    q.Rm = f.m; q.Rx = f.pm; q.Ry = f.t; q.Rc = f.c;
  } else {
    q.Rm = padd(q.Rm, f.m); q.Rx = padd(q.Rx, f.pm); q.Ry = padd(q.Ry, f.t); q.Rc = padd(q.Rc, f.c);
  }
  q.Rm = psub(q.Rm, pshup(f.m));
  q.Rx = psub(q.Rx, pshup(f.dsum));
  q.Ry = psub(q.Ry, pshup(f.t));
  q.Rc = psub(q.Rc, pshup(f.c));
}
template <typename T, bool WALLX, bool INIT, bool EFIX>
__device__ __forceinline__ void row_xedges(const Ctx<T>& c, RowN<T>& q) {
  SideP<T> a, b;
  bool w0, w1;
  xsides<T, WALLX, EFIX>(c, q, a, b, w0, w1);
  xaccum<T, WALLX, INIT>(q, roe_pair<T, EFIX>(a, b, c.gh), w0, w1);
}

// y-edges between row p (below) and row q (above).  WALL: a horizontal
// wall, `lower_is_ghost` telling which side is the real cell.
template <typename T, bool ANISO, bool WALL>
__device__ __forceinline__ void yaccum(const Ctx<T>& c, RowN<T>& p, RowN<T>& q, FluxP<T> f) {
  if (WALL) {
    f.m = psplat<T>(T(0)); f.t = f.m; f.c = f.m;
  }
  if (ANISO) {
    f.m = pmul(f.m, c.rho); f.pm = pmul(f.pm, c.rho); f.dsum = pmul(f.dsum, c.rho);
    f.t = pmul(f.t, c.rho); f.c = pmul(f.c, c.rho);
  }
  p.Rm = padd(p.Rm, f.m); p.Ry = padd(p.Ry, f.pm); p.Rx = padd(p.Rx, f.t); p.Rc = padd(p.Rc, f.c);
  q.Rm = psub(q.Rm, f.m); q.Ry = psub(q.Ry, f.dsum); q.Rx = psub(q.Rx, f.t); q.Rc = psub(q.Rc, f.c);
}
template <typename T, bool ANISO, bool WALL, bool EFIX>
__device__ __forceinline__ void row_yedges(const Ctx<T>& c, RowN<T>& p, RowN<T>& q,
                                           bool lower_is_ghost) {
  SideP<T> a = side_y(p);
  SideP<T> b = side_y(q);
  if (WALL) {
    if (lower_is_ghost) a = mirror(b);
    else b = mirror(a);
  }
  yaccum<T, ANISO, WALL>(c, p, q, roe_pair<T, EFIX>(a, b, c.gh));
}
// Steady rows: the x-edges of row q and the y-edges between p and q
// evaluated together (one vote, two independent streams of work).
template <typename T, bool ANISO, bool WALLX, bool EFIX>
__device__ __forceinline__ void row_xyedges(const Ctx<T>& c, RowN<T>& p, RowN<T>& q) {
  SideP<T> ax, bx;
  bool w0, w1;
  xsides<T, WALLX, EFIX>(c, q, ax, bx, w0, w1);
  const SideP<T> ay = side_y(p);
  const SideP<T> by = side_y(q);
  FluxP<T> fx, fy;
  roe_two<T, EFIX>(ax, bx, ay, by, c.gh, fx, fy);
  xaccum<T, WALLX, true>(q, fx, w0, w1);
  yaccum<T, ANISO, false>(c, p, q, fy);
}

// wave speeds of the y-edges between new rows u (below) and w (above)
template <typename T, bool ANISO, bool WALL>
__device__ __forceinline__ void row_yspeeds(const Ctx<T>& c, RowW<T>& u, RowW<T>& w,
                                            bool lower_is_ghost) {
  Pr<T> ha = u.h, sa = u.s, va = u.vy, hb = w.h, sb = w.s, vb = w.vy;
  if (WALL) {
    if (lower_is_ghost) { ha = hb; sa = sb; va = pneg(vb); }
    else { hb = ha; sb = sa; vb = pneg(va); }
  }
  Pr<T> D = speed_pair<T>(ha, sa, va, hb, sb, vb, c.gh);
  if (ANISO) D = pmul(D, c.rho);
  u.D = padd(u.D, D);
  w.D = padd(w.D, D);
}

// One row of the march.  Row r = y0 - 2 + k arrives into q (p holds row
// r-1); row r-1 is updated into w (u holds the new row r-2).
//   STEADY  r in [y0+2, y1-1]: every part runs, no horizontal wall
//   PAR     0 / 1: k even / odd; 2: decided at run time
// Returns false if a bounded wait gave up.
template <typename T, bool ANISO, bool WALLX, bool EFIX, bool STEADY, int PAR>
__device__ __forceinline__ bool march_row(Ctx<T>& c, int k, RowN<T>& p, RowN<T>& q, RowW<T>& u,
                                          RowW<T>& w) {
  const StepArgs<T>& A = *c.A;
  const int r = c.y0 - 2 + k;
  const bool odd = PAR == 2 ? (k & 1) != 0 : PAR == 1;
  const int s = k >> 1;
  const int st = s % kStages;
  // ---- a1: the row from shared memory ------------------------------------
  if (!odd) {
    const bool ok = mbar_wait_bounded(smem_u32(&c.mbar[st]), (uint32_t)((s / kStages) & 1),
                                      kWaitCycles);
    if (!__all_sync(kFull, ok)) return false;
  }
  {
    const unsigned char* rowp = c.wsm + st * stage_bytes<T>() + (odd ? 5 : 0) * row_bytes<T>() +
                                c.lane * 2 * sizeof(T);
    q.h = lds_pair<T>(rowp + 0 * row_bytes<T>());
    q.qx = lds_pair<T>(rowp + 1 * row_bytes<T>());
    q.qy = lds_pair<T>(rowp + 2 * row_bytes<T>());
    q.hC = lds_pair<T>(rowp + 3 * row_bytes<T>());
    q.H = lds_pair<T>(rowp + 4 * row_bytes<T>());
  }
  if (odd || (!STEADY && k == c.nrows - 1)) {  // stage consumed: refill it
    fence_proxy_async();
    __syncwarp();
    if (2 * (s + kStages) < c.nrows) issue_stage(c, s + kStages);
  }
  {
    const Pr<T> rs = prsq<T>(q.h);
    const Pr<T> ih = pmul(rs, rs);
    q.s = pmul(q.h, rs);
    q.vx = pmul(q.qx, rs);
    q.vy = pmul(q.qy, rs);
    q.ux = pmul(q.qx, ih);
    q.uy = pmul(q.qy, ih);
    q.C = pmul(q.hC, ih);
    q.qux = pmul(q.qx, q.ux);
    q.quy = pmul(q.qy, q.uy);
  }
  // ---- a2/a3: x-edges of row r, y-edges between rows r-1 and r ----------
  if (STEADY) {
    row_xyedges<T, ANISO, WALLX, EFIX>(c, p, q);
  } else {
    if (r >= c.y0 - 1 && r <= c.y1) {
      row_xedges<T, WALLX, true, EFIX>(c, q);
    } else {
      q.Rm = q.Rx = q.Ry = q.Rc = psplat<T>(T(0));
    }
    if (r >= c.y0 - 1) {
      if (r == 0 || r == A.ny) row_yedges<T, ANISO, true, EFIX>(c, p, q, r == 0);
      else row_yedges<T, ANISO, false, EFIX>(c, p, q, false);
    }
    if (r < c.y0) return true;
  }
  // ---- a5: update row r-1 (its residual is complete) ---------------------
  const int rr = r - 1;
  w.h = pfma(c.nkdt, p.Rm, p.h);
  const Pr<T> nqx = pfma(c.nkdt, p.Rx, p.qx);
  const Pr<T> nqy = pfma(c.nkdt, p.Ry, p.qy);
  const Pr<T> nhC = pfma(c.nkdt, p.Rc, p.hC);
  const bool owned_row = STEADY || (rr >= c.y0 && rr < c.y1);
  if (owned_row) {
    // checks: sum * 0 is 0 for finite values and NaN otherwise, so one
    // accumulator flags any non-finite field; a running minimum of h flags a
    // depth <= 0.  Both are read once, at the end of the march.
    const Pr<T> sum = padd(padd(w.h, nqx), padd(nqy, nhC));
    const int64_t off = (int64_t)rr * A.pitch;
    if (c.own == 3u) {
      c.nanacc = pfma(sum, psplat<T>(T(0)), c.nanacc);
      c.hmin = fmin(c.hmin, fmin(w.h.x, w.h.y));
      *reinterpret_cast<Pr<T>*>(c.out[0] + off) = w.h;
      *reinterpret_cast<Pr<T>*>(c.out[1] + off) = nqx;
      *reinterpret_cast<Pr<T>*>(c.out[2] + off) = nqy;
      *reinterpret_cast<Pr<T>*>(c.out[3] + off) = nhC;
    }
    if (c.partial && (c.own == 1u || c.own == 2u)) {  // the grid's last column alone
      const int i = c.own == 1u ? 0 : 1;
      const T hs = i ? w.h.y : w.h.x;
      c.nanacc.x = sfma(i ? sum.y : sum.x, T(0), c.nanacc.x);
      c.hmin = fmin(c.hmin, hs);
      c.out[0][off + i] = hs;
      c.out[1][off + i] = i ? nqx.y : nqx.x;
      c.out[2][off + i] = i ? nqy.y : nqy.x;
      c.out[3][off + i] = i ? nhC.y : nhC.x;
    }
  }
  // ---- a4: wave speeds of the new state ----------------------------------
  Pr<T> nvx;
  {
    const Pr<T> rs = prsq<T>(w.h);
    w.s = pmul(w.h, rs);
    nvx = pmul(nqx, rs);
    w.vy = pmul(nqy, rs);
  }
  if (owned_row) {  // x-edges of the new row
    Pr<T> ha = w.h, sa = w.s, va = nvx;
    Pr<T> hb = pr(w.h.y, shdn(w.h.x)), sb = pr(w.s.y, shdn(w.s.x)), vb = pr(nvx.y, shdn(nvx.x));
    if (WALLX) {
      const int nx = A.nx;
      if (c.xb == -1) { ha.x = hb.x; sa.x = sb.x; va.x = -vb.x; }
      else if (c.xb == nx - 1) { hb.x = ha.x; sb.x = sa.x; vb.x = -va.x; }
      if (c.xb + 1 == -1) { ha.y = hb.y; sa.y = sb.y; va.y = -vb.y; }
      else if (c.xb + 1 == nx - 1) { hb.y = ha.y; sb.y = sa.y; vb.y = -va.y; }
    }
    const Pr<T> D = speed_pair<T>(ha, sa, va, hb, sb, vb, c.gh);
    w.D = padd(D, pshup(D));
  } else {
    w.D = psplat<T>(T(0));
  }
  if (STEADY || r >= c.y0 + 1) {  // y-edges between the new rows rr-1 and rr
    if (!STEADY && (rr == 0 || rr == A.ny)) row_yspeeds<T, ANISO, true>(c, u, w, rr == 0);
    else row_yspeeds<T, ANISO, false>(c, u, w, false);
    if (STEADY || (rr - 1 >= c.y0 && rr - 1 < c.y1)) {
      if (c.own & 1u) c.tmax = fmax(c.tmax, u.D.x);
      if (c.own & 2u) c.tmax = fmax(c.tmax, u.D.y);
    }
  }
  return true;
}

template <typename T, bool ANISO, bool WALLX, bool EFIX>
__device__ __forceinline__ bool general_row(Ctx<T>& c, int k, RowN<T>& P, RowN<T>& Q,
                                            RowW<T>& U, RowW<T>& V) {
  if (k & 1) return march_row<T, ANISO, WALLX, EFIX, false, 2>(c, k, Q, P, V, U);
  return march_row<T, ANISO, WALLX, EFIX, false, 2>(c, k, P, Q, U, V);
}

template <typename T, bool ANISO, bool WALLX, bool EFIX>
__device__ __forceinline__ void march(const StepArgs<T>& A, unsigned char* wsm, uint64_t* mbar,
                                      int band, int y0, int y1, T kdt) {
  constexpr int OWN = 64 - 4;
  Ctx<T> c;
  c.A = &A;
  c.wsm = wsm;
  c.mbar = mbar;
  c.y0 = y0;
  c.y1 = y1;
  c.nrows = y1 - y0 + 4;  // rows y0-2 .. y1+1
  c.lane = threadIdx.x & 31;
  c.xb = band * OWN - 2 + 2 * c.lane;  // logical column of the lane's cell 0
  c.col0 = (int64_t)band * OWN;        // physical column of the window
  c.own = 0;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int x = c.xb + i;
    if (x >= band * OWN && x < band * OWN + OWN && x < A.nx) c.own |= 1u << i;
  }
  c.partial = __any_sync(kFull, c.own == 1u || c.own == 2u);
  c.gh = psplat<T>(A.ghalf);
  c.rho = psplat<T>(A.rho);
  c.nkdt = psplat<T>(-kdt);
  c.tmax = T(0);
  c.flags = 0;
  c.nanacc = psplat<T>(T(0));
  c.hmin = Lim<T>::max();
  for (int f = 0; f < 4; ++f) c.out[f] = A.wout[f] + (int64_t)kPadY * A.pitch + c.col0 + 2 * c.lane;
  {
    const int j = c.lane >= 5 ? 1 : 0;
    const int f = c.lane < 10 ? c.lane - 5 * j : 0;
    const T* base = f == 0 ? A.win[0] : f == 1 ? A.win[1] : f == 2 ? A.win[2]
                  : f == 3 ? A.win[3] : A.H;
    c.src = base + (int64_t)(y0 - 2 + j + kPadY) * A.pitch + c.col0;
    c.dst_off = (uint32_t)(j * 5 + f) * row_bytes<T>();
    c.src_step = 2 * (int64_t)A.pitch;
  }

  const int nstages = (c.nrows + 1) / 2;
  if (c.lane == 0) {
    for (int st = 0; st < kStages; ++st) mbar_init(smem_u32(&mbar[st]), 1);
    mbar_init_fence();
  }
  __syncwarp();
  for (int s = 0; s < kStages && s < nstages; ++s) issue_stage(c, s);

  RowN<T> P, Q;
  RowW<T> U, V;
  P.h = P.qx = P.qy = P.hC = P.H = P.s = P.vx = P.vy = psplat<T>(T(0));
  P.ux = P.uy = P.C = P.qux = P.quy = P.Rm = P.Rx = P.Ry = P.Rc = psplat<T>(T(0));
  U.h = U.s = U.vy = U.D = psplat<T>(T(0));
  // rows alternate between the two register sets: no copies between rows
  int k = 0;
  bool ok = true;
  for (; k < 4 && k < c.nrows; ++k) {
    ok = general_row<T, ANISO, WALLX, EFIX>(c, k, P, Q, U, V);
    if (!ok) break;
  }
  for (; ok && k + 1 <= c.nrows - 3; k += 2) {
    ok = march_row<T, ANISO, WALLX, EFIX, true, 0>(c, k, P, Q, U, V);
    if (!ok) break;
    ok = march_row<T, ANISO, WALLX, EFIX, true, 1>(c, k + 1, Q, P, V, U);
    if (!ok) { ++k; break; }
  }
  for (; ok && k < c.nrows; ++k) {
    ok = general_row<T, ANISO, WALLX, EFIX>(c, k, P, Q, U, V);
    if (!ok) break;
  }
  if (!ok) {
    // give up: report, then wait (bounded) for the copies still in flight
    if (c.lane == 0) atomicOr(A.err, kErrTimeout);
    const int s0 = k >> 1;
    for (int s = s0; s < nstages && s < s0 + kStages; ++s)
      (void)mbar_wait_bounded(smem_u32(&mbar[s % kStages]), (uint32_t)((s / kStages) & 1),
                              kWaitCycles);
    return;
  }
  if (!(c.nanacc.x == T(0) && c.nanacc.y == T(0))) c.flags |= kErrNonfinite;
  if (!(c.hmin > T(0))) c.flags |= kErrDepth;
  if (c.flags) atomicOr(A.err, c.flags);
  warp_max_publish<T>(c.tmax, A.tmax_out);
}

// Minimum resident blocks per SM the register allocation is held to: the
// fp32 step fits 128 registers without spilling (16 warps per SM); the fp64
// step needs about 230 and is bound by the FP64 pipe, not by latency.
#ifndef SWE_STEP_MIN_BLOCKS_F32
#define SWE_STEP_MIN_BLOCKS_F32 4
#endif
template <typename T, bool EFIX> struct MinBlocks { static constexpr int v = 1; };
template <> struct MinBlocks<float, false> { static constexpr int v = SWE_STEP_MIN_BLOCKS_F32; };
#ifndef SWE_STEP_MIN_BLOCKS_F32_EFIX
#define SWE_STEP_MIN_BLOCKS_F32_EFIX 3
#endif
template <> struct MinBlocks<float, true> { static constexpr int v = SWE_STEP_MIN_BLOCKS_F32_EFIX; };

template <typename T, bool ANISO, bool EFIX>
__global__ void __launch_bounds__(kWarpsPerBlock * 32, MinBlocks<T, EFIX>::v)
    cart1_step_kernel(const StepArgs<T> A) {
  constexpr int OWN = 64 - 4;
  extern __shared__ __align__(128) unsigned char smem[];
  const int warp = threadIdx.x >> 5;

  // dt of this step from the previous step's wave-speed maximum (eq. (5)):
  // dt / dx = 2 cfl / max_i (sum_x D + (dx/dy) sum_y D), computed once per
  // block (a double division in every thread would hold up the start of the
  // march on GB300's FP64 pipe)
  __shared__ T kdt_sh;
  pdl_wait();
  if (threadIdx.x == 0) {
    const T tm = *reinterpret_cast<const T*>(A.tmax_in);
    const double dtdx = A.two_cfl / (double)tm;
    kdt_sh = (T)dtdx;
    if (blockIdx.x == 0) {
      const double dt = dtdx * A.dx;
      A.dt_hist[A.step % kHistCap] = dt;
      *A.t_dev += dt;
      if (sizeof(T) == 4) *reinterpret_cast<unsigned*>(A.tmax_clear) = 0u;
      else *reinterpret_cast<unsigned long long*>(A.tmax_clear) = 0ull;
    }
  }
  __syncthreads();
  const T kdt = kdt_sh;

  // warp -> (band, segment): segment-major, band fastest (warps resident
  // together stream the same rows of adjacent bands), then the extra, shorter
  // segments of the two wall bands
  const int nb = A.nbands, S = A.nsegs, Sw = A.nsegs_wall;
  const int nw = nb > 1 ? 2 : 1;
  const int unit = blockIdx.x * kWarpsPerBlock + warp;
  if (unit >= nb * S + nw * (Sw - S)) {
    pdl_trigger();
    return;
  }
  int band, seg;
  if (unit < nb * S) {
    band = unit % nb;
    seg = unit / nb;
  } else {
    const int i = unit - nb * S;
    band = i / (Sw - S) == 0 ? 0 : nb - 1;
    seg = S + i % (Sw - S);
  }
  const int ns = (band == 0 || band == nb - 1) ? Sw : S;
  const int y0 = (int)((int64_t)seg * A.ny / ns);
  const int y1 = (int)((int64_t)(seg + 1) * A.ny / ns);
  unsigned char* wsm = smem + warp * (kStages * stage_bytes<T>());
  uint64_t* mbar =
      reinterpret_cast<uint64_t*>(smem + kWarpsPerBlock * kStages * stage_bytes<T>()) +
      warp * kStages;
  // bands whose window reaches a vertical wall take the checked path
  const bool wallx = band == 0 || band * OWN + 64 - 2 > A.nx - 1;
  if (wallx) march<T, ANISO, true, EFIX>(A, wsm, mbar, band, y0, y1, kdt);
  else march<T, ANISO, false, EFIX>(A, wsm, mbar, band, y0, y1, kdt);
  pdl_trigger();
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
  s = smul(h, rs);
  vx = smul(qx, rs);
  vy = smul(qy, rs);
}

template <typename T>
__global__ void cart1_dt0_kernel(const T* __restrict__ h, const T* __restrict__ qx,
                                 const T* __restrict__ qy, const T* __restrict__ hC,
                                 int nx, int ny, int pitch, T gh, T rho, void* tmax_out,
                                 unsigned* err) {
  T tmax = T(0);
  unsigned bad = 0;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  for (int j = blockIdx.y; i < nx && j < ny; j += gridDim.y) {
    const int64_t o = (int64_t)(j + kPadY) * pitch + i + kPadX;
    const T h0 = h[o], x0 = qx[o], y0 = qy[o], c0 = hC[o];
    if (!(isfinite(h0) && isfinite(x0) && isfinite(y0) && isfinite(c0))) bad |= kErrNonfinite;
    else if (!(h0 > T(0))) bad |= kErrDepth;
    T s0, vx0, vy0, sn, vxn, vyn;
    speed_inputs(h0, x0, y0, s0, vx0, vy0);
    // west and east edges
    T hw = h0, sw = s0, vw = -vx0;
    if (i > 0) { hw = h[o - 1]; speed_inputs(hw, qx[o - 1], qy[o - 1], sn, vxn, vyn); sw = sn; vw = vxn; }
    T he = h0, se = s0, ve = -vx0;
    if (i < nx - 1) { he = h[o + 1]; speed_inputs(he, qx[o + 1], qy[o + 1], sn, vxn, vyn); se = sn; ve = vxn; }
    // south and north edges
    T hs = h0, ss = s0, vs = -vy0;
    if (j > 0) { hs = h[o - pitch]; speed_inputs(hs, qx[o - pitch], qy[o - pitch], sn, vxn, vyn); ss = sn; vs = vyn; }
    T hN = h0, sN = s0, vN = -vy0;
    if (j < ny - 1) { hN = h[o + pitch]; speed_inputs(hN, qx[o + pitch], qy[o + pitch], sn, vxn, vyn); sN = sn; vN = vyn; }
    T sum = sadd(speed_scalar(h0, s0, vx0, he, se, ve, gh), speed_scalar(hw, sw, vw, h0, s0, vx0, gh));
    sum = sadd(sum, smul(speed_scalar(hs, ss, vs, h0, s0, vy0, gh), rho));
    sum = sadd(sum, smul(speed_scalar(h0, s0, vy0, hN, sN, vN, gh), rho));
    tmax = nanmax(tmax, sum);
  }
  if (bad) atomicOr(err, bad);
  warp_max_publish<T>(tmax, tmax_out);
}

// The bounded wait of the march on a barrier nothing arrives on: it must
// give up after `budget` cycles and report kErrTimeout.
__global__ void wait_selftest_kernel(long long budget, unsigned* err) {
  __shared__ uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    mbar_init_fence();
  }
  __syncwarp();
  const bool ok = mbar_wait_bounded(b, 0u, budget);
  if (!__all_sync(kFull, ok) && threadIdx.x == 0) atomicOr(err, kErrTimeout);
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
  return (size_t)kWarpsPerBlock * kStages * stage_bytes<T>() +
         (size_t)kWarpsPerBlock * kStages * sizeof(uint64_t);
}

template <typename T>
cudaError_t step_occupancy(int* blocks_per_sm, size_t* smem_bytes, bool efix) {
  const size_t smem = step_smem_bytes<T>();
  *smem_bytes = smem;
  cudaError_t e;
  auto allow = [&](auto kernel) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  };
  if ((e = allow(cart1_step_kernel<T, false, false>)) != cudaSuccess) return e;
  if ((e = allow(cart1_step_kernel<T, true, false>)) != cudaSuccess) return e;
  if ((e = allow(cart1_step_kernel<T, false, true>)) != cudaSuccess) return e;
  if ((e = allow(cart1_step_kernel<T, true, true>)) != cudaSuccess) return e;
  return efix ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                    blocks_per_sm, cart1_step_kernel<T, false, true>, kWarpsPerBlock * 32, smem)
              : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                    blocks_per_sm, cart1_step_kernel<T, false, false>, kWarpsPerBlock * 32, smem);
}

template <typename T>
cudaError_t launch_step(const StepArgs<T>& a, int blocks, cudaStream_t st) {
  const size_t smem = step_smem_bytes<T>();
  const dim3 nt(kWarpsPerBlock * 32);
  if (a.efix)
    return a.rho == T(1) ? launch_pdl(cart1_step_kernel<T, false, true>, blocks, nt, smem, st, a)
                         : launch_pdl(cart1_step_kernel<T, true, true>, blocks, nt, smem, st, a);
  return a.rho == T(1) ? launch_pdl(cart1_step_kernel<T, false, false>, blocks, nt, smem, st, a)
                       : launch_pdl(cart1_step_kernel<T, true, false>, blocks, nt, smem, st, a);
}

template <typename T>
cudaError_t launch_dt0(const T* const* w, const T* H, int nx, int ny, int pitch, T ghalf, T rho,
                       void* tmax_out, unsigned* err, cudaStream_t st) {
  (void)H;
  dim3 grid((unsigned)((nx + 127) / 128), (unsigned)(ny < 1024 ? ny : 1024));
  cart1_dt0_kernel<T><<<grid, 128, 0, st>>>(w[0], w[1], w[2], w[3], nx, ny, pitch, ghalf, rho,
                                            tmax_out, err);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(long long budget_cycles, unsigned* err, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(budget_cycles, err);
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

template cudaError_t step_occupancy<float>(int*, size_t*, bool);
template cudaError_t step_occupancy<double>(int*, size_t*, bool);
template cudaError_t launch_step<float>(const StepArgs<float>&, int, cudaStream_t);
template cudaError_t launch_step<double>(const StepArgs<double>&, int, cudaStream_t);
template cudaError_t launch_dt0<float>(const float* const*, const float*, int, int, int, float,
                                       float, void*, unsigned*, cudaStream_t);
template cudaError_t launch_dt0<double>(const double* const*, const double*, int, int, int, double,
                                        double, void*, unsigned*, cudaStream_t);
template cudaError_t launch_fill<float>(float*, int64_t, float, cudaStream_t);
template cudaError_t launch_fill<double>(double*, int64_t, double, cudaStream_t);

}  // namespace swe
