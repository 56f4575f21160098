// swe_mesh.cu -- sm_103a kernels of the IR-Roe step on an unstructured
// triangle mesh, one or two layers.
//
// Scheme: An MPI-CUDA implementation of an improved Roe method for two-layer
// shallow water systems, Sec. 2.2 (finite volumes V_i with edges Gamma_ij of
// unit normal eta_ij; update eq. (4), numerical flux steps 1-4, CFL eq. (5))
// and Sec. 3 / Algorithm 1 (edge-parallel flux processing, then per-volume
// accumulation, global dt minimum and volume update).  The one-layer variant
// carries the pollutant of A multi-GPU shallow-water simulation with
// transport of contaminants (abstract: a transport equation for hC).
//
// Three launches per step, no floating-point atomics on results:
//   mesh_edge_kernel    one thread per edge: the rotated Roe flux of the edge
//                       (eq. (2)-(3)), evaluated once for both of its cells;
//                       writes what each side adds to its residual;
//   mesh_gather_kernel  one thread per cell: sums its three edge records in
//                       a fixed order (a CSR gather), stores R / |V_i| and
//                       max-reduces sum L max|lambda| / |V_i| for dt;
//   mesh_update_kernel  W -= dt R / |V_i| in place, checks, dt bookkeeping.
//
// Momentum enters in fluctuation form: each side keeps only P^- d (side a)
// or P^+ d (side b) of the normal component and the tangential transport
// minus its own cell's tangential flux.  The cell's own physical flux sums
// to F(W_i) . sum_j |Gamma_ij| eta_ij = 0 over a closed cell, so this equals
// eq. (4) exactly, and a lake at rest stays at rest to the last bit whatever
// the rounding of the stored normals.  Mass and pollutant stay in flux form
// (one value per edge, added by a and subtracted by b), so they are conserved
// to rounding on any mesh.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "swe_internal.h"
#include "swe_roe2.cuh"

namespace swe {
namespace {

constexpr int kEdgeThreads = 256;
constexpr int kCellThreads = 256;

// ---- one layer ----------------------------------------------------------------
template <typename T>
struct Side1 {
  T h, s, rs, qn, qt, hc, H;
};

// One-layer IR-Roe flux of an edge in the frame of its normal (2 x 2 Roe
// matrix [[0, 1], [c^2 - u^2, 2u]], eigenvalues u -+ c, eigenvectors
// (1, lambda_k)); tangential discharge and pollutant upwinded on the mass
// flux.  out (not yet multiplied by L): m, m C_up, normal fluctuation of a
// and of b, tangential transport m u_t,up, max|lambda|.
//
// EFIX adds the Harten-Hyman entropy fix ([P1] Sec. 2.2, after eq. (5)) as
// numerical viscosity along each wave: with delta_k the spread of the
// speed lambda_k between the two cells' own states (u_eta -+ sqrt(g h)),
// |lambda_k| < delta_k replaces |lambda_k| by (lambda_k^2 + delta_k^2) /
// (2 delta_k), and Phi^- gains nu_k K_k, nu_k = (|lambda_k| - |lambda_k|_d)
// beta_k / 2, beta = K^-1 (W_j - W_i).  The same term leaves side b's
// fluctuation P^+ d, so the pair stays conservative.
template <typename T>
__device__ __forceinline__ T hh_nu(T l, T lL, T lR, T beta) {
  const T del = fmax(T(0), fmax(l - lL, lR - l));
  const T al = fabs(l);
  if (!(al < del)) return T(0);
  return T(0.5) * (al - (l * l + del * del) * M2<T>::rcp(del + del)) * beta;
}
template <typename T, bool EFIX>
__device__ __forceinline__ void edge1(const Side1<T>& a, const Side1<T>& b, T gh, bool wall,
                                      T& m, T& p, T& pa, T& pb, T& t, T& D) {
  const T un = (a.qn * a.rs + b.qn * b.rs) * M2<T>::rcp(a.s + b.s);
  const T cs = gh * (a.h + b.h);  // g hbar
  const T c = M2<T>::sq(cs);
  const T l1 = un - c, l2 = un + c;
  const T iha = a.rs * a.rs, ihb = b.rs * b.rs;
  // d = F(W_j) - F(W_i) - S_ij (H_j - H_i), pressure difference as g hbar dh
  const T d1 = b.qn - a.qn;
  const T d2 = (b.qn * b.qn * ihb - a.qn * a.qn * iha) + cs * ((b.h - a.h) - (b.H - a.H));
  // coordinates in the eigenvector basis: K^-1 d, det K = 2c
  const T i2c = M2<T>::rcp(c + c);
  const T w1 = (l1 < T(0)) ? T(1) : ((l1 > T(0)) ? T(0) : T(0.5));
  const T w2 = (l2 < T(0)) ? T(1) : ((l2 > T(0)) ? T(0) : T(0.5));
  const T a1 = w1 * (l2 * d1 - d2) * i2c;
  const T a2 = w2 * (d2 - l1 * d1) * i2c;
  T pd0 = a1 + a2;
  T pd1 = a1 * l1 + a2 * l2;
  pb = d2 - pd1;
  if (EFIX) {
    const T sg = M2<T>::sq(gh + gh);  // sqrt(g)
    const T ua = a.qn * iha, ub = b.qn * ihb;
    const T ca = sg * a.s, cb = sg * b.s;
    const T dh = b.h - a.h;
    const T n1 = hh_nu(l1, ua - ca, ub - cb, (l2 * dh - d1) * i2c);
    const T n2 = hh_nu(l2, ua + ca, ub + cb, (d1 - l1 * dh) * i2c);
    pd0 += n1 + n2;
    const T cmom = n1 * l1 + n2 * l2;
    pd1 += cmom;
    pb -= cmom;
  }
  m = wall ? T(0) : a.qn + pd0;
  pa = pd1;
  const bool up = m > T(0);
  t = m * (up ? a.qt * iha : b.qt * ihb);
  p = m * (up ? a.hc * iha : b.hc * ihb);
  D = fmax(fabs(l1), fabs(l2));
}

template <typename T>
__device__ __forceinline__ Side1<T> load_side1(const MeshStepArgs<T>& A, int32_t c, T ex, T ey) {
  Side1<T> s;
  const T h = A.w[0][c], qx = A.w[1][c], qy = A.w[2][c];
  s.h = h;
  s.rs = M2<T>::rsq(h);
  s.s = h * s.rs;
  s.qn = qx * ex + qy * ey;
  s.qt = -qx * ey + qy * ex;
  s.hc = A.w[3][c];
  s.H = A.H[c];
  return s;
}

template <typename T>
__device__ __forceinline__ Side2<T> load_side2(const MeshStepArgs<T>& A, int32_t c, T ex, T ey) {
  Side2<T> s;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const T h = A.w[3 * k][c], qx = A.w[3 * k + 1][c], qy = A.w[3 * k + 2][c];
    s.h[k] = h;
    s.rs[k] = M2<T>::rsq(h);
    s.s[k] = h * s.rs[k];
    s.qn[k] = qx * ex + qy * ey;
    s.qt[k] = -qx * ey + qy * ex;
  }
  s.H = A.H[c];
  return s;
}

// (normal, tangential) components in the edge frame -> (x, y), times L
template <typename T>
__device__ __forceinline__ void put_xy(T* buf, int64_t st, int64_t e, int q, T L, T fn, T ft,
                                       T ex, T ey) {
  buf[q * st + e] = L * (fn * ex - ft * ey);
  buf[(q + 1) * st + e] = L * (fn * ey + ft * ex);
}

template <typename T, int NL, bool EFIX = false>
__global__ void __launch_bounds__(kEdgeThreads) mesh_edge_kernel(const MeshStepArgs<T> A) {
  using Lay = MeshLayout<NL>;
  const int64_t e = (int64_t)blockIdx.x * kEdgeThreads + threadIdx.x;
  bool ok = true;
  pdl_wait();
  if (e < A.nedges) {
    const int32_t a = A.ea[e], b = A.eb[e];
    const T ex = A.enx[e], ey = A.eny[e], L = A.elen[e];
    const bool wall = b < 0;
    const T gh = T(0.5) * A.g;
    T* buf = A.ebuf;
    const int64_t st = A.estride;
    if constexpr (NL == 1) {
      const Side1<T> sa = load_side1(A, a, ex, ey);
      Side1<T> sb = sa;  // wall: mirror ghost (normal discharge negated)
      if (wall) sb.qn = -sa.qn;
      else sb = load_side1(A, b, ex, ey);
      T m, p, pa, pb, t, D;
      edge1<T, EFIX>(sa, sb, gh, wall, m, p, pa, pb, t, D);
      buf[0 * st + e] = L * m;
      buf[1 * st + e] = L * p;
      const T ta = t - sa.qn * (sa.qt * sa.rs * sa.rs);
      put_xy(buf, st, e, Lay::a_mom, L, pa, ta, ex, ey);
      if (!wall) {
        const T tb = sb.qn * (sb.qt * sb.rs * sb.rs) - t;
        put_xy(buf, st, e, Lay::b_mom, L, pb, tb, ex, ey);
      }
      buf[Lay::d * st + e] = L * D;
    } else {
      const Side2<T> sa = load_side2(A, a, ex, ey);
      Side2<T> sb;
      if (wall) mirror2(sb, sa);
      else sb = load_side2(A, b, ex, ey);
      T out[NEQ];
      ok = edge2<T, true, EFIX>(sa, sb, A.g, gh, A.r, wall, out);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const T m = out[k ? E_M2 : E_M1];
        const T t = out[k ? E_T2 : E_T1];
        buf[k * st + e] = L * m;
        const T ta = t - sa.qn[k] * (sa.qt[k] * sa.rs[k] * sa.rs[k]);
        put_xy(buf, st, e, Lay::a_mom + 2 * k, L, out[k ? E_PM2 : E_PM1], ta, ex, ey);
        if (!wall) {
          const T tb = sb.qn[k] * (sb.qt[k] * sb.rs[k] * sb.rs[k]) - t;
          put_xy(buf, st, e, Lay::b_mom + 2 * k, L, out[k ? E_PS2 : E_PS1], tb, ex, ey);
        }
      }
      buf[Lay::d * st + e] = L * out[E_D];
    }
  }
  pdl_trigger();
  if (NL == 2 && !__all_sync(kFull2, ok) && (threadIdx.x & 31) == 0) atomicOr(A.err, kErrHyperbolic);
}

// ---- two layers, fp32: two edges per thread on the packed FP32x2 pipe -------
// (edge2p and its FP32x2 helpers are in swe_roe2.cuh)

__device__ __forceinline__ void load_side2p(const MeshStepArgs<float>& A, int32_t c0, int32_t c1,
                                            float2 ex, float2 ey, Side2P& s) {
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float2 h = f2(A.w[3 * k][c0], A.w[3 * k][c1]);
    const float2 qx = f2(A.w[3 * k + 1][c0], A.w[3 * k + 1][c1]);
    const float2 qy = f2(A.w[3 * k + 2][c0], A.w[3 * k + 2][c1]);
    s.h[k] = h;
    s.rs[k] = rsq2(h);
    s.s[k] = mul2(h, s.rs[k]);
    s.qn[k] = fma2(qx, ex, mul2(qy, ey));
    s.qt[k] = fma2(qy, ex, f2(-(qx.x * ey.x), -(qx.y * ey.y)));
  }
  s.H = f2(A.H[c0], A.H[c1]);
}

// Two layers, fp32: edges 2t and 2t + 1.  Every edge array is 256-byte
// aligned with room for one element past an odd count, so the pair loads
// and stores stay inside the allocation; the missing second edge of an odd
// count takes the first edge's data and its results land in that padding.
constexpr int kPairThreads = 128;
// Blocks per SM the registers are held to: six (80 registers) leave the
// per-edge convergence state unspilled; seven spilled 32 bytes and ran 2 %
// slower on the 2.1M-triangle two-layer mesh.
#ifndef SWE_PAIR_MIN_BLOCKS
#define SWE_PAIR_MIN_BLOCKS 6
#endif
__global__ void __launch_bounds__(kPairThreads, SWE_PAIR_MIN_BLOCKS)
    mesh_edge2_pair_kernel(const MeshStepArgs<float> A) {
  const int64_t e0 = 2 * ((int64_t)blockIdx.x * kPairThreads + threadIdx.x);
  bool ok = true;
  pdl_wait();
  if (e0 < A.nedges) {
    const bool both = e0 + 1 < A.nedges;
    int2 ia = *reinterpret_cast<const int2*>(A.ea + e0);
    int2 ib = *reinterpret_cast<const int2*>(A.eb + e0);
    float2 ex = *reinterpret_cast<const float2*>(A.enx + e0);
    float2 ey = *reinterpret_cast<const float2*>(A.eny + e0);
    float2 L = *reinterpret_cast<const float2*>(A.elen + e0);
    if (!both) {
      ia.y = ia.x; ib.y = ib.x; ex.y = ex.x; ey.y = ey.x; L.y = L.x;
    }
    const bool w0 = ib.x < 0, w1 = ib.y < 0;
    Side2P sa, sb;
    load_side2p(A, ia.x, ia.y, ex, ey, sa);
    load_side2p(A, w0 ? ia.x : ib.x, w1 ? ia.y : ib.y, ex, ey, sb);
    // walls: the mirror ghost has the normal discharge negated
    if (w0) { sb.qn[0].x = -sa.qn[0].x; sb.qn[1].x = -sa.qn[1].x; }
    if (w1) { sb.qn[0].y = -sa.qn[0].y; sb.qn[1].y = -sa.qn[1].y; }
    float2 out[NEQ];
    ok = edge2p(sa, sb, A.g, 0.5f * A.g, A.r, w0, w1, out) == 3u;
    float* buf = A.ebuf;
    const int64_t st = A.estride;
    auto put = [&](int q, float2 v) { *reinterpret_cast<float2*>(buf + q * st + e0) = v; };
    using Lay = MeshLayout<2>;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float2 m = out[k ? E_M2 : E_M1];
      const float2 t = out[k ? E_T2 : E_T1];
      put(k, mul2(L, m));
      const float2 ta = sub2(t, mul2(sa.qn[k], mul2(sa.qt[k], mul2(sa.rs[k], sa.rs[k]))));
      const float2 tb = sub2(mul2(sb.qn[k], mul2(sb.qt[k], mul2(sb.rs[k], sb.rs[k]))), t);
      const float2 pa = out[k ? E_PM2 : E_PM1], pb = out[k ? E_PS2 : E_PS1];
      // (normal, tangential) -> (x, y), times L
      put(Lay::a_mom + 2 * k, mul2(L, fma2(pa, ex, f2(-(ta.x * ey.x), -(ta.y * ey.y)))));
      put(Lay::a_mom + 2 * k + 1, mul2(L, fma2(pa, ey, mul2(ta, ex))));
      put(Lay::b_mom + 2 * k, mul2(L, fma2(pb, ex, f2(-(tb.x * ey.x), -(tb.y * ey.y)))));
      put(Lay::b_mom + 2 * k + 1, mul2(L, fma2(pb, ey, mul2(tb, ex))));
    }
    put(Lay::d, mul2(L, out[E_D]));
  }
  pdl_trigger();
  if (!__all_sync(kFull2, ok) && (threadIdx.x & 31) == 0) atomicOr(A.err, kErrHyperbolic);
}

// residual of one cell: its three edges, summed as e0 + (e1 + e2)
template <typename T, int NL>
__global__ void __launch_bounds__(kCellThreads) mesh_gather_kernel(const MeshStepArgs<T> A) {
  using Lay = MeshLayout<NL>;
  constexpr int NF = Lay::nf;
  const int64_t c = (int64_t)blockIdx.x * kCellThreads + threadIdx.x;
  T m = T(0);
  pdl_wait();
  if (c < A.ncells) {
    const T* buf = A.ebuf;
    const int64_t st = A.estride;
    T v[3][NF], d[3];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int32_t ref = A.ref[k][c];
      const int64_t e = ref >> 1;
      const bool bside = ref & 1;
      const int q = bside ? Lay::b_mom : Lay::a_mom;
      const T s = bside ? T(-1) : T(1);
      if constexpr (NL == 1) {
        v[k][0] = s * buf[0 * st + e];
        v[k][1] = buf[q * st + e];
        v[k][2] = buf[(q + 1) * st + e];
        v[k][3] = s * buf[1 * st + e];
      } else {
        v[k][0] = s * buf[0 * st + e];
        v[k][1] = buf[q * st + e];
        v[k][2] = buf[(q + 1) * st + e];
        v[k][3] = s * buf[1 * st + e];
        v[k][4] = buf[(q + 2) * st + e];
        v[k][5] = buf[(q + 3) * st + e];
      }
      d[k] = buf[Lay::d * st + e];
    }
    const T ia = A.inv_area[c];
#pragma unroll
    for (int f = 0; f < NF; ++f) A.R[f][c] = (v[0][f] + (v[1][f] + v[2][f])) * ia;
    m = (d[0] + (d[1] + d[2])) * ia;
  }
  pdl_trigger();
  block_max_publish<T, kCellThreads / 32>(m, A.tmax_out);
}

// Vector width of the update: 16-byte loads and stores.
template <typename T> struct Vec;
template <> struct Vec<float> { using type = float4; static constexpr int n = 4; };
template <> struct Vec<double> { using type = double2; static constexpr int n = 2; };

template <typename T, int NL>
__global__ void __launch_bounds__(256) mesh_update_kernel(const MeshUpdateArgs<T> A) {
  constexpr int NF = MeshLayout<NL>::nf;
  using V = typename Vec<T>::type;
  constexpr int VN = Vec<T>::n;
  // dt = 2 cfl / max_i (sum L max|lambda| / |V_i|), once per block
  __shared__ T k_sh;
  pdl_wait();
  if (threadIdx.x == 0) {
    const T tm = *reinterpret_cast<const T*>(A.tmax_in);
    const double dt = A.two_cfl / (double)tm;
    k_sh = (T)dt;
    if (blockIdx.x == 0) {
      A.dt_hist[A.step % kHistCap] = dt;
      *A.t_dev += dt;
      if (sizeof(T) == 4) *reinterpret_cast<unsigned*>(A.tmax_clear) = 0u;
      else *reinterpret_cast<unsigned long long*>(A.tmax_clear) = 0ull;
    }
  }
  __syncthreads();
  const T k = k_sh;
  unsigned bad = 0;
  auto check = [&](const T* w) {
    T sum = T(0);
#pragma unroll
    for (int f = 0; f < NF; ++f) sum += w[f];
    if (!(fabs(sum) <= M2<T>::big())) bad |= kErrNonfinite;
    if (!(w[0] > T(0))) bad |= kErrDepth;
    if (NL == 2 && !(w[3] > T(0))) bad |= kErrDepth;
  };
  // field arrays start 256-byte aligned: whole vectors, then a scalar tail
  const int64_t nvec = A.ncells / VN;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec; i += stride) {
    V wv[NF], rv[NF];
#pragma unroll
    for (int f = 0; f < NF; ++f) {
      wv[f] = reinterpret_cast<const V*>(A.w[f])[i];
      rv[f] = reinterpret_cast<const V*>(A.R[f])[i];
    }
#pragma unroll
    for (int f = 0; f < NF; ++f) {
      T* w = reinterpret_cast<T*>(&wv[f]);
      const T* r = reinterpret_cast<const T*>(&rv[f]);
#pragma unroll
      for (int j = 0; j < VN; ++j) w[j] = w[j] - k * r[j];
      reinterpret_cast<V*>(A.w[f])[i] = wv[f];
    }
#pragma unroll
    for (int j = 0; j < VN; ++j) {
      T w[NF];
#pragma unroll
      for (int f = 0; f < NF; ++f) w[f] = reinterpret_cast<const T*>(&wv[f])[j];
      check(w);
    }
  }
  for (int64_t c = nvec * VN + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < A.ncells;
       c += stride) {
    T w[NF];
#pragma unroll
    for (int f = 0; f < NF; ++f) {
      w[f] = A.w[f][c] - k * A.R[f][c];
      A.w[f][c] = w[f];
    }
    check(w);
  }
  pdl_trigger();
  if (bad) atomicOr(A.err, bad);
}

template <typename T>
__global__ void mesh_check_kernel(const Fields6<T> w, int nf, int nl, int64_t n, unsigned* err) {
  unsigned bad = 0;
  for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < n;
       c += (int64_t)gridDim.x * blockDim.x) {
    T s = T(0);
    for (int f = 0; f < nf; ++f) s += w.p[f][c];
    if (!isfinite(s)) bad |= kErrNonfinite;
    if (!(w.p[0][c] > T(0))) bad |= kErrDepth;
    if (nl == 2 && !(w.p[3][c] > T(0))) bad |= kErrDepth;
  }
  if (bad) atomicOr(err, bad);
}

template <typename T>
struct Ptr6 {
  T* p[6];
};

template <typename T>
__global__ void mesh_permute_kernel(Ptr6<T> dst, Fields6<T> src, int nf, const int32_t* idx,
                                    int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t j = idx[i];
    for (int f = 0; f < nf; ++f) dst.p[f][i] = src.p[f][j];
  }
}

unsigned grid_1d(int64_t n, int threads, int64_t cap) {
  int64_t b = (n + threads - 1) / threads;
  if (b > cap) b = cap;
  if (b < 1) b = 1;
  return (unsigned)b;
}

}  // namespace

template <typename T>
cudaError_t launch_mesh_step(const MeshStepArgs<T>& f, const MeshUpdateArgs<T>& u, int n_layers,
                             cudaStream_t st, const cudaEvent_t* marks) {
  const unsigned ge = grid_1d(f.nedges, kEdgeThreads, INT32_MAX);
  const unsigned gc = grid_1d(f.ncells, kCellThreads, INT32_MAX);
  const unsigned gu = grid_1d((u.ncells + Vec<T>::n - 1) / Vec<T>::n, 256, 152 * 8);
  auto mark = [&](int k) {
    if (marks) cudaEventRecord(marks[k], st);
  };
  mark(0);
  cudaError_t e;
  if (n_layers == 2 && f.efix) {
    // with the entropy fix both precisions take the one-edge-per-thread form
    e = launch_pdl(mesh_edge_kernel<T, 2, true>, ge, kEdgeThreads, 0, st, f);
  } else if (n_layers == 2) {
    if constexpr (sizeof(T) == 4) {
      const unsigned gp = grid_1d((f.nedges + 1) / 2, kPairThreads, INT32_MAX);
      e = launch_pdl(mesh_edge2_pair_kernel, gp, kPairThreads, 0, st, f);
    } else {
      e = launch_pdl(mesh_edge_kernel<T, 2>, ge, kEdgeThreads, 0, st, f);
    }
  } else if (f.efix) {
    e = launch_pdl(mesh_edge_kernel<T, 1, true>, ge, kEdgeThreads, 0, st, f);
  } else {
    e = launch_pdl(mesh_edge_kernel<T, 1>, ge, kEdgeThreads, 0, st, f);
  }
  if (e != cudaSuccess) return e;
  mark(1);
  e = n_layers == 2 ? launch_pdl(mesh_gather_kernel<T, 2>, gc, kCellThreads, 0, st, f)
                    : launch_pdl(mesh_gather_kernel<T, 1>, gc, kCellThreads, 0, st, f);
  if (e != cudaSuccess) return e;
  mark(2);
  e = n_layers == 2 ? launch_pdl(mesh_update_kernel<T, 2>, gu, 256, 0, st, u)
                    : launch_pdl(mesh_update_kernel<T, 1>, gu, 256, 0, st, u);
  if (e != cudaSuccess) return e;
  mark(3);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_mesh_check(const Fields6<T>& w, int n_layers, int64_t ncells, unsigned* err,
                              cudaStream_t st) {
  mesh_check_kernel<T><<<grid_1d(ncells, 256, 4096), 256, 0, st>>>(
      w, n_layers == 2 ? 6 : 4, n_layers, ncells, err);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_mesh_permute(T* const* dst, const T* const* src, int nf, const int32_t* idx,
                                int64_t n, cudaStream_t st) {
  Ptr6<T> d{};
  Fields6<T> s{};
  for (int f = 0; f < nf; ++f) {
    d.p[f] = dst[f];
    s.p[f] = src[f];
  }
  mesh_permute_kernel<T><<<grid_1d(n, 256, 4096), 256, 0, st>>>(d, s, nf, idx, n);
  return cudaGetLastError();
}

template cudaError_t launch_mesh_step<float>(const MeshStepArgs<float>&,
                                             const MeshUpdateArgs<float>&, int, cudaStream_t,
                                             const cudaEvent_t*);
template cudaError_t launch_mesh_step<double>(const MeshStepArgs<double>&,
                                              const MeshUpdateArgs<double>&, int, cudaStream_t,
                                              const cudaEvent_t*);
template cudaError_t launch_mesh_check<float>(const Fields6<float>&, int, int64_t, unsigned*,
                                              cudaStream_t);
template cudaError_t launch_mesh_check<double>(const Fields6<double>&, int, int64_t, unsigned*,
                                               cudaStream_t);
template cudaError_t launch_mesh_permute<float>(float* const*, const float* const*, int,
                                                const int32_t*, int64_t, cudaStream_t);
template cudaError_t launch_mesh_permute<double>(double* const*, const double* const*, int,
                                                 const int32_t*, int64_t, cudaStream_t);

}  // namespace swe
