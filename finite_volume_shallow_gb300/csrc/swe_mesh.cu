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
// Two launches per step, no floating-point atomics on results:
//   mesh_tile_kernel    tiles of consecutive cells (compact patches,
//                       swe_mesh_prep.cpp), each staged with its halo in
//                       shared memory: the rotated Roe flux of every edge of
//                       the tile once (eq. (2)-(3)), then each cell's three
//                       edges summed in a fixed order, R / |V_i| stored and
//                       sum L max|lambda| / |V_i| max-reduced for dt;
//   mesh_update_kernel  W -= dt R / |V_i| in place, checks, dt bookkeeping.
// Algorithm 1's edge and volume loops thus meet in shared memory; the
// per-edge results never travel through DRAM.
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

// ---- the tile kernel -------------------------------------------------------
// Per tile (see swe_internal.h) three phases:
//   1. the tile's cells and its halo cells (W^n and H) into shared memory;
//   2. every slot of the tile: the Roe flux of the edge from the staged
//      cells, written per slot to shared memory, what each side adds;
//   3. every cell of the tile: its three slots summed as e0 + (e1 + e2), the
//      residual R / |V_i| stored, and sum L max|lambda| / |V_i| max-reduced
//      for dt.
// An edge on a tile border is evaluated by both tiles from the same inputs,
// so both sides see the same flux and mass and pollutant stay conserved.

// staged cells: field f of local cell i at cw[f * kTileCap + i] (H last)
template <typename T>
__device__ __forceinline__ Side1<T> side1_of(const T* cw, int i, T ex, T ey) {
  Side1<T> s;
  const T h = cw[i], qx = cw[kTileCap + i], qy = cw[2 * kTileCap + i];
  s.h = h;
  s.rs = M2<T>::rsq(h);
  s.s = h * s.rs;
  s.qn = qx * ex + qy * ey;
  s.qt = -qx * ey + qy * ex;
  s.hc = cw[3 * kTileCap + i];
  s.H = cw[4 * kTileCap + i];
  return s;
}

template <typename T>
__device__ __forceinline__ Side2<T> side2_of(const T* cw, int i, T ex, T ey) {
  Side2<T> s;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const T h = cw[3 * k * kTileCap + i], qx = cw[(3 * k + 1) * kTileCap + i];
    const T qy = cw[(3 * k + 2) * kTileCap + i];
    s.h[k] = h;
    s.rs[k] = M2<T>::rsq(h);
    s.s[k] = h * s.rs[k];
    s.qn[k] = qx * ex + qy * ey;
    s.qt[k] = -qx * ey + qy * ex;
  }
  s.H = cw[6 * kTileCap + i];
  return s;
}

// (normal, tangential) components in the edge frame -> (x, y), times L, into
// result q of slot j
template <typename T>
__device__ __forceinline__ void put_xy(T* er, int j, int q, T L, T fn, T ft, T ex, T ey) {
  er[q * kTileSlots + j] = L * (fn * ex - ft * ey);
  er[(q + 1) * kTileSlots + j] = L * (fn * ey + ft * ex);
}

// One slot: the edge's flux from the staged cells into er.  Returns false
// when a two-layer Roe matrix has a complex pair of eigenvalues.
template <typename T>
struct Slot {
  int32_t ab;
  T ex, ey, L;
};
template <typename T>
__device__ __forceinline__ Slot<T> load_slot(const MeshStepArgs<T>& A, int64_t gs) {
  return Slot<T>{A.slot_ab[gs], A.slot_nx[gs], A.slot_ny[gs], A.slot_len[gs]};
}

template <typename T, int NL, bool EFIX>
__device__ __forceinline__ bool tile_edge(const MeshStepArgs<T>& A, const T* cw, T* er, int j,
                                          const Slot<T>& sl) {
  using Lay = MeshLayout<NL>;
  const int la = sl.ab & 0xffff, lb = (sl.ab >> 16) & 0xffff;
  const T ex = sl.ex, ey = sl.ey, L = sl.L;
  const bool wall = lb == kTileWall;
  const T gh = T(0.5) * A.g;
  if constexpr (NL == 1) {
    const Side1<T> sa = side1_of(cw, la, ex, ey);
    Side1<T> sb = sa;  // wall: mirror ghost (normal discharge negated)
    if (wall) sb.qn = -sa.qn;
    else sb = side1_of(cw, lb, ex, ey);
    T m, p, pa, pb, t, D;
    edge1<T, EFIX>(sa, sb, gh, wall, m, p, pa, pb, t, D);
    er[0 * kTileSlots + j] = L * m;
    er[1 * kTileSlots + j] = L * p;
    const T ta = t - sa.qn * (sa.qt * sa.rs * sa.rs);
    put_xy(er, j, Lay::a_mom, L, pa, ta, ex, ey);
    if (!wall) {
      const T tb = sb.qn * (sb.qt * sb.rs * sb.rs) - t;
      put_xy(er, j, Lay::b_mom, L, pb, tb, ex, ey);
    }
    er[Lay::d * kTileSlots + j] = L * D;
    return true;
  } else {
    const Side2<T> sa = side2_of(cw, la, ex, ey);
    Side2<T> sb;
    if (wall) mirror2(sb, sa);
    else sb = side2_of(cw, lb, ex, ey);
    T out[NEQ];
    const bool ok = edge2<T, true, EFIX>(sa, sb, A.g, gh, A.r, wall, out);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const T m = out[k ? E_M2 : E_M1];
      const T t = out[k ? E_T2 : E_T1];
      er[k * kTileSlots + j] = L * m;
      const T ta = t - sa.qn[k] * (sa.qt[k] * sa.rs[k] * sa.rs[k]);
      put_xy(er, j, Lay::a_mom + 2 * k, L, out[k ? E_PM2 : E_PM1], ta, ex, ey);
      if (!wall) {
        const T tb = sb.qn[k] * (sb.qt[k] * sb.rs[k] * sb.rs[k]) - t;
        put_xy(er, j, Lay::b_mom + 2 * k, L, out[k ? E_PS2 : E_PS1], tb, ex, ey);
      }
    }
    er[Lay::d * kTileSlots + j] = L * out[E_D];
    return ok;
  }
}

// Two layers, fp32: slots j and j + 1 on the packed FP32x2 pipe (edge2p).
// Every tile's slot range starts at an even index and has even length.
__device__ __forceinline__ void side2p_of(const float* cw, int i0, int i1, float2 ex, float2 ey,
                                          Side2P& s) {
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float* f = cw + 3 * k * kTileCap;
    const float2 h = f2(f[i0], f[i1]);
    const float2 qx = f2(f[kTileCap + i0], f[kTileCap + i1]);
    const float2 qy = f2(f[2 * kTileCap + i0], f[2 * kTileCap + i1]);
    s.h[k] = h;
    s.rs[k] = rsq2(h);
    s.s[k] = mul2(h, s.rs[k]);
    s.qn[k] = fma2(qx, ex, mul2(qy, ey));
    s.qt[k] = fma2(qy, ex, f2(-(qx.x * ey.x), -(qx.y * ey.y)));
  }
  s.H = f2(cw[6 * kTileCap + i0], cw[6 * kTileCap + i1]);
}

struct SlotPair {
  int2 ab;
  float2 ex, ey, L;
};
__device__ __forceinline__ SlotPair load_slot_pair(const MeshStepArgs<float>& A, int64_t gs) {
  return SlotPair{*reinterpret_cast<const int2*>(A.slot_ab + gs),
                  *reinterpret_cast<const float2*>(A.slot_nx + gs),
                  *reinterpret_cast<const float2*>(A.slot_ny + gs),
                  *reinterpret_cast<const float2*>(A.slot_len + gs)};
}

template <bool EFIX>
__device__ __forceinline__ bool tile_edge_pair(const MeshStepArgs<float>& A, const float* cw,
                                               float* er, int j, const SlotPair& sp) {
  const int2 ab = sp.ab;
  const float2 ex = sp.ex, ey = sp.ey, L = sp.L;
  const int la0 = ab.x & 0xffff, lb0 = (ab.x >> 16) & 0xffff;
  const int la1 = ab.y & 0xffff, lb1 = (ab.y >> 16) & 0xffff;
  const bool w0 = lb0 == kTileWall, w1 = lb1 == kTileWall;
  Side2P sa, sb;
  side2p_of(cw, la0, la1, ex, ey, sa);
  side2p_of(cw, w0 ? la0 : lb0, w1 ? la1 : lb1, ex, ey, sb);
  // walls: the mirror ghost has the normal discharge negated
  if (w0) { sb.qn[0].x = -sa.qn[0].x; sb.qn[1].x = -sa.qn[1].x; }
  if (w1) { sb.qn[0].y = -sa.qn[0].y; sb.qn[1].y = -sa.qn[1].y; }
  float2 out[NEQ];
  const bool ok = edge2p<EFIX>(sa, sb, A.g, 0.5f * A.g, A.r, w0, w1, out) == 3u;
  auto put = [&](int q, float2 v) { *reinterpret_cast<float2*>(er + q * kTileSlots + j) = v; };
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
  return ok;
}

// Residual of cell c from its three slots, summed as e0 + (e1 + e2): stores
// R / |V_c| and returns sum L max|lambda| / |V_c|.
template <typename T, int NL>
__device__ __forceinline__ T cell_residual(const MeshStepArgs<T>& A, const T* er, int64_t c,
                                           uint2 cr, T ia) {
  using Lay = MeshLayout<NL>;
  constexpr int NF = Lay::nf;
  const uint32_t rk[3] = {cr.x & 0xffffu, cr.x >> 16, cr.y & 0xffffu};
  T v[3][NF], d[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    const int j = (int)(rk[k] & 0x7fffu);
    const bool bside = (rk[k] >> 15) != 0;
    const int q = bside ? Lay::b_mom : Lay::a_mom;
    const T sg = bside ? T(-1) : T(1);
    v[k][0] = sg * er[0 * kTileSlots + j];
    v[k][1] = er[q * kTileSlots + j];
    v[k][2] = er[(q + 1) * kTileSlots + j];
    v[k][3] = sg * er[1 * kTileSlots + j];
    if constexpr (NL == 2) {
      v[k][4] = er[(q + 2) * kTileSlots + j];
      v[k][5] = er[(q + 3) * kTileSlots + j];
    }
    d[k] = er[Lay::d * kTileSlots + j];
  }
#pragma unroll
  for (int f = 0; f < NF; ++f) A.R[f][c] = (v[0][f] + (v[1][f] + v[2][f])) * ia;
  return (d[0] + (d[1] + d[2])) * ia;
}

// ---- mesh_tile_kernel: persistent and pipelined ------------------------------
// Each block walks the tiles blockIdx.x, blockIdx.x + gridDim.x, ... and,
// while it evaluates tile k, stages in shared memory with cp.async: the
// cells and halo cells of tile k + 1 (into the other of two buffers), the
// halo indices of tile k + 2 (which the addresses of its halo cells need)
// and the header of tile k + 3 (which the halo indices need).  The slot data
// of tile k + 1 is read into registers after the edge phase of tile k.  All
// of it has the whole edge and cell phases of a tile to land, so a block's
// loads overlap its own arithmetic; with tiles of equal size the blocks of
// one SM would otherwise load, and then compute, at the same time.
// Threads per block: 256, but 512 for two layers in fp64 without the
// entropy fix (one slot per thread): there the shared memory holds one
// block per SM, and the FP64 pipe wants more warps than eight.
template <typename T, int NL, bool EFIX>
constexpr int pipe_threads() {
  return (sizeof(T) == 8 && NL == 2 && !EFIX) ? 512 : 256;
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
template <typename T>
__device__ __forceinline__ void cp_async_el(T* dst, const T* src) {
  if constexpr (sizeof(T) == 8) cp_async8(dst, src);
  else cp_async4(dst, src);
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// shared memory: two cell buffers (nf fields and H of the tile's cells and
// halo), three halo-index buffers, the slot results.  Three blocks of the
// two-layer form take at most 196 KB of shared memory, so the SM keeps the
// larger of its L1 configurations for the few registers that spill.
template <int NL>
constexpr int pipe_cell_words() {
  return (MeshLayout<NL>::nf + 1) * kTileCap;
}
template <typename T, int NL>
constexpr size_t pipe_smem() {
  return (size_t)(2 * pipe_cell_words<NL>() + MeshLayout<NL>::ne * kTileSlots) * sizeof(T) +
         (size_t)3 * kTileHalo * sizeof(int32_t);
}

struct TileHdr {
  int32_t c0, nct, h0, nh, s0, ns;
};
// header entry: tile_cell, tile_halo and tile_slot at t and t + 1
template <typename T>
__device__ __forceinline__ void request_hdr(const MeshStepArgs<T>& A, int32_t* e, int t) {
  const int i = threadIdx.x;
  if (i < 6) {
    const int32_t* src = i < 2 ? A.tile_cell : (i < 4 ? A.tile_halo : A.tile_slot);
    cp_async4(e + i, src + t + (i & 1));
  }
}
__device__ __forceinline__ TileHdr read_hdr(const int32_t* e) {
  return TileHdr{e[0], e[1] - e[0], e[2], e[3] - e[2], e[4], e[5] - e[4]};
}
template <int NT, typename T>
__device__ __forceinline__ void request_hidx(const MeshStepArgs<T>& A, int32_t* hidx,
                                             const TileHdr& h) {
  for (int k = threadIdx.x; k < h.nh; k += NT) cp_async4(hidx + k, A.halo + h.h0 + k);
}
template <int NT, typename T, int NL>
__device__ __forceinline__ void request_cells(const MeshStepArgs<T>& A, T* buf,
                                              const int32_t* hidx, const TileHdr& h) {
  constexpr int NF = MeshLayout<NL>::nf;
  for (int i = threadIdx.x; i < h.nct + h.nh; i += NT) {
    const int64_t c = i < h.nct ? (int64_t)h.c0 + i : (int64_t)hidx[i - h.nct];
#pragma unroll
    for (int f = 0; f < NF; ++f) cp_async_el(buf + f * kTileCap + i, A.w[f] + c);
    cp_async_el(buf + NF * kTileCap + i, A.H + c);
  }
}

// slot data of one tile in registers: a pair per thread (PAIR, 256
// threads), else kTileSlots / NT single slots
template <typename T, bool PAIR, int NT> struct PipeSlots {
  Slot<T> s[kTileSlots / NT];
};
template <int NT> struct PipeSlots<float, true, NT> {
  SlotPair p;
};
template <int NT, typename T, bool PAIR>
__device__ __forceinline__ void load_slots(const MeshStepArgs<T>& A, const TileHdr& h,
                                           PipeSlots<T, PAIR, NT>& r) {
  if constexpr (PAIR) {
    const int j = 2 * threadIdx.x;
    if (j < h.ns) r.p = load_slot_pair(A, (int64_t)h.s0 + j);
  } else {
#pragma unroll
    for (int k = 0; k < kTileSlots / NT; ++k) {
      const int j = threadIdx.x + k * NT;
      if (j < h.ns) r.s[k] = load_slot(A, (int64_t)h.s0 + j);
    }
  }
}

#ifndef SWE_PIPE_PAIR_MIN_BLOCKS
#define SWE_PIPE_PAIR_MIN_BLOCKS 2
#endif
// Blocks per SM the registers are held to: as many as the shared memory
// admits in fp32 (the packed two-layer form spills a little at three); in
// fp64 the FP64 pipe is the bound and one or two blocks keep it busy.
template <typename T, int NL, bool EFIX, bool PAIR> struct PipeMinBlocks {
  static constexpr int v = 1;
};
template <> struct PipeMinBlocks<float, 2, false, true> {
  static constexpr int v = SWE_PIPE_PAIR_MIN_BLOCKS;
};
template <> struct PipeMinBlocks<float, 2, true, true> { static constexpr int v = 2; };
template <> struct PipeMinBlocks<float, 1, false, false> { static constexpr int v = 4; };
template <> struct PipeMinBlocks<float, 1, true, false> { static constexpr int v = 4; };

// Overlapped form (OVL): two slot-result buffers, so that one phase
// evaluates the edges of tile k + 1 and sums the cells of tile k, with one
// barrier per tile instead of two; the staging runs one tile further ahead
// (cells k + 2, halo indices k + 3, headers k + 4) and each tile's cell
// references and areas are staged too.  It needs more shared memory: chosen
// per variant by measurement (SWE_MESH_OVERLAP: bit 0 one layer fp32, 1 two
// layers fp32, 2 one layer fp64, 3 two layers fp64).  On the 2.1M-triangle
// workloads (CUDA events per step): two layers fp32 0.0876 ms against
// 0.1014, fp64 2.670 against 2.699; one layer fp32 0.0673 against 0.0553
// and fp64 0.853 against 0.773, where the extra shared memory costs a block
// per SM.
#ifndef SWE_MESH_OVERLAP
#define SWE_MESH_OVERLAP 0xa
#endif
template <typename T, int NL>
constexpr bool pipe_overlap() {
  return (SWE_MESH_OVERLAP >> ((sizeof(T) == 8 ? 2 : 0) + (NL == 2 ? 1 : 0))) & 1;
}
// shared memory of the tile kernel
template <typename T, int NL>
constexpr size_t tile_smem() {
  if (!pipe_overlap<T, NL>()) return pipe_smem<T, NL>();
  return (size_t)(2 * pipe_cell_words<NL>() + 2 * MeshLayout<NL>::ne * kTileSlots +
                  2 * kTileCells) * sizeof(T) +
         (size_t)2 * kTileCells * sizeof(uint2) + (size_t)3 * kTileHalo * sizeof(int32_t);
}

template <int NT, typename T>
__device__ __forceinline__ void request_crefs(const MeshStepArgs<T>& A, uint2* cr, T* ia,
                                              const TileHdr& h) {
  for (int i = threadIdx.x; i < h.nct; i += NT) {
    cp_async8(cr + i, A.cref + (int64_t)h.c0 + i);
    cp_async_el(ia + i, A.inv_area + (int64_t)h.c0 + i);
  }
}

template <typename T, int NL, bool EFIX, bool PAIR>
__global__ void __launch_bounds__((pipe_threads<T, NL, EFIX>()), (PipeMinBlocks<T, NL, EFIX, PAIR>::v))
    mesh_tile_kernel(const MeshStepArgs<T> A) {
  constexpr int NT = pipe_threads<T, NL, EFIX>();
  constexpr int NSL = kTileSlots / NT;
  constexpr int NCL = (kTileCells + NT - 1) / NT;
  constexpr int NE = MeshLayout<NL>::ne * kTileSlots;
  static_assert(!PAIR || NT == 256, "the packed pair form has 256 threads");
  extern __shared__ __align__(16) unsigned char tile_smem[];
  const int G = gridDim.x, nt = (int)A.ntiles, tid = threadIdx.x;
  const int t0 = blockIdx.x;  // < nt: the grid never exceeds the tile count
  auto valid = [&](int k) { return t0 + k * G < nt; };
  bool ok = true;
  T m = T(0);
  PipeSlots<T, PAIR, NT> sl;
  // the edges of a staged tile into er
  auto edges = [&](const T* cw, T* er, const int32_t* h) {
    const int ns = h[5] - h[4];
    if constexpr (PAIR) {
      static_assert(sizeof(T) == 4, "the packed pair form is fp32");
      if (2 * tid < ns) ok &= tile_edge_pair<EFIX>(A, cw, er, 2 * tid, sl.p);
    } else {
#pragma unroll
      for (int k = 0; k < NSL; ++k) {
        const int j = tid + k * NT;
        if (j < ns) ok &= tile_edge<T, NL, EFIX>(A, cw, er, j, sl.s[k]);
      }
    }
  };
  pdl_wait();
  if constexpr (!pipe_overlap<T, NL>()) {
    __shared__ __align__(16) int32_t ring[4][8];
    T* const cbuf = reinterpret_cast<T*>(tile_smem);
    T* const er = cbuf + 2 * pipe_cell_words<NL>();
    int32_t* const hbuf = reinterpret_cast<int32_t*>(er + NE);
    // prologue: headers of tiles 0-2 of this block, halo indices of tiles
    // 0-1, cells of tile 0, slots of tile 0
    for (int k = 0; k < 3; ++k)
      if (valid(k)) request_hdr(A, ring[k], t0 + k * G);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    for (int k = 0; k < 2; ++k)
      if (valid(k)) request_hidx<NT>(A, hbuf + k * kTileHalo, read_hdr(ring[k]));
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    request_cells<NT, T, NL>(A, cbuf, hbuf, read_hdr(ring[0]));
    cp_async_commit();
    load_slots<NT>(A, read_hdr(ring[0]), sl);
    cp_async_wait_all();
    __syncthreads();
    for (int it = 0;; ++it) {
      const int t = t0 + it * G;
      const bool more = valid(it + 1);
      const int32_t* hcur = ring[it & 3];
      // staging ahead: header k + 3, halo indices k + 2, cells k + 1
      if (valid(it + 3)) request_hdr(A, ring[(it + 3) & 3], t + 3 * G);
      if (valid(it + 2))
        request_hidx<NT>(A, hbuf + ((it + 2) % 3) * kTileHalo, read_hdr(ring[(it + 2) & 3]));
      if (more)
        request_cells<NT, T, NL>(A, cbuf + ((it + 1) & 1) * pipe_cell_words<NL>(),
                                 hbuf + ((it + 1) % 3) * kTileHalo, read_hdr(ring[(it + 1) & 3]));
      cp_async_commit();
      edges(cbuf + (it & 1) * pipe_cell_words<NL>(), er, hcur);
      // the next tile's slots; this tile's cell references and areas
      if (more) load_slots<NT>(A, read_hdr(ring[(it + 1) & 3]), sl);
      const int c0 = hcur[0], nct = hcur[1] - hcur[0];
      uint2 cr[NCL];
      T ia[NCL];
#pragma unroll
      for (int k = 0; k < NCL; ++k) {
        const int i = tid + k * NT;
        if (i < nct) {
          cr[k] = A.cref[(int64_t)c0 + i];
          ia[k] = A.inv_area[(int64_t)c0 + i];
        }
      }
      __syncthreads();  // slot results complete
#pragma unroll
      for (int k = 0; k < NCL; ++k) {
        const int i = tid + k * NT;
        if (i < nct) m = nanmax2(m, cell_residual<T, NL>(A, er, (int64_t)c0 + i, cr[k], ia[k]));
      }
      cp_async_wait_all();
      __syncthreads();  // what was staged landed; slot results free
      if (!more) break;
    }
  } else {
    __shared__ __align__(16) int32_t ring[8][8];
    T* const cbuf = reinterpret_cast<T*>(tile_smem);
    T* const erb = cbuf + 2 * pipe_cell_words<NL>();
    T* const iab = erb + 2 * NE;
    uint2* const crb = reinterpret_cast<uint2*>(iab + 2 * kTileCells);
    int32_t* const hbuf = reinterpret_cast<int32_t*>(crb + 2 * kTileCells);
    auto cbuf_of = [&](int k) { return cbuf + (k & 1) * pipe_cell_words<NL>(); };
    auto hidx_of = [&](int k) { return hbuf + (k % 3) * kTileHalo; };
    // prologue: headers of tiles 0-3, halo indices of tiles 0-2, cells of
    // tiles 0-1, cell references of tile 0, slots of tile 0; edges of tile 0
    for (int k = 0; k < 4; ++k)
      if (valid(k)) request_hdr(A, ring[k], t0 + k * G);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    for (int k = 0; k < 3; ++k)
      if (valid(k)) request_hidx<NT>(A, hidx_of(k), read_hdr(ring[k]));
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    for (int k = 0; k < 2; ++k)
      if (valid(k)) request_cells<NT, T, NL>(A, cbuf_of(k), hidx_of(k), read_hdr(ring[k]));
    request_crefs<NT>(A, crb, iab, read_hdr(ring[0]));
    cp_async_commit();
    load_slots<NT>(A, read_hdr(ring[0]), sl);
    cp_async_wait_all();
    __syncthreads();
    edges(cbuf_of(0), erb, ring[0]);
    if (valid(1)) load_slots<NT>(A, read_hdr(ring[1]), sl);
    __syncthreads();
    for (int it = 0;; ++it) {
      const int t = t0 + it * G;
      const bool more = valid(it + 1);
      // staging ahead: header k + 4, halo indices k + 3, cells k + 2, cell
      // references k + 1
      if (valid(it + 4)) request_hdr(A, ring[(it + 4) & 7], t + 4 * G);
      if (valid(it + 3)) request_hidx<NT>(A, hidx_of(it + 3), read_hdr(ring[(it + 3) & 7]));
      if (valid(it + 2))
        request_cells<NT, T, NL>(A, cbuf_of(it + 2), hidx_of(it + 2), read_hdr(ring[(it + 2) & 7]));
      if (more)
        request_crefs<NT>(A, crb + ((it + 1) & 1) * kTileCells, iab + ((it + 1) & 1) * kTileCells,
                          read_hdr(ring[(it + 1) & 7]));
      cp_async_commit();
      // edges of the next tile
      if (more) {
        edges(cbuf_of(it + 1), erb + ((it + 1) & 1) * NE, ring[(it + 1) & 7]);
        if (valid(it + 2)) load_slots<NT>(A, read_hdr(ring[(it + 2) & 7]), sl);
      }
      // cells of this tile
      {
        const int32_t* h = ring[it & 7];
        const int c0 = h[0], nct = h[1] - h[0];
        const T* er = erb + (it & 1) * NE;
        const uint2* cr = crb + (it & 1) * kTileCells;
        const T* ia = iab + (it & 1) * kTileCells;
        for (int i = tid; i < nct; i += NT)
          m = nanmax2(m, cell_residual<T, NL>(A, er, (int64_t)c0 + i, cr[i], ia[i]));
      }
      cp_async_wait_all();
      __syncthreads();  // staged data landed; next slot results complete
      if (!more) break;
    }
  }
  pdl_trigger();
  if (NL == 2 && !__syncthreads_and(ok) && tid == 0) atomicOr(A.err, kErrHyperbolic);
  block_max_publish<T, NT / 32>(m, A.tmax_out);
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

template <typename T, int NL, bool EFIX, bool PAIR>
cudaError_t pipe_prepare(int64_t ntiles, int* grid) {
  cudaError_t e = cudaFuncSetAttribute(mesh_tile_kernel<T, NL, EFIX, PAIR>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)tile_smem<T, NL>());
  if (e != cudaSuccess) return e;
  int bpsm = 0, dev = 0, sms = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &bpsm, mesh_tile_kernel<T, NL, EFIX, PAIR>, pipe_threads<T, NL, EFIX>(), tile_smem<T, NL>());
  if (e != cudaSuccess) return e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  int64_t g = (int64_t)(bpsm > 0 ? bpsm : 1) * sms;
  if (g > ntiles) g = ntiles;
  *grid = (int)(g > 0 ? g : 1);
  return cudaSuccess;
}

}  // namespace

template <typename T>
cudaError_t mesh_prepare(int n_layers, int efix, int64_t ntiles, int* grid) {
  constexpr bool F32 = sizeof(T) == 4;
  if (n_layers == 2 && efix) return pipe_prepare<T, 2, true, F32>(ntiles, grid);
  if (n_layers == 2) return pipe_prepare<T, 2, false, F32>(ntiles, grid);
  if (efix) return pipe_prepare<T, 1, true, false>(ntiles, grid);
  return pipe_prepare<T, 1, false, false>(ntiles, grid);
}

int mesh_tile_warps(int precision, int n_layers, int efix) {
  if (precision == 64 && n_layers == 2 && !efix) return pipe_threads<double, 2, false>() / 32;
  return pipe_threads<float, 1, false>() / 32;
}

namespace {

template <typename T, int NL, bool EFIX, bool PAIR>
cudaError_t launch_pipe(const MeshStepArgs<T>& f, cudaStream_t st) {
  return launch_pdl(mesh_tile_kernel<T, NL, EFIX, PAIR>, (unsigned)f.grid,
                    pipe_threads<T, NL, EFIX>(), tile_smem<T, NL>(), st, f);
}

// The tile kernel of a step: two layers in fp32 two slots per thread on the
// FP32x2 pipe, else one.
template <typename T>
cudaError_t launch_tile(const MeshStepArgs<T>& f, int n_layers, cudaStream_t st) {
  constexpr bool F32 = sizeof(T) == 4;
  if (n_layers == 2 && f.efix) return launch_pipe<T, 2, true, F32>(f, st);
  if (n_layers == 2) return launch_pipe<T, 2, false, F32>(f, st);
  if (f.efix) return launch_pipe<T, 1, true, false>(f, st);
  return launch_pipe<T, 1, false, false>(f, st);
}

}  // namespace

template <typename T>
cudaError_t launch_mesh_step(const MeshStepArgs<T>& f, const MeshUpdateArgs<T>& u, int n_layers,
                             cudaStream_t st, const cudaEvent_t* marks) {
  const unsigned gu = grid_1d((u.ncells + Vec<T>::n - 1) / Vec<T>::n, 256, 152 * 8);
  auto mark = [&](int k) {
    if (marks) cudaEventRecord(marks[k], st);
  };
  mark(0);
  cudaError_t e = launch_tile<T>(f, n_layers, st);
  if (e != cudaSuccess) return e;
  mark(1);
  e = n_layers == 2 ? launch_pdl(mesh_update_kernel<T, 2>, gu, 256, 0, st, u)
                    : launch_pdl(mesh_update_kernel<T, 1>, gu, 256, 0, st, u);
  if (e != cudaSuccess) return e;
  mark(2);
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

template cudaError_t mesh_prepare<float>(int, int, int64_t, int*);
template cudaError_t mesh_prepare<double>(int, int, int64_t, int*);
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
