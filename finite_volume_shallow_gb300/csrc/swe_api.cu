// swe_api.cu -- host side of the libswe C ABI (include/swe.h): argument
// checking, device memory, launch orchestration and the dt bookkeeping of
// the time loop of An MPI-CUDA implementation of an improved Roe method for
// two-layer shallow water systems, Sec. 3 and Algorithm 1 (edges, per-volume
// dt, global minimum, volume update, t += dt), on one GPU.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <new>
#include <vector>

#include "../../include/swe.h"
#include "swe_internal.h"
#include "swe_plan.h"

using namespace swe;

struct swe_state {
  int nx = 0, ny = 0;
  double dx = 0, dy = 0;
  swe_params p{};
  int prec = 0;
  int nl = 1;        // layers
  int nf = 4;        // conserved fields: 4 (h, qx, qy, hC) or 6 (two layers)
  size_t esz = 0;
  int pitch = 0;
  int64_t rows = 0;  // allocated rows per field
  int64_t field_stride = 0;  // elements between field bases in the allocation
  void* dev = nullptr;
  size_t dev_bytes = 0;
  void* w[2][6] = {{nullptr}};  // two buffers of the 4 (one layer) or 6 fields
  void* R[6] = {nullptr};        // residual scratch (two layers: buffer 0; meshes)
  void* R1[6] = {nullptr};       // two layers on a grid: residual buffer 1
  int lazy2 = -1;     // two layers on a grid: buffer holding a step whose
                      // update is still to be applied (inside swe_run only)
  double cfl2 = 0;    // the cfl of that step
  void* H = nullptr;
  void* slots = nullptr;      // 3 wave-speed maxima (8 bytes each)
  double* dt_hist = nullptr;
  double* t_dev = nullptr;
  unsigned* err = nullptr;
  int cur = 0;
  int64_t step = 0;
  cudaStream_t stream = nullptr;
  int nbands = 0, nsegs = 0, nsegs_wall = 0, blocks = 0;
  double* h_dt = nullptr;     // pinned readback
  unsigned* h_err = nullptr;
  double* h_t = nullptr;
  unsigned sticky = 0;
  // triangle meshes
  bool mesh = false;
  int64_t ncells = 0, nedges = 0, ntiles = 0;
  int mesh_grid = 0;                 // blocks of the (persistent) tile kernel
  void* tile_cell = nullptr;         // int32 [ntiles + 1]
  void* tile_halo = nullptr;
  void* tile_slot = nullptr;
  void* halo = nullptr;              // int32 [halo entries]
  void* slot_ab = nullptr;           // int32 [slots]
  void* slot_nx = nullptr;           // T [slots]
  void* slot_ny = nullptr;
  void* slot_len = nullptr;
  void* cref = nullptr;              // uint2 [ncells]
  void* inv_area = nullptr;          // T [ncells]
  int32_t* new_of_old = nullptr;     // device [ncells]
  int32_t* old_of_new = nullptr;
  std::vector<int32_t> h_new_of_old;  // host copy (swe_cell_index)
  struct Timing* timing = nullptr;    // per-kernel event ring (swe_set_timing)
  const cudaEvent_t* marks = nullptr; // events of the step being enqueued, or null
  int* mark_kid = nullptr;            // with marks: kernel index of each interval
  int* mark_n = nullptr;              // with marks: intervals recorded so far
  // one layer with wet/dry fronts on a grid (swe_params.wet_dry)
  bool wd = false;
};

// Per-kernel device time: a ring of event sets, one set per step; a set is
// read back when its slot comes round again (so the host runs at most
// kSlots steps ahead while timing) and on swe_get_timing.
struct Timing {
  static constexpr int kSlots = 64, kMaxK = 3;
  cudaEvent_t ev[kSlots][kMaxK + 1] = {};
  int kid[kSlots][kMaxK] = {};  // kernel of the interval ev[k] .. ev[k + 1]
  int cnt[kSlots] = {};         // intervals of the slot's step
  bool pending[kSlots] = {};
  int next = 0, nk = 0;
  const char* names[kMaxK] = {};
  double ms[kMaxK] = {};
  int64_t launches[kMaxK] = {};
  bool on = false;
};

namespace {

swe_status status_of_bits(unsigned bits) {
  if (bits & kErrTimeout) return SWE_ERR_TIMEOUT;
  if (bits & kErrHyperbolic) return SWE_ERR_HYPERBOLIC;
  if (bits & kErrNonfinite) return SWE_ERR_NONFINITE;
  if (bits & kErrDepth) return SWE_ERR_DEPTH;
  return SWE_OK;
}

swe_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return SWE_OK;
  (void)cudaGetLastError();  // clear a non-sticky error
  return e == cudaErrorMemoryAllocation ? SWE_ERR_OOM : SWE_ERR_CUDA;
}

#define CK(call)                                   \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) return cuda_status(e_); \
  } while (0)

int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// Launch shape: one warp per (column band, row segment), see plan_step.

template <typename T>
swe_status plan_launch(swe_state* s) {
  int bpsm = 0;
  size_t smem = 0;
  CK(step_occupancy<T>(&bpsm, &smem, s->p.entropy_fix != 0));
  int dev = 0, sms = 0;
  CK(cudaGetDevice(&dev));
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  if (bpsm < 1) return SWE_ERR_CUDA;
  const int64_t slots = (int64_t)sms * bpsm * kWarpsPerBlock;
  const int own = band_owned<T>();
  const StepPlan pl = plan_step(slots, (s->nx + own - 1) / own, s->ny);
  s->nbands = pl.nbands;
  s->nsegs = pl.nsegs;
  s->nsegs_wall = pl.nsegs_wall;
  s->blocks = (pl.units + kWarpsPerBlock - 1) / kWarpsPerBlock;
  return SWE_OK;
}

// Two layers: one warp per (band of kBand2 columns, row segment), about one
// unit per resident warp; segments of at least 16 rows.
template <typename T>
swe_status plan_launch2(swe_state* s) {
  int bpsm = 0, dev = 0, sms = 0;
  CK(march2_occupancy<T>(&bpsm, s->p.entropy_fix != 0));
  CK(cudaGetDevice(&dev));
  CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  if (bpsm < 1) return SWE_ERR_CUDA;
  const int64_t slots = (int64_t)sms * bpsm * kMarch2Warps;
  const int64_t nb = (s->nx + kBand2 - 1) / kBand2;
  int64_t S = slots / nb;
  const int64_t most = s->ny / 16 > 1 ? s->ny / 16 : 1;
  if (S > most) S = most;
  if (S < 1) S = 1;
  s->nbands = (int)nb;
  s->nsegs = (int)S;
  s->nsegs_wall = (int)S;
  return SWE_OK;
}

template <typename T>
swe_status enqueue_dt0(swe_state* s) {
  // all three wave-speed slots to zero, then slot (step % 3) <- max of W^n
  CK(cudaMemsetAsync(s->slots, 0, 3 * sizeof(uint64_t), s->stream));
  const T* w[4] = {(const T*)s->w[s->cur][0], (const T*)s->w[s->cur][1],
                   (const T*)s->w[s->cur][2], (const T*)s->w[s->cur][3]};
  void* slot = (char*)s->slots + (s->step % 3) * sizeof(uint64_t);
  CK(launch_dt0<T>(w, (const T*)s->H, s->nx, s->ny, s->pitch, (T)(0.5 * s->p.g),
                   (T)(s->dx / s->dy), slot, s->err, s->stream));
  return SWE_OK;
}

template <typename T>
swe_status enqueue_step(swe_state* s, double cfl) {
  StepArgs<T> a;
  for (int f = 0; f < 4; ++f) {
    a.win[f] = (const T*)s->w[s->cur][f];
    a.wout[f] = (T*)s->w[s->cur ^ 1][f];
  }
  a.H = (const T*)s->H;
  a.nx = s->nx;
  a.ny = s->ny;
  a.pitch = s->pitch;
  a.nbands = s->nbands;
  a.nsegs = s->nsegs;
  a.nsegs_wall = s->nsegs_wall;
  a.ghalf = (T)(0.5 * s->p.g);
  a.rho = (T)(s->dx / s->dy);
  a.two_cfl = 2.0 * cfl;
  a.dx = s->dx;
  char* sl = (char*)s->slots;
  a.tmax_in = sl + (s->step % 3) * sizeof(uint64_t);
  a.tmax_out = sl + ((s->step + 1) % 3) * sizeof(uint64_t);
  a.tmax_clear = sl + ((s->step + 2) % 3) * sizeof(uint64_t);
  a.dt_hist = s->dt_hist;
  a.t_dev = s->t_dev;
  a.step = s->step;
  a.err = s->err;
  a.efix = s->p.entropy_fix;
  if (s->marks) CK(cudaEventRecord(s->marks[0], s->stream));
  CK(launch_step<T>(a, s->blocks, s->stream));
  if (s->marks) CK(cudaEventRecord(s->marks[1], s->stream));
  s->cur ^= 1;
  s->step += 1;
  return SWE_OK;
}

// Two layers: the flux pass of step n reduces the wave-speed maximum of W^n
// into slot n % 3 (zeroed by the update of step n - 1 or at set-up); the
// update pass of step n reads it and zeroes slot (n + 1) % 3.
template <typename T>
swe_status enqueue_check2(swe_state* s) {
  CK(cudaMemsetAsync(s->slots, 0, 3 * sizeof(uint64_t), s->stream));
  Fields6<T> w;
  for (int f = 0; f < 6; ++f) w.p[f] = (const T*)s->w[0][f];
  CK(launch_check2<T>(w, s->nx, s->ny, s->pitch, s->err, s->stream));
  return SWE_OK;
}

// Per-kernel timing of a step whose kernels vary: mark(k) before kernel k,
// mark_end() after the last.
swe_status mark(swe_state* s, int kid) {
  if (!s->marks) return SWE_OK;
  const int n = *s->mark_n;
  CK(cudaEventRecord(s->marks[n], s->stream));
  s->mark_kid[n] = kid;
  *s->mark_n = n + 1;
  return SWE_OK;
}
swe_status mark_end(swe_state* s) {
  if (!s->marks) return SWE_OK;
  CK(cudaEventRecord(s->marks[*s->mark_n], s->stream));
  return SWE_OK;
}

// Step m of a two-layer grid.  Without a pending update: the flux pass of
// W^m (buffer 0).  With one (step m - 1 left W^{m-1}, R^{m-1} in buffer a):
// the fused pass, which applies it and evaluates the fluxes of W^m into
// buffer a ^ 1.  `last`: then apply step m's own update into buffer 0.
// Wave-speed slots: the flux of step m reduces into slot m % 3, which must
// be zero; the update of step m (fused or not) reads it and zeroes slot
// (m + 1) % 3; the update that ends a run also zeroes slot (m + 2) % 3, the
// one the first fused pass of the next run reduces into (the set-up zeroes
// all three).
template <typename T>
swe_status enqueue_step2(swe_state* s, double cfl, bool last) {
  char* sl = (char*)s->slots;
  auto slot = [&](int64_t m) { return (void*)(sl + (m % 3) * sizeof(uint64_t)); };
  auto rbuf = [&](int b) { return b == 0 ? s->R : s->R1; };
  const int64_t m = s->step;
  Step2Args<T> f;
  f.H = (const T*)s->H;
  f.nx = s->nx;
  f.ny = s->ny;
  f.pitch = s->pitch;
  f.g = (T)s->p.g;
  f.r = (T)s->p.r;
  f.rho = (T)(s->dx / s->dy);
  f.tmax_out = slot(m);
  f.err = s->err;
  f.efix = s->p.entropy_fix;
  f.nbands = s->nbands;
  f.nsegs = s->nsegs;
  auto upd_args = [&](Update2Args<T>& u, int a, int dst, int64_t step, double c, bool end) {
    for (int k = 0; k < 6; ++k) {
      u.win[k] = (const T*)s->w[a][k];
      u.w[k] = (T*)s->w[dst][k];
      u.R[k] = (const T*)rbuf(a)[k];
    }
    u.nx = s->nx;
    u.ny = s->ny;
    u.pitch = s->pitch;
    u.two_cfl = 2.0 * c;
    u.dx = s->dx;
    u.tmax_in = slot(step);
    u.tmax_clear = slot(m + 1);
    u.tmax_clear2 = end ? slot(m + 2) : nullptr;
    u.dt_hist = s->dt_hist;
    u.t_dev = s->t_dev;
    u.step = step;
    u.err = s->err;
  };
  int a;
  swe_status st;
  if (s->lazy2 < 0) {
    a = 0;
    for (int k = 0; k < 6; ++k) {
      f.w[k] = (const T*)s->w[0][k];
      f.R[k] = (T*)s->R[k];
    }
    if ((st = mark(s, 0)) != SWE_OK) return st;
    CK(launch_flux2<T>(f, s->stream));
  } else {
    const int p = s->lazy2;
    a = p ^ 1;
    for (int k = 0; k < 6; ++k) {
      f.w[k] = (const T*)s->w[p][k];
      f.R[k] = (T*)rbuf(a)[k];
    }
    Update2Args<T> u;
    upd_args(u, p, a, m - 1, s->cfl2, false);
    if ((st = mark(s, 1)) != SWE_OK) return st;
    CK(launch_fused2<T>(f, u, s->stream));
  }
  s->step = m + 1;
  s->lazy2 = a;
  s->cfl2 = cfl;
  if (last) {
    Update2Args<T> u;
    upd_args(u, a, 0, m, cfl, true);
    if ((st = mark(s, 2)) != SWE_OK) return st;
    CK(launch_update2<T>(u, s->stream));
    s->lazy2 = -1;
  }
  return mark_end(s);
}

// Meshes: the tile pass of step n reduces into slot n % 3, the update of
// step n reads it and zeroes slot (n + 1) % 3 (as for two layers on a grid).
template <typename T>
swe_status enqueue_mesh_check(swe_state* s) {
  CK(cudaMemsetAsync(s->slots, 0, 3 * sizeof(uint64_t), s->stream));
  Fields6<T> w{};
  for (int f = 0; f < s->nf; ++f) w.p[f] = (const T*)s->w[0][f];
  CK(launch_mesh_check<T>(w, s->nl, s->ncells, s->err, s->stream));
  return SWE_OK;
}

template <typename T>
swe_status enqueue_mesh_step(swe_state* s, double cfl) {
  MeshStepArgs<T> f{};
  MeshUpdateArgs<T> u{};
  char* sl = (char*)s->slots;
  for (int k = 0; k < s->nf; ++k) {
    f.w[k] = (const T*)s->w[0][k];
    f.R[k] = (T*)s->R[k];
    u.w[k] = (T*)s->w[0][k];
    u.R[k] = (const T*)s->R[k];
  }
  f.H = (const T*)s->H;
  f.tile_cell = (const int32_t*)s->tile_cell;
  f.tile_halo = (const int32_t*)s->tile_halo;
  f.tile_slot = (const int32_t*)s->tile_slot;
  f.halo = (const int32_t*)s->halo;
  f.slot_ab = (const int32_t*)s->slot_ab;
  f.slot_nx = (const T*)s->slot_nx;
  f.slot_ny = (const T*)s->slot_ny;
  f.slot_len = (const T*)s->slot_len;
  f.cref = (const uint2*)s->cref;
  f.inv_area = (const T*)s->inv_area;
  f.ncells = u.ncells = s->ncells;
  f.ntiles = s->ntiles;
  f.grid = s->mesh_grid;
  f.g = (T)s->p.g;
  f.r = (T)s->p.r;
  f.tmax_out = sl + (s->step % 3) * sizeof(uint64_t);
  f.err = u.err = s->err;
  f.efix = s->p.entropy_fix;
  u.two_cfl = 2.0 * cfl;
  u.tmax_in = sl + (s->step % 3) * sizeof(uint64_t);
  u.tmax_clear = sl + ((s->step + 1) % 3) * sizeof(uint64_t);
  u.dt_hist = s->dt_hist;
  u.t_dev = s->t_dev;
  u.step = s->step;
  CK(launch_mesh_step<T>(f, u, s->nl, s->stream, s->marks));
  s->step += 1;
  return SWE_OK;
}

// Wet/dry: the cell pass of step n reduces into slot n % 3, the update of
// step n reads it and zeroes slot (n + 1) % 3 (all three zero at set-up).
template <typename T>
swe_status enqueue_wd_check(swe_state* s) {
  CK(cudaMemsetAsync(s->slots, 0, 3 * sizeof(uint64_t), s->stream));
  const T* w[4] = {(const T*)s->w[s->cur][0], (const T*)s->w[s->cur][1],
                   (const T*)s->w[s->cur][2], (const T*)s->w[s->cur][3]};
  CK(launch_wd_check<T>(w, s->nx, s->ny, s->pitch, s->err, s->stream));
  return SWE_OK;
}

template <typename T>
swe_status enqueue_wd_step(swe_state* s, double cfl) {
  WdStepArgs a{};
  for (int f = 0; f < 4; ++f) {
    a.win[f] = s->w[s->cur][f];
    a.wout[f] = s->w[s->cur ^ 1][f];
  }
  a.H = s->H;
  a.nx = s->nx;
  a.ny = s->ny;
  a.pitch = s->pitch;
  a.g = s->p.g;
  a.h_dry = s->p.h_dry;
  a.dx = s->dx;
  a.dy = s->dy;
  a.two_cfl = 2.0 * cfl;
  char* sl = (char*)s->slots;
  a.tmax_slot = sl + (s->step % 3) * sizeof(uint64_t);
  a.tmax_clear = sl + ((s->step + 1) % 3) * sizeof(uint64_t);
  a.dt_hist = s->dt_hist;
  a.t_dev = s->t_dev;
  a.step = s->step;
  a.err = s->err;
  a.efix = s->p.entropy_fix;
  CK(launch_wd_step<T>(a, s->stream, s->marks));
  s->cur ^= 1;
  s->step += 1;
  return SWE_OK;
}

swe_status enqueue_dt0_any(swe_state* s) {
  if (s->wd) return s->prec == 32 ? enqueue_wd_check<float>(s) : enqueue_wd_check<double>(s);
  if (s->mesh)
    return s->prec == 32 ? enqueue_mesh_check<float>(s) : enqueue_mesh_check<double>(s);
  if (s->nl == 2) return s->prec == 32 ? enqueue_check2<float>(s) : enqueue_check2<double>(s);
  return s->prec == 32 ? enqueue_dt0<float>(s) : enqueue_dt0<double>(s);
}
swe_status timing_harvest(Timing* tm, int slot) {
  if (!tm->pending[slot]) return SWE_OK;
  const int n = tm->cnt[slot];
  CK(cudaEventSynchronize(tm->ev[slot][n]));
  for (int k = 0; k < n; ++k) {
    float f = 0.f;
    CK(cudaEventElapsedTime(&f, tm->ev[slot][k], tm->ev[slot][k + 1]));
    tm->ms[tm->kid[slot][k]] += f;
    tm->launches[tm->kid[slot][k]] += 1;
  }
  tm->pending[slot] = false;
  return SWE_OK;
}

swe_status timing_harvest_all(swe_state* s) {
  Timing* tm = s->timing;
  if (!tm) return SWE_OK;
  for (int i = 0; i < Timing::kSlots; ++i) {
    const int slot = (tm->next + i) % Timing::kSlots;  // oldest first
    const swe_status st = timing_harvest(tm, slot);
    if (st != SWE_OK) return st;
  }
  return SWE_OK;
}

swe_status enqueue_step_timed(swe_state* s, double cfl, bool last);

// `last`: the last step of a swe_run / swe_step call (a two-layer grid then
// applies its pending update).
swe_status enqueue_step_any(swe_state* s, double cfl, bool last) {
  if (s->timing && s->timing->on) return enqueue_step_timed(s, cfl, last);
  if (s->wd) return s->prec == 32 ? enqueue_wd_step<float>(s, cfl) : enqueue_wd_step<double>(s, cfl);
  if (s->mesh)
    return s->prec == 32 ? enqueue_mesh_step<float>(s, cfl) : enqueue_mesh_step<double>(s, cfl);
  if (s->nl == 2)
    return s->prec == 32 ? enqueue_step2<float>(s, cfl, last)
                         : enqueue_step2<double>(s, cfl, last);
  return s->prec == 32 ? enqueue_step<float>(s, cfl) : enqueue_step<double>(s, cfl);
}

swe_status enqueue_step_timed(swe_state* s, double cfl, bool last) {
  Timing* tm = s->timing;
  const int slot = tm->next;
  swe_status st = timing_harvest(tm, slot);  // the slot's previous step
  if (st != SWE_OK) return st;
  s->marks = tm->ev[slot];
  s->mark_kid = tm->kid[slot];
  s->mark_n = &tm->cnt[slot];
  tm->cnt[slot] = 0;
  tm->on = false;  // plain enqueue below
  st = enqueue_step_any(s, cfl, last);
  tm->on = true;
  s->marks = nullptr;
  s->mark_kid = nullptr;
  s->mark_n = nullptr;
  if (st != SWE_OK) return st;
  if (s->mesh || s->nl == 1) {  // a fixed kernel sequence, marked by the launcher
    tm->cnt[slot] = tm->nk;
    for (int k = 0; k < tm->nk; ++k) tm->kid[slot][k] = k;
  }
  tm->pending[slot] = true;
  tm->next = (slot + 1) % Timing::kSlots;
  return SWE_OK;
}

void timing_names(swe_state* s, Timing* tm) {
  if (s->wd) {
    tm->nk = 2;
    tm->names[0] = "wd_speed_kernel";
    tm->names[1] = "wd_tile_kernel";
  } else if (s->mesh) {
    tm->nk = 2;
    tm->names[0] = "mesh_tile_kernel";
    tm->names[1] = "mesh_update_kernel";
  } else if (s->nl == 2) {
    tm->nk = 3;
    tm->names[0] = "cart2_march_kernel<plain>";
    tm->names[1] = "cart2_march_kernel<fused>";
    tm->names[2] = "cart2_update_kernel";
  } else {
    tm->nk = 1;
    tm->names[0] = "cart1_step_kernel";
  }
}

void timing_destroy(Timing* tm) {
  if (!tm) return;
  for (int i = 0; i < Timing::kSlots; ++i)
    for (int k = 0; k <= Timing::kMaxK; ++k)
      if (tm->ev[i][k]) cudaEventDestroy(tm->ev[i][k]);
  delete tm;
}

// Copy n host fields into the padded layout of `dst`.
swe_status upload(swe_state* s, void* const* dst, const void* const* src, int n) {
  const size_t row = (size_t)s->nx * s->esz;
  const size_t dpitch = (size_t)s->pitch * s->esz;
  const size_t off = ((size_t)kPadY * s->pitch + kPadX) * s->esz;
  for (int f = 0; f < n; ++f)
    CK(cudaMemcpy2DAsync((char*)dst[f] + off, dpitch, src[f], row, row, (size_t)s->ny,
                         cudaMemcpyHostToDevice, s->stream));
  return SWE_OK;
}

// Mesh fields: host (caller numbering) -> staging R -> internal order, and
// back.  R is scratch that every step rewrites before reading.
swe_status mesh_upload(swe_state* s, void* const* dst, const void* const* src, int n) {
  const size_t bytes = (size_t)s->ncells * s->esz;
  for (int f = 0; f < n; ++f)
    CK(cudaMemcpyAsync(s->R[f], src[f], bytes, cudaMemcpyHostToDevice, s->stream));
  if (s->prec == 32)
    CK(launch_mesh_permute<float>((float* const*)dst, (const float* const*)s->R, n,
                                  s->old_of_new, s->ncells, s->stream));
  else
    CK(launch_mesh_permute<double>((double* const*)dst, (const double* const*)s->R, n,
                                   s->old_of_new, s->ncells, s->stream));
  return SWE_OK;
}

swe_status mesh_download(swe_state* s, void* const* dst) {
  if (s->prec == 32)
    CK(launch_mesh_permute<float>((float* const*)s->R, (const float* const*)s->w[0], s->nf,
                                  s->new_of_old, s->ncells, s->stream));
  else
    CK(launch_mesh_permute<double>((double* const*)s->R, (const double* const*)s->w[0], s->nf,
                                   s->new_of_old, s->ncells, s->stream));
  const size_t bytes = (size_t)s->ncells * s->esz;
  for (int f = 0; f < s->nf; ++f)
    CK(cudaMemcpyAsync(dst[f], s->R[f], bytes, cudaMemcpyDeviceToHost, s->stream));
  return SWE_OK;
}

swe_status read_err(swe_state* s) {
  CK(cudaMemcpyAsync(s->h_err, s->err, sizeof(unsigned), cudaMemcpyDeviceToHost, s->stream));
  CK(cudaStreamSynchronize(s->stream));
  s->sticky |= *s->h_err;
  return SWE_OK;
}

bool finite_pos(double v) { return isfinite(v) && v > 0.0; }

template <typename T>
swe_status fill_pads(swe_state* s) {
  // whole padded arrays: depths 1, everything else 0; interiors are then
  // copied (a resting state in the padding keeps every padded edge benign)
  const int64_t n = s->field_stride;
  for (int b = 0; b < 2; ++b)
    for (int f = 0; f < s->nf; ++f) {
      const bool depth = f == 0 || (s->nl == 2 && f == 3);
      CK(launch_fill<T>((T*)s->w[b][f], n, depth ? T(1) : T(0), s->stream));
    }
  if (s->nl == 2)
    for (int f = 0; f < 6; ++f) {
      CK(launch_fill<T>((T*)s->R[f], n, T(0), s->stream));
      CK(launch_fill<T>((T*)s->R1[f], n, T(0), s->stream));
    }
  CK(launch_fill<T>((T*)s->H, n, T(0), s->stream));
  return SWE_OK;
}

swe_status check_params(const swe_params* params) {
  if (params->precision != 32 && params->precision != 64) return SWE_ERR_ARG;
  if (!finite_pos(params->g)) return SWE_ERR_ARG;
  if (!(params->cfl > 0.0 && params->cfl <= 1.0)) return SWE_ERR_ARG;
  if (params->n_layers != 1 && params->n_layers != 2) return SWE_ERR_ARG;
  if (params->n_layers == 1 && params->pollutant != 1) return SWE_ERR_UNSUPPORTED;
  if (params->entropy_fix != 0 && params->entropy_fix != 1) return SWE_ERR_ARG;
  if (params->wet_dry != 0 && params->wet_dry != 1) return SWE_ERR_ARG;
  if (params->wet_dry == 1) {
    if (!(isfinite(params->h_dry) && params->h_dry >= 0.0)) return SWE_ERR_ARG;
    if (params->n_layers != 1) return SWE_ERR_UNSUPPORTED;
  }
  if (params->n_layers == 2) {
    if (params->pollutant != 0) return SWE_ERR_UNSUPPORTED;
    if (!(params->r >= 0.0 && params->r < 1.0)) return SWE_ERR_ARG;
  }
  return SWE_OK;
}

void init_common(swe_state* s, const swe_params* params) {
  s->p = *params;
  s->prec = params->precision;
  s->nl = params->n_layers;
  s->nf = s->nl == 2 ? 6 : 4;
  s->esz = s->prec == 32 ? 4 : 8;
  s->stream = (cudaStream_t)params->stream;
}

// Carve the slots, dt history, clock and error word from p; pinned readback.
swe_status carve_aux(swe_state* s, char* p) {
  s->slots = p;
  p += 256;
  s->dt_hist = (double*)p;
  p += round_up((int64_t)kHistCap * 8, 256);
  s->t_dev = (double*)p;
  p += 256;
  s->err = (unsigned*)p;
  cudaError_t e = cudaMallocHost(&s->h_dt, 64);
  if (e != cudaSuccess) {
    s->h_dt = nullptr;
    return cuda_status(e);
  }
  s->h_err = (unsigned*)(s->h_dt + 1);
  s->h_t = s->h_dt + 2;
  return SWE_OK;
}
constexpr int64_t kAuxBytes = 256 + ((int64_t)kHistCap * 8 + 255) / 256 * 256 + 256 + 256;

// Synchronous copy of a double host array to the device as T.
template <typename T>
swe_status put_as(void* dst, const std::vector<double>& src) {
  if (sizeof(T) == sizeof(double)) {
    CK(cudaMemcpy(dst, src.data(), src.size() * sizeof(double), cudaMemcpyHostToDevice));
    return SWE_OK;
  }
  std::vector<T> tmp(src.begin(), src.end());
  CK(cudaMemcpy(dst, tmp.data(), tmp.size() * sizeof(T), cudaMemcpyHostToDevice));
  return SWE_OK;
}

constexpr int64_t kMaxMeshCells = (int64_t)1 << 28;

}  // namespace

extern "C" {

const char* swe_status_str(swe_status st) {
  switch (st) {
    case SWE_OK: return "ok";
    case SWE_ERR_ARG: return "invalid argument";
    case SWE_ERR_CUDA: return "CUDA runtime error";
    case SWE_ERR_OOM: return "out of device memory";
    case SWE_ERR_DEPTH: return "a depth h <= 0 appeared";
    case SWE_ERR_NONFINITE: return "a non-finite value appeared";
    case SWE_ERR_HYPERBOLIC: return "loss of hyperbolicity";
    case SWE_ERR_UNSUPPORTED: return "not supported by this build";
    case SWE_ERR_TIMEOUT: return "a bounded device wait gave up";
  }
  return "unknown status";
}

swe_status swe_selftest_wait(int64_t budget_cycles) {
  if (budget_cycles < 1 || budget_cycles > 4000000000LL) return SWE_ERR_ARG;
  unsigned* err = nullptr;
  cudaError_t e = cudaMalloc(&err, sizeof(unsigned));
  if (e != cudaSuccess) return cuda_status(e);
  unsigned bits = 0;
  e = cudaMemset(err, 0, sizeof(unsigned));
  if (e == cudaSuccess) e = launch_wait_selftest((long long)budget_cycles, err, nullptr);
  if (e == cudaSuccess) e = cudaMemcpy(&bits, err, sizeof(unsigned), cudaMemcpyDeviceToHost);
  cudaFree(err);
  if (e != cudaSuccess) return cuda_status(e);
  return status_of_bits(bits);
}

void swe_destroy(swe_state* s) {
  if (!s) return;
  if (s->stream || s->dev) cudaStreamSynchronize(s->stream);
  timing_destroy(s->timing);
  if (s->dev) cudaFree(s->dev);
  if (s->h_dt) cudaFreeHost(s->h_dt);
  delete s;
}

swe_status swe_create_grid(const swe_grid* grid, const void* H, const void* const* W0,
                           const swe_params* params, swe_state** out) {
  if (!out) return SWE_ERR_ARG;
  *out = nullptr;
  if (!grid || !H || !W0 || !params) return SWE_ERR_ARG;
  const int nfields = params->n_layers == 2 ? 6 : 4;
  for (int f = 0; f < nfields; ++f)
    if (!W0[f]) return SWE_ERR_ARG;
  if (grid->nx < 1 || grid->ny < 1) return SWE_ERR_ARG;
  if (!finite_pos(grid->dx) || !finite_pos(grid->dy)) return SWE_ERR_ARG;
  {
    const swe_status pst = check_params(params);
    if (pst != SWE_OK) return pst;
  }
  // index arithmetic inside the kernels is 32-bit per row and column
  if ((int64_t)grid->nx > (1 << 30) || (int64_t)grid->ny > (1 << 30) - 8) return SWE_ERR_ARG;
  // wet/dry: one block per 8 rows in the launch's y dimension
  if (params->wet_dry == 1 && ((int64_t)grid->ny + 7) / 8 > 65535) return SWE_ERR_ARG;

  swe_state* s = new (std::nothrow) swe_state();
  if (!s) return SWE_ERR_OOM;
  s->nx = grid->nx;
  s->ny = grid->ny;
  s->dx = grid->dx;
  s->dy = grid->dy;
  init_common(s, params);
  if (s->nl == 1) {
    s->pitch = (int)(s->prec == 32 ? grid_pitch<float>(s->nx) : grid_pitch<double>(s->nx));
    s->rows = s->ny + 2 * kPadY;
  } else {
    s->pitch = (int)(s->prec == 32 ? grid_pitch2<float>(s->nx) : grid_pitch2<double>(s->nx));
    s->rows = s->prec == 32 ? grid_rows2<float>(s->ny) : grid_rows2<double>(s->ny);
  }

  swe_status st = SWE_OK;
  auto fail = [&](swe_status e) {
    swe_destroy(s);
    return e;
  };
  const int64_t felems = s->rows * s->pitch;
  const int64_t fbytes = round_up(felems * (int64_t)s->esz, 256);
  s->field_stride = fbytes / (int64_t)s->esz;
  const int64_t aux = kAuxBytes;
  // two buffers of the fields (+ two of the residual for two layers) + H
  const int nalloc = s->nl == 2 ? 25 : 9;
  s->wd = params->wet_dry == 1;
  s->dev_bytes = (size_t)(nalloc * fbytes + aux);
  cudaError_t e = cudaMalloc(&s->dev, s->dev_bytes);
  if (e != cudaSuccess) {
    s->dev = nullptr;
    return fail(cuda_status(e));
  }
  char* p = (char*)s->dev;
  if (s->nl == 1) {
    for (int b = 0; b < 2; ++b)
      for (int f = 0; f < 4; ++f) {
        s->w[b][f] = p;
        p += fbytes;
      }
  } else {
    for (int b = 0; b < 2; ++b)
      for (int f = 0; f < 6; ++f) {
        s->w[b][f] = p;
        p += fbytes;
      }
    for (int f = 0; f < 6; ++f) {
      s->R[f] = p;
      p += fbytes;
    }
    for (int f = 0; f < 6; ++f) {
      s->R1[f] = p;
      p += fbytes;
    }
  }
  s->H = p;
  p += fbytes;
  if ((st = carve_aux(s, p)) != SWE_OK) return fail(st);

  if (s->nl == 1) st = s->prec == 32 ? plan_launch<float>(s) : plan_launch<double>(s);
  else st = s->prec == 32 ? plan_launch2<float>(s) : plan_launch2<double>(s);
  if (st != SWE_OK) return fail(st);
  if (s->wd && (e = s->prec == 32 ? wd_prepare<float>() : wd_prepare<double>()) != cudaSuccess)
    return fail(cuda_status(e));
  st = s->prec == 32 ? fill_pads<float>(s) : fill_pads<double>(s);
  if (st != SWE_OK) return fail(st);
  void* hdst[1] = {s->H};
  const void* hsrc[1] = {H};
  if ((st = upload(s, hdst, hsrc, 1)) != SWE_OK) return fail(st);
  if ((st = upload(s, s->w[0], W0, s->nf)) != SWE_OK) return fail(st);
  if ((e = cudaMemsetAsync(s->t_dev, 0, 256 + 256, s->stream)) != cudaSuccess)
    return fail(cuda_status(e));
  s->cur = 0;
  s->step = 0;
  if ((st = enqueue_dt0_any(s)) != SWE_OK) return fail(st);
  if ((st = read_err(s)) != SWE_OK) return fail(st);
  if (s->sticky) return fail(SWE_ERR_ARG);
  *out = s;
  return SWE_OK;
}

swe_status swe_create_mesh(const swe_mesh* mesh, const void* H, const void* const* W0,
                           const swe_params* params, swe_state** out) {
  if (!out) return SWE_ERR_ARG;
  *out = nullptr;
  if (!mesh || !H || !W0 || !params) return SWE_ERR_ARG;
  {
    const swe_status pst = check_params(params);
    if (pst != SWE_OK) return pst;
  }
  if (params->wet_dry) return SWE_ERR_UNSUPPORTED;
  const int nfields = params->n_layers == 2 ? 6 : 4;
  for (int f = 0; f < nfields; ++f)
    if (!W0[f]) return SWE_ERR_ARG;
  if (!mesh->xy || !mesh->tri || mesh->n_vertices < 3 || mesh->n_cells < 1) return SWE_ERR_ARG;
  if (mesh->n_vertices > INT32_MAX || mesh->n_cells > kMaxMeshCells) return SWE_ERR_ARG;
  if (mesh->reorder != 0 && mesh->reorder != 1) return SWE_ERR_ARG;

  MeshPrep prep;
  const int rc = prepare_mesh(mesh->n_vertices, mesh->xy, mesh->n_cells, mesh->tri,
                              mesh->reorder == 1, &prep);
  if (rc == -3) return SWE_ERR_OOM;
  if (rc == -2) return SWE_ERR_UNSUPPORTED;
  if (rc != 0) return SWE_ERR_ARG;

  swe_state* s = new (std::nothrow) swe_state();
  if (!s) return SWE_ERR_OOM;
  auto fail = [&](swe_status e) {
    swe_destroy(s);
    return e;
  };
  init_common(s, params);
  s->mesh = true;
  s->ncells = prep.ncells;
  s->nedges = prep.nedges;
  s->nx = (int)prep.ncells;
  s->ny = 1;
  try {
    s->h_new_of_old = prep.new_of_old;
  } catch (const std::bad_alloc&) {
    return fail(SWE_ERR_OOM);
  }
  s->ntiles = prep.ntiles;
  const int64_t nc = s->ncells, esz = (int64_t)s->esz;
  const int64_t nt1 = prep.ntiles + 1, nhalo = (int64_t)prep.halo.size();
  const int64_t nsl = (int64_t)prep.slot_ab.size();
  const int64_t fb = round_up(nc * esz, 256), ib = round_up(nc * 4, 256);
  const int64_t tb = round_up(nt1 * 4, 256), hb = round_up(nhalo * 4 + 4, 256);
  const int64_t sib = round_up(nsl * 4, 256), stb = round_up(nsl * esz, 256);
  const int64_t cb = round_up(nc * 8, 256);
  s->field_stride = fb / esz;
  s->dev_bytes = (size_t)((2 * s->nf + 2) * fb + 2 * ib + 3 * tb + hb + sib + 3 * stb + cb +
                          kAuxBytes);
  cudaError_t e = cudaMalloc(&s->dev, s->dev_bytes);
  if (e != cudaSuccess) {
    s->dev = nullptr;
    return fail(cuda_status(e));
  }
  char* p = (char*)s->dev;
  auto take = [&](int64_t bytes) {
    void* q = p;
    p += bytes;
    return q;
  };
  for (int f = 0; f < s->nf; ++f) s->w[0][f] = take(fb);
  for (int f = 0; f < s->nf; ++f) s->R[f] = take(fb);
  s->H = take(fb);
  s->inv_area = take(fb);
  s->new_of_old = (int32_t*)take(ib);
  s->old_of_new = (int32_t*)take(ib);
  s->tile_cell = take(tb);
  s->tile_halo = take(tb);
  s->tile_slot = take(tb);
  s->halo = take(hb);
  s->slot_ab = take(sib);
  s->slot_nx = take(stb);
  s->slot_ny = take(stb);
  s->slot_len = take(stb);
  s->cref = take(cb);
  swe_status st;
  if ((st = carve_aux(s, p)) != SWE_OK) return fail(st);
  e = s->prec == 32 ? mesh_prepare<float>(s->nl, s->p.entropy_fix, s->ntiles, &s->mesh_grid)
                     : mesh_prepare<double>(s->nl, s->p.entropy_fix, s->ntiles, &s->mesh_grid);
  if (e != cudaSuccess) return fail(cuda_status(e));

  // geometry, tiles and orderings (synchronous copies from the temporary arrays)
  auto put_raw = [&](void* dst, const void* src, int64_t bytes) {
    if (bytes == 0) return SWE_OK;
    return cuda_status(cudaMemcpy(dst, src, (size_t)bytes, cudaMemcpyHostToDevice));
  };
  if ((st = put_raw(s->new_of_old, prep.new_of_old.data(), nc * 4)) != SWE_OK) return fail(st);
  if ((st = put_raw(s->old_of_new, prep.old_of_new.data(), nc * 4)) != SWE_OK) return fail(st);
  if ((st = put_raw(s->tile_cell, prep.tile_cell.data(), nt1 * 4)) != SWE_OK) return fail(st);
  if ((st = put_raw(s->tile_halo, prep.tile_halo.data(), nt1 * 4)) != SWE_OK) return fail(st);
  if ((st = put_raw(s->tile_slot, prep.tile_slot.data(), nt1 * 4)) != SWE_OK) return fail(st);
  if ((st = put_raw(s->halo, prep.halo.data(), nhalo * 4)) != SWE_OK) return fail(st);
  if ((st = put_raw(s->slot_ab, prep.slot_ab.data(), nsl * 4)) != SWE_OK) return fail(st);
  if ((st = put_raw(s->cref, prep.cref.data(), nc * 8)) != SWE_OK) return fail(st);
  try {
    void* dsts[4] = {s->slot_nx, s->slot_ny, s->slot_len, s->inv_area};
    const std::vector<double>* srcs[4] = {&prep.slot_nx, &prep.slot_ny, &prep.slot_len,
                                          &prep.inv_area};
    for (int k = 0; k < 4; ++k) {
      st = s->prec == 32 ? put_as<float>(dsts[k], *srcs[k]) : put_as<double>(dsts[k], *srcs[k]);
      if (st != SWE_OK) return fail(st);
    }
  } catch (const std::bad_alloc&) {
    return fail(SWE_ERR_OOM);
  }
  // H and the initial state, caller numbering -> internal order
  void* hdst[1] = {s->H};
  const void* hsrc[1] = {H};
  if ((st = mesh_upload(s, hdst, hsrc, 1)) != SWE_OK) return fail(st);
  if ((st = mesh_upload(s, s->w[0], W0, s->nf)) != SWE_OK) return fail(st);
  if ((e = cudaMemsetAsync(s->t_dev, 0, 256 + 256, s->stream)) != cudaSuccess)
    return fail(cuda_status(e));
  s->cur = 0;
  s->step = 0;
  if ((st = enqueue_dt0_any(s)) != SWE_OK) return fail(st);
  if ((st = read_err(s)) != SWE_OK) return fail(st);
  if (s->sticky) return fail(SWE_ERR_ARG);
  *out = s;
  return SWE_OK;
}

swe_status swe_mesh_info(const swe_mesh* mesh, int32_t* new_of_old, int64_t* n_edges,
                         int64_t* n_tiles, int64_t* n_edge_evals, int64_t* n_halo) {
  if (!mesh || !mesh->xy || !mesh->tri || mesh->n_vertices < 3 || mesh->n_cells < 1)
    return SWE_ERR_ARG;
  if (mesh->n_vertices > INT32_MAX || mesh->n_cells > kMaxMeshCells) return SWE_ERR_ARG;
  if (mesh->reorder != 0 && mesh->reorder != 1) return SWE_ERR_ARG;
  MeshPrep prep;
  const int rc = prepare_mesh(mesh->n_vertices, mesh->xy, mesh->n_cells, mesh->tri,
                              mesh->reorder == 1, &prep);
  if (rc == -3) return SWE_ERR_OOM;
  if (rc == -2) return SWE_ERR_UNSUPPORTED;
  if (rc != 0) return SWE_ERR_ARG;
  if (new_of_old)
    memcpy(new_of_old, prep.new_of_old.data(), (size_t)prep.ncells * sizeof(int32_t));
  if (n_edges) *n_edges = prep.nedges;
  if (n_tiles) *n_tiles = prep.ntiles;
  if (n_edge_evals) *n_edge_evals = prep.edge_evals;
  if (n_halo) *n_halo = (int64_t)prep.halo.size();
  return SWE_OK;
}

swe_status swe_set_timing(swe_state* s, int32_t on) {
  if (!s || (on != 0 && on != 1)) return SWE_ERR_ARG;
  if (!on) {
    if (!s->timing) return SWE_OK;
    const swe_status st = timing_harvest_all(s);
    s->timing->on = false;
    return st;
  }
  if (!s->timing) {
    Timing* tm = new (std::nothrow) Timing();
    if (!tm) return SWE_ERR_OOM;
    for (int i = 0; i < Timing::kSlots; ++i)
      for (int k = 0; k <= Timing::kMaxK; ++k) {
        const cudaError_t e = cudaEventCreate(&tm->ev[i][k]);
        if (e != cudaSuccess) {
          tm->ev[i][k] = nullptr;
          timing_destroy(tm);
          return cuda_status(e);
        }
      }
    s->timing = tm;
  }
  Timing* tm = s->timing;
  const swe_status st = timing_harvest_all(s);
  if (st != SWE_OK) return st;
  timing_names(s, tm);
  for (int k = 0; k < Timing::kMaxK; ++k) {
    tm->ms[k] = 0.0;
    tm->launches[k] = 0;
  }
  tm->on = true;
  return SWE_OK;
}

swe_status swe_get_timing(const swe_state* cs, swe_kernel_time* out, int32_t max, int32_t* n) {
  swe_state* s = const_cast<swe_state*>(cs);
  if (!s || !n || max < 0 || (max > 0 && !out)) return SWE_ERR_ARG;
  *n = 0;
  if (!s->timing) return SWE_OK;
  const swe_status st = timing_harvest_all(s);
  if (st != SWE_OK) return st;
  const Timing* tm = s->timing;
  const int cnt = tm->nk < max ? tm->nk : max;
  for (int k = 0; k < cnt; ++k) {
    memset(out[k].name, 0, sizeof(out[k].name));
    strncpy(out[k].name, tm->names[k], sizeof(out[k].name) - 1);
    out[k].launches = tm->launches[k];
    out[k].ms = tm->ms[k];
  }
  *n = cnt;
  return SWE_OK;
}

swe_status swe_cell_index(const swe_state* s, int64_t* idx) {
  if (!s || !idx) return SWE_ERR_ARG;
  if (s->mesh) {
    for (int64_t c = 0; c < s->ncells; ++c) idx[c] = s->h_new_of_old[c];
    return SWE_OK;
  }
  for (int64_t j = 0; j < s->ny; ++j)
    for (int64_t i = 0; i < s->nx; ++i)
      idx[j * s->nx + i] = (j + kPadY) * s->pitch + i + kPadX;
  return SWE_OK;
}

swe_status swe_set_state(swe_state* s, const void* const* fields, double t) {
  if (!s || !fields) return SWE_ERR_ARG;
  for (int f = 0; f < s->nf; ++f)
    if (!fields[f]) return SWE_ERR_ARG;
  if (!isfinite(t)) return SWE_ERR_ARG;
  swe_status st;
  if (s->mesh) st = mesh_upload(s, s->w[0], fields, s->nf);
  else st = upload(s, s->w[s->cur], fields, s->nf);
  if (st != SWE_OK) return st;
  *s->h_t = t;
  CK(cudaMemcpyAsync(s->t_dev, s->h_t, sizeof(double), cudaMemcpyHostToDevice, s->stream));
  CK(cudaMemsetAsync(s->err, 0, sizeof(unsigned), s->stream));
  s->step = 0;
  s->sticky = 0;
  if ((st = enqueue_dt0_any(s)) != SWE_OK) return st;
  if ((st = read_err(s)) != SWE_OK) return st;
  if (s->sticky) {
    // keep the state usable for another set_state, but refuse to step it
    return SWE_ERR_ARG;
  }
  return SWE_OK;
}

swe_status swe_step(swe_state* s, double cfl, double* dt_out) {
  if (!s) return SWE_ERR_ARG;
  if (!(cfl > 0.0 && cfl <= 1.0)) return SWE_ERR_ARG;
  if (s->sticky) return status_of_bits(s->sticky);
  swe_status st = enqueue_step_any(s, cfl, true);
  if (st != SWE_OK) {
    s->lazy2 = -1;
    return st;
  }
  CK(cudaMemcpyAsync(s->h_dt, s->dt_hist + ((s->step - 1) % kHistCap), sizeof(double),
                     cudaMemcpyDeviceToHost, s->stream));
  if ((st = read_err(s)) != SWE_OK) return st;
  if (dt_out) *dt_out = *s->h_dt;
  return status_of_bits(s->sticky);
}

swe_status swe_run(swe_state* s, int64_t nsteps) {
  if (!s || nsteps < 0) return SWE_ERR_ARG;
  if (s->sticky) return status_of_bits(s->sticky);
  for (int64_t n = 0; n < nsteps; ++n) {
    swe_status st = enqueue_step_any(s, s->p.cfl, n == nsteps - 1);
    if (st != SWE_OK) {
      s->lazy2 = -1;  // a failed launch leaves the state undefined
      return st;
    }
  }
  swe_status st = read_err(s);
  if (st != SWE_OK) return st;
  return status_of_bits(s->sticky);
}

swe_status swe_get_state(const swe_state* cs, void* const* fields_out, double* t_out) {
  swe_state* s = const_cast<swe_state*>(cs);
  if (!s || !fields_out) return SWE_ERR_ARG;
  for (int f = 0; f < s->nf; ++f)
    if (!fields_out[f]) return SWE_ERR_ARG;
  if (s->mesh) {
    swe_status st = mesh_download(s, fields_out);
    if (st != SWE_OK) return st;
  } else {
    const size_t row = (size_t)s->nx * s->esz;
    const size_t spitch = (size_t)s->pitch * s->esz;
    const size_t off = ((size_t)kPadY * s->pitch + kPadX) * s->esz;
    for (int f = 0; f < s->nf; ++f)
      CK(cudaMemcpy2DAsync(fields_out[f], row, (const char*)s->w[s->cur][f] + off, spitch, row,
                           (size_t)s->ny, cudaMemcpyDeviceToHost, s->stream));
  }
  CK(cudaMemcpyAsync(s->h_t, s->t_dev, sizeof(double), cudaMemcpyDeviceToHost, s->stream));
  CK(cudaStreamSynchronize(s->stream));
  if (t_out) *t_out = *s->h_t;
  return SWE_OK;
}

swe_status swe_get_dt_history(const swe_state* cs, double* dts, int64_t max, int64_t* n) {
  swe_state* s = const_cast<swe_state*>(cs);
  if (!s || !n || max < 0 || (max > 0 && !dts)) return SWE_ERR_ARG;
  int64_t have = s->step < kHistCap ? s->step : kHistCap;
  int64_t cnt = have < max ? have : max;
  // the cnt most recent entries, oldest first
  int64_t first = s->step - cnt;
  int64_t done = 0;
  while (done < cnt) {
    int64_t idx = (first + done) % kHistCap;
    int64_t run = kHistCap - idx;
    if (run > cnt - done) run = cnt - done;
    CK(cudaMemcpyAsync(dts + done, s->dt_hist + idx, (size_t)run * sizeof(double),
                       cudaMemcpyDeviceToHost, s->stream));
    done += run;
  }
  CK(cudaStreamSynchronize(s->stream));
  *n = cnt;
  return SWE_OK;
}

swe_status swe_get_info(const swe_state* s, swe_info* info) {
  if (!s || !info) return SWE_ERR_ARG;
  swe_state* m = const_cast<swe_state*>(s);
  CK(cudaMemcpyAsync(m->h_t, m->t_dev, sizeof(double), cudaMemcpyDeviceToHost, m->stream));
  CK(cudaStreamSynchronize(m->stream));
  info->steps = s->step;
  info->t = *m->h_t;
  info->nx = s->nx;
  info->ny = s->ny;
  info->precision = s->prec;
  info->pitch = s->pitch;
  info->field_offset = (int64_t)kPadY * s->pitch + kPadX;
  info->device_bytes = (int64_t)s->dev_bytes;
  info->bands = s->nbands;
  info->segments = s->nsegs;
  info->warps_per_block = kWarpsPerBlock;
  info->n_layers = s->nl;
  if (s->mesh) {
    info->pitch = 0;
    info->field_offset = 0;
    info->n_cells = s->ncells;
    info->n_edges = s->nedges;
    info->mesh = 1;
    info->bands = (int32_t)s->ntiles;
    info->segments = s->mesh_grid;
    info->warps_per_block = mesh_tile_warps(s->prec, s->nl, s->p.entropy_fix);
  } else {
    info->n_cells = (int64_t)s->nx * s->ny;
    info->n_edges = (int64_t)(s->nx + 1) * s->ny + (int64_t)s->nx * (s->ny + 1);
    info->mesh = 0;
  }
  return SWE_OK;
}

swe_status swe_device_fields(swe_state* s, void** ptrs) {
  if (!s || !ptrs) return SWE_ERR_ARG;
  for (int f = 0; f < s->nf; ++f) ptrs[f] = s->w[s->cur][f];
  ptrs[s->nf] = s->H;
  return SWE_OK;
}

}  // extern "C"
