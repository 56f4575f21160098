// swe_internal.h -- shared between the host side of libswe and its kernels.
//
// Device layout of a Cartesian state (one allocation per handle):
//   every field is a padded 2D array of (ny + 2*kPadY) rows of `pitch`
//   elements; logical cell (x, y) sits at element (y + kPadY) * pitch +
//   (x + kPadX).  The padding is never updated after creation: it only
//   keeps the fixed-width row windows the step kernel loads inside the
//   allocation.  Wall (mirror) states are formed in registers.
//   Column windows: the grid is cut into vertical bands of kOwn<T> owned
//   columns; band b loads the 32*kCpt<T> physical columns starting at
//   b*kOwn<T>, i.e. its owned columns plus two halo columns on each side.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

namespace swe {

constexpr int kPadX = 2;
constexpr int kPadY = 2;
constexpr int kHistCap = 65536;   // dt history ring length

// error bits written by the kernels into the sticky error word
constexpr unsigned kErrDepth = 1u;
constexpr unsigned kErrNonfinite = 2u;
constexpr unsigned kErrTimeout = 4u;
constexpr unsigned kErrHyperbolic = 8u;

// Every lane of the step kernel owns two adjacent cells of a row.
template <typename T> struct Cpt { static constexpr int v = 2; };

template <typename T> constexpr int cells_per_lane() { return Cpt<T>::v; }
template <typename T> constexpr int band_window() { return 32 * Cpt<T>::v; }
template <typename T> constexpr int band_owned() { return 32 * Cpt<T>::v - 4; }

// Pipeline depth (rows in flight per warp) and warps per block of the step.
#ifndef SWE_STAGES
#define SWE_STAGES 4
#endif
#ifndef SWE_WARPS_PER_BLOCK
#define SWE_WARPS_PER_BLOCK 4
#endif
constexpr int kStages = SWE_STAGES;
constexpr int kWarpsPerBlock = SWE_WARPS_PER_BLOCK;

// Row pitch (elements) for an nx-wide grid of element type T.
template <typename T>
inline int64_t grid_pitch(int nx) {
  int64_t own = band_owned<T>();
  int64_t nb = (nx + own - 1) / own;
  int64_t need = own * (nb - 1) + band_window<T>();
  return (need + 31) / 32 * 32;
}

template <typename T>
struct StepArgs {
  const T* win[4];      // W^n: h, qx, qy, hC (field bases, padded layout)
  T* wout[4];           // W^{n+1}
  const T* H;           // bottom depth (padded layout)
  int nx, ny, pitch;
  int nbands, nsegs;    // column bands; row segments per band
  int nsegs_wall;       // row segments of the first and the last band (>= nsegs)
  T ghalf;              // g / 2
  T rho;                // dx / dy (y-edge weight relative to x-edges)
  double two_cfl;       // 2 * cfl of this step
  double dx;
  const void* tmax_in;  // max over cells of sum D (this step), raw bits
  void* tmax_out;       // accumulated for the next step (must start at 0)
  void* tmax_clear;     // slot zeroed for the step after next
  double* dt_hist;      // dt ring
  double* t_dev;        // simulated time
  int64_t step;         // index of this step (selects the history slot)
  unsigned* err;        // sticky error bits
  int efix;             // 1: the Harten-Hyman entropy fix of the flux
};

// ---- two layers (swe_cart2.cu) ----------------------------------------------
// A warp marches over a band of kBand2 owned columns and reads one halo
// column on each side (lane l of band b: column kBand2 * b - 1 + l), so a
// row must hold 30 * ceil(nx / 30) + 1 columns past the padding; rows are
// padded to whole groups of Tile2Y<T> (the update kernel's blocks).
constexpr int kTile2X = 32;
constexpr int kBand2 = 30;
constexpr int kMarch2Warps = 4;
template <typename T> struct Tile2Y { static constexpr int v = 8; };
template <> struct Tile2Y<double> { static constexpr int v = 4; };

template <typename T>
inline int64_t grid_pitch2(int nx) {
  int64_t tiles = (int64_t)(nx + kTile2X - 1) / kTile2X * kTile2X;
  int64_t bands = (int64_t)(nx + kBand2 - 1) / kBand2 * kBand2 + 1;
  int64_t cols = (tiles > bands ? tiles : bands) + 2 * kPadX;
  return (cols + 31) / 32 * 32;
}
template <typename T>
inline int64_t grid_rows2(int ny) {
  return (int64_t)(ny + Tile2Y<T>::v - 1) / Tile2Y<T>::v * Tile2Y<T>::v + 2 * kPadY;
}

template <typename T>
struct Fields6 {
  const T* p[6];
};

template <typename T>
struct Step2Args {
  const T* w[6];   // h1, q1x, q1y, h2, q2x, q2y (padded layout)
  const T* H;
  T* R[6];         // residual sum_j L F / dx (scratch, padded layout)
  int nx, ny, pitch;
  T g, r, rho;     // gravity, density ratio, dx / dy
  void* tmax_out;  // max over cells of sum_x D + rho sum_y D (must start at 0)
  unsigned* err;
  int efix;        // 1: the Harten-Hyman entropy fix
  int nbands, nsegs;  // launch shape: one warp per (band, row segment)
};
// The update W_out = W_in - (dt/dx) R of step `step`, dt from the wave-speed
// maximum in tmax_in.  cart2_update_kernel reads win and writes w (the same
// buffer, or buffer 0 at the end of a run); the fused march writes the
// updated cells it owns to w.
template <typename T>
struct Update2Args {
  const T* win[6];
  T* w[6];
  const T* R[6];
  int nx, ny, pitch;
  double two_cfl, dx;
  const void* tmax_in;
  void* tmax_clear;
  void* tmax_clear2;  // a second slot to zero, or null
  double* dt_hist;
  double* t_dev;
  int64_t step;
  unsigned* err;
};

// Resident four-warp blocks per SM of the march (efix: the entropy-fix variant).
template <typename T>
cudaError_t march2_occupancy(int* blocks_per_sm, bool efix);
template <typename T>
cudaError_t launch_flux2(const Step2Args<T>& f, cudaStream_t st);
template <typename T>
cudaError_t launch_fused2(const Step2Args<T>& f, const Update2Args<T>& u, cudaStream_t st);
template <typename T>
cudaError_t launch_update2(const Update2Args<T>& u, cudaStream_t st);
template <typename T>
cudaError_t launch_check2(const Fields6<T>& w6, int nx, int ny, int pitch, unsigned* err,
                          cudaStream_t st);

// ---- triangle meshes (swe_mesh.cu, swe_mesh_prep.cpp) ------------------------
// A mesh state keeps its cells in an internal order (the Hilbert curve through
// the cell centroids unless the caller asked for its own), one contiguous
// array per field, and cuts that order into tiles: consecutive cells, each
// tile with at most kTileSlots edge slots, kTileCells cells, kTileHalo halo
// cells and kTileCap cells plus halo cells.  A tile's edge slots are the edges with at least one cell in
// the tile: an edge inside a tile has one slot, an edge between two tiles
// one slot in each (the two evaluate it identically).  Every edge keeps one
// orientation: cells a < b (b a wall on the mesh boundary) and the unit
// normal (nx, ny) pointing from a to b, length L.
//
// Per slot (tile-major, each tile's range starts at an even index):
//   slot_ab  tile-local index of a | tile-local index of b << 16 (0xffff: wall);
//            local indices 0 .. nct-1 are the tile's cells, nct .. the halo
//   slot_nx, slot_ny, slot_len
// Per cell: cref = its three edges in the order of its vertices (edge k
// joins vertex k and vertex k + 1) as slot | side << 15 (side 1: the cell
// is b), packed 16 bits each into (x: edges 0, 1; y: edge 2).
//
// In shared memory the tile kernel keeps, per slot, what each side adds to
// its residual, already multiplied by L and rotated back to x / y:
//   two layers  [0] m1  [1] m2           mass fluxes a -> b (a adds, b subtracts)
//               [2..5] a: (x, y) momentum of layer 1, then of layer 2
//               [6..9] b: the same for b
//               [10] L * max |lambda|
//   one layer   [0] m  [1] m C_upwind    mass and pollutant fluxes a -> b
//               [2, 3] a: (x, y) momentum   [4, 5] b: (x, y) momentum
//               [6] L * max |lambda|
constexpr int kTileSlots = 512;
constexpr int kTileCap = 640;
constexpr int kTileHalo = 256;
constexpr int kTileCells = 512;
constexpr int kTileWall = 0xffff;
template <int NL> struct MeshLayout;
template <> struct MeshLayout<1> {
  static constexpr int nf = 4, ne = 7, a_mom = 2, b_mom = 4, d = 6;
};
template <> struct MeshLayout<2> {
  static constexpr int nf = 6, ne = 11, a_mom = 2, b_mom = 6, d = 10;
};

template <typename T>
struct MeshStepArgs {
  const T* w[6];              // state, internal cell order
  const T* H;
  T* R[6];                    // residual / area (scratch)
  const int32_t* tile_cell;   // [ntiles + 1]: first cell of each tile
  const int32_t* tile_halo;   // [ntiles + 1]: first entry of each tile in halo
  const int32_t* tile_slot;   // [ntiles + 1]: first slot of each tile
  const int32_t* halo;        // halo cells (internal index), tile by tile
  const int32_t* slot_ab;
  const T* slot_nx;           // unit normal from a to b
  const T* slot_ny;
  const T* slot_len;          // edge length
  const uint2* cref;          // [ncells]
  const T* inv_area;          // 1 / |V_i|
  int64_t ncells, ntiles;
  int grid;                   // blocks of the tile kernel (mesh_prepare)
  T g, r;
  void* tmax_out;             // max over cells of sum L max|lambda| / |V_i| (starts at 0)
  unsigned* err;
  int efix;                   // 1: the Harten-Hyman entropy fix
};
template <typename T>
struct MeshUpdateArgs {
  T* w[6];
  const T* R[6];
  int64_t ncells;
  double two_cfl;
  const void* tmax_in;
  void* tmax_clear;
  double* dt_hist;
  double* t_dev;
  int64_t step;
  unsigned* err;
};

// Sets the shared-memory limit of the tile kernel a mesh state of this
// kind runs on the current device and returns its grid: one block per
// resident slot (the kernel is persistent), at most ntiles.
template <typename T>
cudaError_t mesh_prepare(int n_layers, int efix, int64_t ntiles, int* grid);
// warps per block of that tile kernel
int mesh_tile_warps(int precision, int n_layers, int efix);
template <typename T>
cudaError_t launch_mesh_step(const MeshStepArgs<T>& f, const MeshUpdateArgs<T>& u, int n_layers,
                             cudaStream_t st, const cudaEvent_t* marks = nullptr);
template <typename T>
cudaError_t launch_mesh_check(const Fields6<T>& w, int n_layers, int64_t ncells, unsigned* err,
                              cudaStream_t st);
// dst[f][i] = src[f][idx[i]] for f < nf, i < n
template <typename T>
cudaError_t launch_mesh_permute(T* const* dst, const T* const* src, int nf, const int32_t* idx,
                                int64_t n, cudaStream_t st);

// Host preparation of a triangle mesh (swe_mesh_prep.cpp): geometry in
// double precision, edges, cell order, tiles and the per-cell slot references.
struct MeshPrep {
  int64_t ncells = 0, nedges = 0, ntiles = 0;
  std::vector<int32_t> ea, eb;            // [nedges], internal order, a < b (b = -1: wall)
  std::vector<double> enx, eny, elen;     // [nedges]
  std::vector<int32_t> ref;               // [3 * ncells]: 2 * edge + side of edge k of cell c at k * ncells + c
  std::vector<double> inv_area;           // [ncells], internal order
  std::vector<int32_t> new_of_old;        // caller cell -> internal cell
  std::vector<int32_t> old_of_new;        // internal cell -> caller cell
  std::vector<int32_t> tile_cell, tile_halo, tile_slot;  // [ntiles + 1]
  std::vector<int32_t> halo;
  std::vector<int32_t> slot_ab;
  std::vector<double> slot_nx, slot_ny, slot_len;
  std::vector<uint32_t> cref;             // [2 * ncells]
  int64_t edge_evals = 0;                 // slots without the even padding
};
// 0 on success; -1 for an invalid mesh (index out of range, non-finite
// coordinate, clockwise or degenerate triangle, an edge used by more than two
// triangles or twice in the same direction); -2 if the tiles failed their
// consistency check (not expected for any valid mesh); -3 when host memory
// runs out.
int prepare_mesh(int64_t n_vertices, const double* xy, int64_t n_cells, const int32_t* tri,
                 bool reorder, MeshPrep* out);

// ---- one layer with wet/dry fronts on a grid (swe_wetdry.cu) ----------------
// State in the one-layer padded layout, W^n in win, W^{n+1} written to wout;
// per step a speed pass (sum of L ||D|| reduced into tmax_slot) and a tile
// pass (edges, draining times, update), which reads tmax_slot and zeroes
// tmax_clear.
struct WdStepArgs {
  void* win[4];
  void* wout[4];
  const void* H;
  int nx, ny, pitch;
  double g, h_dry, dx, dy;
  double two_cfl;
  void* tmax_slot;
  void* tmax_clear;
  double* dt_hist;
  double* t_dev;
  int64_t step;
  unsigned* err;
  int efix;
};
// Launch attributes of the wet/dry kernels on the current device (once per
// handle, before the first step).
template <typename T>
cudaError_t wd_prepare();
template <typename T>
cudaError_t launch_wd_step(const WdStepArgs& a, cudaStream_t st, const cudaEvent_t* marks);
template <typename T>
cudaError_t launch_wd_check(const T* const* w, int nx, int ny, int pitch, unsigned* err,
                            cudaStream_t st);

// Programmatic dependent launch: consecutive step kernels on a stream are
// launched with programmatic stream serialisation, so the next kernel's
// launch overlaps the end of the previous one.  Each such kernel waits
// (griddepcontrol.wait: until the previous grid has completed and its memory
// is visible) before it reads anything, and lets its dependent launch once
// its own main work is issued.
#ifndef SWE_PDL
#define SWE_PDL 1
#endif
__device__ __forceinline__ void pdl_wait() {
#if SWE_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}
__device__ __forceinline__ void pdl_trigger() {
#if SWE_PDL
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = SWE_PDL;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// The multi-kernel launchers take an optional array of events: when given,
// marks[k] is recorded on the stream before kernel k and marks[nk] after the
// last one (per-kernel device time, swe_set_timing).

// host-side launchers (swe_cart1.cu)
template <typename T>
cudaError_t launch_step(const StepArgs<T>& a, int blocks, cudaStream_t st);
template <typename T>
cudaError_t launch_dt0(const T* const* w, const T* H, int nx, int ny, int pitch,
                       T ghalf, T rho, void* tmax_out, unsigned* err,
                       cudaStream_t st);
template <typename T>
cudaError_t launch_fill(T* base, int64_t count, T value, cudaStream_t st);
// One warp running the step kernel's bounded mbarrier wait on a barrier
// nothing arrives on; sets kErrTimeout in *err when the wait gives up.
cudaError_t launch_wait_selftest(long long budget_cycles, unsigned* err, cudaStream_t st);
// Resident blocks per SM of the one-layer step kernel (efix: the variant
// with the entropy fix) and its dynamic shared memory; sets its attributes.
template <typename T>
cudaError_t step_occupancy(int* blocks_per_sm, size_t* smem_bytes, bool efix = false);

}  // namespace swe
