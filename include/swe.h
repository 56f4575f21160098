/*
 * swe.h -- C ABI of the GB300 shallow-water finite-volume library (libswe).
 *
 * The library advances the 2D shallow-water equations with the first-order,
 * path-conservative Roe-type ("IR-Roe") finite-volume scheme of
 *
 *   [P1] de la Asuncion, Mantas, Castro, Fernandez-Nieto, "An MPI-CUDA
 *        implementation of an improved Roe method for two-layer shallow
 *        water systems": Sec. 2.1 (model, eq. (1); rotation invariance,
 *        eq. (2)-(3)), Sec. 2.2 (update eq. (4), numerical flux steps 1-4,
 *        CFL condition eq. (5)), Sec. 3 and Algorithm 1 (time loop: edge
 *        fluxes, per-volume dt, global minimum, volume update);
 *   [P2] Vinas et al., "A multi-GPU shallow-water simulation with transport
 *        of contaminants": abstract (one layer + a pollutant carried by a
 *        transport equation) and Figure 4 (each edge's flux computed once per
 *        tile and shared between its two cells).
 *
 * One explicit step, for every cell V_i with neighbours j:
 *     W_i^{n+1} = W_i^n - dt_n / |V_i| * sum_j |Gamma_ij| F_ij^-      (eq. (4))
 *     dt_n = min_i 2 cfl |V_i| / sum_j |Gamma_ij| ||D_ij||_inf          (eq. (5))
 * with W = (h, qx, qy, hC): depth, discharge and pollutant mass per area, or,
 * for the two-layer system of [P1] eq. (1), W = (h1, q1x, q1y, h2, q2x, q2y)
 * (layer 1 on top, r = rho1/rho2 < 1) with the 4x4 Roe matrix of [P1]
 * Sec. 2.2.
 * H is the depth of the bottom below a fixed reference level (positive
 * downward, [P1] Sec. 2.1), so the free surface is h - H.  Domain boundaries
 * are reflective walls (mirror ghost: same h, hC, H; normal discharge
 * negated).  dt_n is reduced on the device from the state W^n; the host never
 * sits between two steps unless it asks for dt.
 *
 * Conventions of every call:
 *  - Every function returns a swe_status; nothing aborts or prints.
 *  - Host arrays are in the caller's memory, owned by the caller, and copied
 *    during the call.  Their element type is the state's precision: float
 *    when swe_params.precision == 32, double when it is 64.
 *  - Grid fields are nx*ny values, cell (i, j) at index j*nx + i (row-major,
 *    x fastest), centre ((i+1/2) dx, (j+1/2) dy).  Mesh fields are n_cells
 *    values, triangle c at index c of the caller's numbering (the library
 *    may reorder cells internally; every host array in and out of it is in
 *    the caller's numbering).
 *  - Field order: h, qx, qy, hC (one layer); h1, q1x, q1y, h2, q2x, q2y (two).
 *  - A handle is not thread-safe; it may be used from any one thread at a
 *    time.  All device work of a handle is ordered on swe_params.stream.
 *  - Device-detected errors (SWE_ERR_DEPTH, SWE_ERR_NONFINITE,
 *    SWE_ERR_HYPERBOLIC, SWE_ERR_TIMEOUT) are sticky: every later swe_step /
 *    swe_run returns them until swe_set_state installs a new state.  The handle stays valid and
 *    destroyable after any error.
 */
#ifndef SWE_H
#define SWE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SWE_OK = 0,
  SWE_ERR_ARG = -1,         /* invalid argument (NULL, size, parameter)     */
  SWE_ERR_CUDA = -2,        /* a CUDA runtime call failed                   */
  SWE_ERR_OOM = -3,         /* device memory exhausted                      */
  SWE_ERR_DEPTH = -4,       /* a depth h <= 0 appeared (h < 0 with wet_dry) */
  SWE_ERR_NONFINITE = -5,   /* a non-finite value appeared in the state     */
  SWE_ERR_HYPERBOLIC = -6,  /* the two-layer Roe matrix lost hyperbolicity  */
  SWE_ERR_UNSUPPORTED = -7, /* valid request this build does not implement  */
  SWE_ERR_TIMEOUT = -8      /* a bounded device wait gave up                */
} swe_status;

/* Cartesian grid of nx x ny rectangular cells of size dx x dy, walls on all
 * four sides ([P1] Sec. 2.2 volumes V_i with |V_i| = dx dy; edges of length
 * dy (normal (1, 0)) and dx (normal (0, 1))). */
typedef struct {
  int32_t nx, ny;
  double dx, dy;
} swe_grid;

/* Unstructured mesh of triangles ([P1] Sec. 2.2: finite volumes V_i, here
 * triangles; the edge Gamma_ij shared by V_i and V_j has length |Gamma_ij|
 * and the unit normal eta_ij pointing from V_i to V_j; an edge of a single
 * triangle is a reflective wall).
 *  n_vertices  >= 3
 *  xy          host, 2*n_vertices doubles: vertex v at (xy[2v], xy[2v+1])
 *  n_cells     1 <= n_cells <= 2^28: number of triangles
 *  tri         host, 3*n_cells int32: the vertices of triangle c at
 *              tri[3c], tri[3c+1], tri[3c+2], counter-clockwise
 *  reorder     1: store the cells in the order of the Hilbert curve through
 *              their centroids, so that runs of consecutive cells (the
 *              tiles of a step, see swe_create_mesh) are compact patches;
 *              0: keep the caller's order (still correct, but tiles of cells
 *              far apart evaluate more edges twice and load more halo
 *              cells).  Results are in the caller's numbering either way. */
typedef struct {
  int64_t n_vertices;
  const double *xy;
  int64_t n_cells;
  const int32_t *tri;
  int32_t reorder;
} swe_mesh;

/* Model and run parameters.
 *  n_layers   1, or 2 for the two-layer system of [P1] eq. (1)
 *  precision  32 or 64: arithmetic and storage type of the state
 *  pollutant  1 with one layer (the state carries hC, [P2] transport
 *             equation); 0 with two layers (no pollutant there)
 *  g          gravity (> 0)
 *  r          density ratio rho1/rho2, 0 <= r < 1, two layers; ignored for 1
 *  cfl        gamma of eq. (5), 0 < cfl <= 1, used by swe_run
 *  stream     cudaStream_t the handle orders its work on; NULL = legacy
 *             default stream
 *  entropy_fix  0: P^- of [P1] Sec. 2.2 as printed; 1: the Harten-Hyman
 *             entropy fix that [P1] Sec. 2.2 (after eq. (5)) names for
 *             sonic rarefactions.  Per characteristic speed lambda_k of the
 *             Roe matrix, delta_k = max(0, lambda_k - lambda_k(W_i),
 *             lambda_k(W_j) - lambda_k), lambda_k(W) the k-th eigenvalue of
 *             the Jacobian of the side's own state (u_eta -+ sqrt(g h) for
 *             one layer; the k-th root of the same quartic with the side's
 *             own velocities and depths for two); where |lambda_k| <
 *             delta_k the scheme uses (lambda_k^2 + delta_k^2) / (2 delta_k)
 *             in place of |lambda_k|, i.e. Phi^- gains
 *             (|lambda_k| - |lambda_k|_d) beta_k K_k / 2 with beta = K^-1
 *             (W_j - W_i).  Two layers: a side state whose own system is
 *             not hyperbolic is reported as SWE_ERR_HYPERBOLIC.  Any value
 *             other than 0 or 1 returns SWE_ERR_ARG.
 *  wet_dry    0: every depth must stay > 0 (h <= 0 is SWE_ERR_DEPTH), the
 *             scheme as printed; 1 (one layer on a grid only, else
 *             SWE_ERR_UNSUPPORTED): wet/dry fronts, which [P1] leaves open,
 *             by two published techniques.  A cell with h <= h_dry is dry
 *             and carries no velocity or concentration; an edge between two
 *             dry cells passes nothing; an edge between a wet cell and a dry
 *             cell whose bed (-H) is at or above the wet free surface (h - H)
 *             is a reflective wall for both (Brufau, Vazquez-Cendon and
 *             Garcia-Navarro, Int. J. Numer. Meth. Fluids 39, 2002); every
 *             term of an edge is scaled by min(1, tau_d / dt), tau_d = h_d
 *             |V_d| / (the mass that leaves cell d per unit time) of the cell
 *             its mass flux leaves, so no depth turns negative (the draining
 *             time of Bollermann, Chen, Kurganov and Noelle, J. Sci. Comput.
 *             56, 2013).  After each step a depth below zero (rounding) is
 *             clamped to 0 and a dry cell's discharge is set to 0.  h = 0
 *             is then a valid input; dt stays eq. (5).  Runs as two
 *             kernels per step (wave speeds; a tile pass of edges, draining
 *             times and update) instead of the fused step.  Any value other
 *             than 0 or 1 returns SWE_ERR_ARG.
 *  h_dry      with wet_dry = 1: the depth at or below which a cell is dry,
 *             >= 0 and finite.  It must exceed the thin-film scale of the
 *             problem: a film just above h_dry next to deep water receives
 *             the deep side's pressure and can be driven to unphysical
 *             speeds, which collapses dt.  In the oracle, water at rest
 *             around emerging hills needed 1e-4 m (1e-6 m: km/s); a column
 *             of water flooding up a slope needed 1e-2 m (1e-4 m: 130 m/s,
 *             dt down 440-fold).  Ignored when wet_dry = 0. */
typedef struct {
  int32_t n_layers;
  int32_t precision;
  int32_t pollutant;
  double g;
  double r;
  double cfl;
  void *stream;
  int32_t entropy_fix;
  int32_t wet_dry;
  double h_dry;
} swe_params;

typedef struct swe_state swe_state;

/* Create a simulation on a Cartesian grid ([P1] Algorithm 1, before the time
 * loop: mesh construction and initial state).
 *  grid    grid size and spacing; nx, ny >= 1, dx, dy > 0 and finite;
 *          nx <= 2^30, ny <= 2^30 - 8; with wet_dry also ny <= 524280
 *          (65535 blocks of 8 rows)
 *  H       host, nx*ny values: bottom depth below the reference level
 *  W0      host, array of 4 pointers (h, qx, qy, hC), or 6 (h1, q1x, q1y,
 *          h2, q2x, q2y) for two layers, nx*ny values each; depths > 0
 *  params  see swe_params
 *  out     receives the handle (NULL on failure)
 * Allocates the device state (9 padded fields of the chosen precision for one
 * layer: two buffers of the 4 fields and H; 25 for two: two buffers of the 6
 * fields and of their residuals, and H), copies H and W0 to the device and
 * checks the state there (one layer: also dt_0).
 * Errors: SWE_ERR_ARG (bad argument, h <= 0 or non-finite input),
 * SWE_ERR_UNSUPPORTED, SWE_ERR_OOM, SWE_ERR_CUDA. */
swe_status swe_create_grid(const swe_grid *grid, const void *H,
                           const void *const *W0, const swe_params *params,
                           swe_state **out);

/* Create a simulation on a triangle mesh ([P1] Algorithm 1, before the time
 * loop; the mesh of [P1] Sec. 2.2).
 *  mesh    see swe_mesh
 *  H, W0   host, n_cells values per field in the caller's numbering, with
 *          the field order and precision of swe_create_grid
 *  params  see swe_params
 *  out     receives the handle (NULL on failure)
 * Computes on the host, in double precision, every triangle's area and every
 * edge's length and unit normal, pairs the triangles across their shared
 * edges, orders the cells (swe_mesh.reorder) and cuts that order into tiles:
 * runs of consecutive cells with at most 512 edges touching them, 512 cells,
 * 256 neighbouring (halo) cells and 640 cells and halo cells together.  Then
 * allocates the device state and copies the geometry, H and W0 there.  Each
 * step runs two kernels ([P1] Algorithm 1, edge processing then volume
 * processing): the tile kernel stages each tile's cells and halo in shared
 * memory, evaluates the Roe flux of each of its edges once and sums every
 * cell's three edges in a fixed order (an edge between two tiles is
 * evaluated by both, identically), then the update.  The device keeps about
 * (2 nf + 2) values and 4 int32 per cell, 3 values and 1 int32 per edge
 * evaluation, 1 int32 per halo entry.
 * Errors: SWE_ERR_ARG (bad argument; an index out of range, a non-finite
 * coordinate, a clockwise or degenerate triangle, an edge traversed twice in
 * the same direction -- which includes any edge of three or more triangles;
 * h <= 0 or non-finite input), SWE_ERR_UNSUPPORTED (also if the tiles fail
 * the consistency check run on every preparation, which no valid mesh is
 * expected to), SWE_ERR_OOM, SWE_ERR_CUDA. */
swe_status swe_create_mesh(const swe_mesh *mesh, const void *H,
                           const void *const *W0, const swe_params *params,
                           swe_state **out);

/* Host-only preview of the preparation swe_create_mesh does (no device
 * work): checks the mesh and reports, for each caller cell, its internal
 * index (new_of_old, n_cells int32, may be NULL), the number of edges walls
 * included (*n_edges), the number of tiles (*n_tiles), the flux evaluations
 * per step (*n_edge_evals: n_edges plus one for every edge shared by two
 * tiles) and the halo cells loaded per step (*n_halo); each output may be
 * NULL.  Errors: SWE_ERR_ARG as for swe_create_mesh, SWE_ERR_OOM. */
swe_status swe_mesh_info(const swe_mesh *mesh, int32_t *new_of_old,
                         int64_t *n_edges, int64_t *n_tiles,
                         int64_t *n_edge_evals, int64_t *n_halo);

/* Advance one step of eq. (4) with dt_n from eq. (5) evaluated on the
 * current state with CFL number cfl (0 < cfl <= 1).  Waits for the step to
 * finish; *dt_out (if not NULL) receives dt_n.  Returns the sticky device
 * error, if any, after the step (two layers: SWE_ERR_HYPERBOLIC when an
 * edge's Roe matrix has complex eigenvalues). */
swe_status swe_step(swe_state *s, double cfl, double *dt_out);

/* Advance nsteps >= 0 steps with params.cfl: the time loop of [P1]
 * Algorithm 1 (per step: edge fluxes, per-volume dt of eq. (5) and its
 * minimum, the update of eq. (4), the clock), with the minimum taken on the
 * device.  Enqueues all steps on the
 * handle's stream without host synchronisation, then waits once and reports
 * the sticky device error.  On a two-layer grid the update of each step is
 * applied inside the next step's flux pass (and the last one by a separate
 * pass); the result equals nsteps calls of swe_step bit for bit. */
swe_status swe_run(swe_state *s, int64_t nsteps);

/* Copy the current state to the host.  fields_out: array of 4 host pointers
 * (h, qx, qy, hC), or 6 for two layers, of nx*ny elements of the state's
 * precision; t_out (may be
 * NULL) receives the simulated time (sum of the dt of all steps since the
 * last swe_create_grid / swe_set_state, plus the t given there). */
swe_status swe_get_state(const swe_state *s, void *const *fields_out,
                         double *t_out);

/* Replace the state (a restart), set the simulated time to t, clear the
 * sticky error and recompute dt on the device.  Same layout as
 * swe_get_state.  Errors: SWE_ERR_ARG for h <= 0 or non-finite input. */
swe_status swe_set_state(swe_state *s, const void *const *fields, double t);

/* dt of the most recent steps, oldest first: up to max values are written
 * to dts (host) and *n receives the count written.  The library keeps the
 * last 65536 steps. */
swe_status swe_get_dt_history(const swe_state *s, double *dts, int64_t max,
                              int64_t *n);

/* Information about a handle. */
typedef struct {
  int64_t steps;        /* steps taken since create / set_state            */
  double t;             /* simulated time                                  */
  int32_t nx, ny;
  int32_t precision;
  int32_t pitch;        /* elements between rows of a device field         */
  int64_t field_offset; /* elements from a field's base to cell (0, 0)     */
  int64_t device_bytes; /* device memory held by the handle                */
  int32_t bands, segments, warps_per_block; /* launch shape: one layer on */
                        /* a grid: column bands, row segments per band and */
                        /* warps per block of the step kernel; a mesh:     */
                        /* tiles, blocks and warps per block of the tile   */
                        /* kernel                                          */
  int32_t n_layers;
  int64_t n_cells;      /* nx*ny, or the mesh's triangles                  */
  int64_t n_edges;      /* edges, walls included                           */
  int32_t mesh;         /* 1 for a triangle mesh (nx = n_cells, ny = 1,     */
                        /* pitch = field_offset = 0), 0 for a grid         */
} swe_info;
swe_status swe_get_info(const swe_state *s, swe_info *info);

/* Device pointers of the current state's fields followed by H (5 pointers
 * for one layer: h, qx, qy, hC, H; 7 for two), for zero-copy inspection on
 * the device; ptrs must hold that many entries.  Cell (i, j) of field k is at
 * ptrs[k] + field_offset + j*pitch + i (see swe_info); on a mesh, cell c is
 * at ptrs[k] + idx[c] with idx from swe_cell_index.  The pointers stay owned
 * by the handle; a one-layer grid's change after every step (double
 * buffering), the others' stay fixed. */
swe_status swe_device_fields(swe_state *s, void **ptrs);

/* idx (host, n_cells int64 values, see swe_info) receives, for every cell in
 * the caller's numbering, the element index of that cell within each device
 * field of swe_device_fields. */
swe_status swe_cell_index(const swe_state *s, int64_t *idx);

/* Per-kernel device time.  swe_set_timing(s, 1) starts (or restarts, from
 * zero) accounting: every step enqueued afterwards records CUDA events on the
 * handle's stream before, between and after its kernels, and the elapsed
 * times are summed per kernel; while on, swe_run keeps at most 64 steps in
 * flight ahead of the host.  swe_set_timing(s, 0) stops it (the sums stay).
 * swe_get_timing waits for the recorded steps and writes up to max entries
 * (one per kernel the handle's steps launch, in launch order: one for a
 * one-layer grid; flux pass, fused update-and-flux pass and update for a
 * two-layer grid; edge, gather and update passes for a mesh) to out; *n
 * receives the count.  Errors: SWE_ERR_ARG, SWE_ERR_OOM, SWE_ERR_CUDA. */
typedef struct {
  char name[32];     /* kernel name, NUL-terminated                        */
  int64_t launches;  /* launches timed                                      */
  double ms;         /* summed device time of those launches, milliseconds */
} swe_kernel_time;
swe_status swe_set_timing(swe_state *s, int32_t on);
swe_status swe_get_timing(const swe_state *s, swe_kernel_time *out, int32_t max,
                          int32_t *n);

/* Allocation-free time loop.  The papers have no counterpart of this entry
 * point: it exists for callers that must not allocate device memory after
 * start-up -- a framework whose memory pool already holds (nearly) all of the
 * GPU's memory, where cudaMalloc would fail or fragment it, and real-time or
 * embedded loops that forbid allocation because cudaMalloc can block and
 * synchronise the device.  It runs nsteps steps of the same kernels as
 * swe_run on buffers the caller owns, and allocates nothing: no cudaMalloc,
 * no cudaFree, no allocating library routine.
 *
 *  grid, params  as for swe_create_grid, one layer with pollutant only:
 *                n_layers = 2, pollutant != 1 or wet_dry != 0 gives
 *                SWE_ERR_UNSUPPORTED, any other n_layers than 1 or 2 gives
 *                SWE_ERR_ARG;
 *                params.cfl is used for every step, params.entropy_fix
 *                selects the step with the entropy fix, params.stream
 *                orders all work
 *  H             device, the bottom depth in the padded layout below
 *  W_a           4 device pointers (h, qx, qy, hC), padded layout: the state
 *                to advance on input, the state after nsteps steps on output
 *  W_b           4 device pointers, padded layout: work buffers (overwritten)
 *  pitch         elements per row of every field: a multiple of 32, at least
 *                32 * ceil((60 * ceil(nx / 60) + 4) / 32)
 *  nsteps        0 <= nsteps <= SWE_NOALLOC_MAX_STEPS
 *  dts_out       host, nsteps doubles (may be NULL): dt of each step
 * Padded layout: each field is (ny + 4) rows of `pitch` elements of the
 * precision's type, 16-byte aligned; cell (i, j) is element
 * (j + 2) * pitch + (i + 2).  The padding may hold anything; it is read but
 * never affects a result and never written.
 * The scratch (wave-speed maxima, error word, clock and the dt of at most
 * SWE_NOALLOC_MAX_STEPS steps, about 8.4 KB) is one static device array per
 * GPU, held until the process exits.  CUDA loads a library's device code
 * lazily, so that array is reserved on a device by the first call there,
 * which also looks up the array's device address and sets the step kernel's
 * launch attributes.  A caller whose pool will claim nearly all of a device's
 * memory should make that first call -- a call with nsteps = 0 does -- before
 * the pool does; it should also make it before any stream capture starts on
 * that device.  Every call clears the parts of the array that must start at
 * zero; all calls share the array, so calls that overlap on the GPU (other
 * streams, other threads) race and must be serialised.  The call waits for
 * its stream before returning.
 * Errors: SWE_ERR_ARG (bad argument, nsteps beyond SWE_NOALLOC_MAX_STEPS,
 * pitch too small, unaligned buffer); SWE_ERR_DEPTH / SWE_ERR_NONFINITE for
 * an invalid input state or one that appears (not sticky: nothing persists
 * between calls); SWE_ERR_TIMEOUT, SWE_ERR_CUDA. */
#define SWE_NOALLOC_MAX_STEPS 1024
swe_status swe_run_noalloc(const swe_grid *grid, const swe_params *params,
                           const void *H, void *const *W_a, void *const *W_b,
                           int32_t pitch, int64_t nsteps, double *dts_out);

/* Failure-detection self test of the step kernel's bounded device wait.
 * The one-layer step kernel waits on an mbarrier for each row staged into
 * shared memory; if the copy never lands, the wait gives up after a budget
 * of SM clock cycles (about two seconds in the step kernel) and the step
 * reports SWE_ERR_TIMEOUT instead of hanging.  This call runs that same
 * bounded wait, on the current device, in a one-warp kernel on a barrier that
 * nothing ever arrives on, with the given budget.
 *  budget_cycles  1 <= budget_cycles <= 4e9 (SM clock cycles)
 * Returns SWE_ERR_TIMEOUT when the wait gave up as designed (the expected
 * outcome; the CUDA context stays usable), SWE_OK if the barrier completed
 * (never expected), SWE_ERR_ARG, SWE_ERR_OOM or SWE_ERR_CUDA.  Allocates and
 * frees one word of device memory; synchronises the device. */
swe_status swe_selftest_wait(int64_t budget_cycles);

/* Release every resource of the handle.  NULL is accepted. */
void swe_destroy(swe_state *s);

/* Static English description of a status code. */
const char *swe_status_str(swe_status st);

#ifdef __cplusplus
}
#endif
#endif /* SWE_H */
