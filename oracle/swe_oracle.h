/*
 * swe_oracle.h -- plain fp64 CPU oracle of the IR-Roe finite-volume step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this code; only the tests, the package smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header or constant with the CUDA
 * path.
 *
 * What it computes: An MPI-CUDA implementation of an improved Roe method for
 * two-layer shallow water systems (de la Asuncion, Mantas, Castro,
 * Fernandez-Nieto), Sec. 2.2: the update of eq. (4) with the numerical flux
 * of steps 1-4 and the time step of the CFL condition eq. (5), restricted to
 * one layer, plus a passive pollutant transported as in A multi-GPU
 * shallow-water simulation with transport of contaminants (Vinas et al.),
 * abstract.  The mesh is a generic polygon mesh: every cell lists its edges
 * (neighbour, outward unit normal, length); a neighbour of -1 is a reflective
 * wall.  Everything is fp64 and single threaded.
 */
#ifndef SWE_ORACLE_H
#define SWE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Polygon mesh in compressed per-cell edge lists.  Cell i owns the edge
 * entries e in [edge_start[i], edge_start[i+1]); nbr[e] is the neighbour
 * cell j (or -1 for a wall), (eta_x[e], eta_y[e]) the unit normal of the
 * common edge pointing from i towards j, and len[e] its length |Gamma_ij|.
 * area[i] is |V_i|.  An interior edge appears twice, once from each side. */
typedef struct {
  int64_t n_cells;
  const double *area;
  const int64_t *edge_start;
  const int64_t *nbr;
  const double *eta_x;
  const double *eta_y;
  const double *len;
} om_mesh;

/* status codes */
#define OM_OK 0
#define OM_ERR_DEPTH (-4)     /* a depth h <= 0 appeared */
#define OM_ERR_NONFINITE (-5) /* a non-finite value appeared */
#define OM_ERR_ARG (-1)
#define OM_ERR_HYPERBOLIC (-6) /* the Roe matrix has complex eigenvalues */

/* Number of edge entries of the nx x ny Cartesian grid as a polygon mesh. */
int64_t om_grid_edges(int64_t nx, int64_t ny);

/* Fill the polygon-mesh arrays of the nx x ny Cartesian grid with spacing
 * (dx, dy).  Cell (i, j) is index j*nx + i; its edges are listed East,
 * North, West, South. */
void om_grid_mesh(int64_t nx, int64_t ny, double dx, double dy, double *area,
                  int64_t *edge_start, int64_t *nbr, double *eta_x,
                  double *eta_y, double *len);

/* Polygon-mesh arrays of a triangle mesh: n_vertices points xy (2 per
 * vertex) and n_cells triangles tri (3 vertex indices each, counter-
 * clockwise).  Cell c lists its edges in the order (v0 v1), (v1 v2),
 * (v2 v0); the neighbour across an edge is the other triangle sharing both
 * vertices (-1 on the boundary: a wall), the normal is the outward unit
 * normal of the edge, the length its length; area is the shoelace area.
 * Returns OM_OK, or OM_ERR_ARG for a vertex index out of range, a triangle
 * that is not counter-clockwise, or an edge shared by more than two
 * triangles.  The arrays must hold 3 * n_cells edge entries. */
int om_tri_mesh(int64_t n_vertices, const double *xy, int64_t n_cells,
                const int32_t *tri, double *area, int64_t *edge_start,
                int64_t *nbr, double *eta_x, double *eta_y, double *len);

/* Numerical flux F_ij^- of eq. (4) (one layer + pollutant) for the state
 * Wi = (h, qx, qy, hC) of cell i, Wj of cell j, bathymetry Hi, Hj and unit
 * normal (ex, ey) from i to j.  Writes the Cartesian flux F[4] and the
 * spectral radius ||D_ij||_inf of the Roe matrix. */
void om_flux1(const double *Wi, const double *Wj, double Hi, double Hj,
              double ex, double ey, double g, double *F, double *Dinf);

/* Mirror ghost state of a reflective wall with outward normal (ex, ey). */
void om_wall_ghost1(const double *Wi, double ex, double ey, double *Wg);

/* Switch the Harten-Hyman entropy fix of the flux on (1) or off (0, the
 * default) for every later call, one layer or two. */
void om_set_entropy_fix(int on);

/* Switch the wet/dry treatment of the one-layer scheme on (1, with depth
 * threshold h_dry >= 0: a cell with h <= h_dry is dry) or off (0, the
 * default) for every later call: dry cells carry no velocity, a dry cell
 * whose bed is at or above its wet neighbour's surface is a wall, and each
 * edge is scaled by the draining ratio of the cell its mass flux leaves, so
 * that depths stay >= 0 (see swe_oracle.c for the two published sources).
 * With it on, h = 0 is a valid state. */
void om_set_wet_dry(int on, double h_dry);

/* Time step of eq. (5): min_i 2 cfl |V_i| / sum_j |Gamma_ij| ||D_ij||_inf.
 * W holds the four fields h, qx, qy, hC as separate arrays (W[0..3]). */
double om_dt1(const om_mesh *m, const double *const *W, const double *H,
              double g, double cfl);

/* One explicit step of eq. (4) with the given dt, in place.  work must hold
 * 4 * n_cells doubles.  Returns OM_OK or an error code. */
int om_update1(const om_mesh *m, double *const *W, const double *H, double g,
               double dt, double *work);

/* The updated state after one step of size dt, at the listed cells only
 * (out[k*n_sel + s] is field k of cell cells[s]); W is left unchanged. */
void om_update1_at(const om_mesh *m, const double *const *W, const double *H,
                   double g, double dt, const int64_t *cells, int64_t n_sel,
                   double *out);

/* nsteps steps: dt from eq. (5) on the current state, then eq. (4).  The dt
 * of each step is written to dts (may be NULL).  Returns OM_OK or the error
 * of the first failing step; *steps_done counts completed steps. */
int om_run1(const om_mesh *m, double *const *W, const double *H, double g,
            double cfl, int64_t nsteps, double *dts, double *work,
            int64_t *steps_done);

/* The same three operations on the nx x ny Cartesian grid (cell (i, j) is
 * index j*nx + i, edges East, North, West, South) without storing a mesh:
 * each cell's edges are generated on the fly exactly as om_grid_mesh lists
 * them.  For grids too large to hold as explicit meshes. */
double om_grid_dt1(int64_t nx, int64_t ny, double dx, double dy,
                   const double *const *W, const double *H, double g, double cfl);
int om_grid_update1(int64_t nx, int64_t ny, double dx, double dy, double *const *W,
                    const double *H, double g, double dt, double *work);
int om_grid_run1(int64_t nx, int64_t ny, double dx, double dy, double *const *W,
                 const double *H, double g, double cfl, int64_t nsteps, double *dts,
                 double *work, int64_t *steps_done);

/* ---- two layers: W = (h1, q1x, q1y, h2, q2x, q2y), 1 = upper layer,
 * r = rho1 / rho2 ([P1] Sec. 2.1 eq. (1)) ---------------------------------- */

/* Mirror ghost of both layers at a wall with outward normal (ex, ey). */
void om_wall_ghost2(const double *Wi, double ex, double ey, double *Wg);

/* Real eigenvalues, ascending, of the 2-layer Roe matrix A_ij with averaged
 * normal velocities u1, u2 and c1s = g hbar1, c2s = g hbar2: the roots of
 * ((l - u1)^2 - c1s)((l - u2)^2 - c2s) - r c1s c2s.  Returns OM_OK or
 * OM_ERR_HYPERBOLIC when the inner pair is complex. */
int om_roots2(double u1, double u2, double c1s, double c2s, double r, double *lam);

/* F_ij^- of eq. (4) for two layers (six Cartesian components) and
 * ||D_ij||_inf.  Returns OM_OK or OM_ERR_HYPERBOLIC. */
int om_flux2(const double *Wi, const double *Wj, double Hi, double Hj,
             double ex, double ey, double g, double r, double *F, double *Dinf);

/* eq. (5), eq. (4) and the time loop for two layers on a mesh or on the
 * implicit nx x ny grid; W holds six field arrays.  dt2 reports a loss of
 * hyperbolicity through *status (may be NULL). */
double om_dt2(const om_mesh *m, const double *const *W, const double *H,
              double g, double r, double cfl, int *status);
int om_update2(const om_mesh *m, double *const *W, const double *H, double g,
               double r, double dt, double *work);
/* The update of eq. (4) of the listed cells only, from the state W (which is
 * not modified): out[c * n_sel + s] is field c of cells[s] after one step of
 * size dt.  Returns OM_ERR_HYPERBOLIC if an edge of a listed cell has a
 * complex pair of eigenvalues. */
int om_update2_at(const om_mesh *m, const double *const *W, const double *H, double g,
                  double r, double dt, const int64_t *cells, int64_t n_sel, double *out);
int om_run2(const om_mesh *m, double *const *W, const double *H, double g,
            double r, double cfl, int64_t nsteps, double *dts, double *work,
            int64_t *steps_done);
double om_grid_dt2(int64_t nx, int64_t ny, double dx, double dy,
                   const double *const *W, const double *H, double g, double r,
                   double cfl, int *status);
int om_grid_update2(int64_t nx, int64_t ny, double dx, double dy, double *const *W,
                    const double *H, double g, double r, double dt, double *work);
int om_grid_run2(int64_t nx, int64_t ny, double dx, double dy, double *const *W,
                 const double *H, double g, double r, double cfl, int64_t nsteps,
                 double *dts, double *work, int64_t *steps_done);

#ifdef __cplusplus
}
#endif
#endif
