/*
 * swe_oracle.c -- plain fp64 CPU oracle of the IR-Roe finite-volume step.
 *
 * TEST INFRASTRUCTURE ONLY (see swe_oracle.h): only the tests, the package
 * smoke check and the bench's CPU-baseline leg may load it.
 *
 * Source of every formula: An MPI-CUDA implementation of an improved Roe
 * method for two-layer shallow water systems, Sec. 2.1 (model, eq. (1),
 * rotation invariance eq. (2)-(3)) and Sec. 2.2 (IR-Roe scheme: update
 * eq. (4), numerical flux steps 1-4, CFL condition eq. (5)), with the two
 * layers reduced to one; and A multi-GPU shallow-water simulation with
 * transport of contaminants, abstract (pollutant transport equation).
 *
 * The code follows the pages' order literally and makes no attempt at speed:
 * every cell evaluates F_ij^- for each of its edges from its own side (an
 * interior edge is therefore evaluated twice), builds the 2x2 Roe matrix,
 * its eigenvectors K, K^-1 and P^- = 1/2 K (I - sgn D) K^-1 explicitly, and
 * sums its edges' contributions.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - walls: a wall edge sees a mirror ghost (same h, hC and H, normal
 *    discharge negated, tangential discharge kept);
 *  - sgn(0) = 0;
 *  - pollutant: the transported concentration C = hC/h is upwinded with the
 *    mass flux exactly like the tangential velocity of step 3;
 *  - the time step uses the Roe eigenvalues of every edge, walls included;
 *  - a cell sums its edge terms pairwise in edge-list order.
 */
#include "swe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define OM_MAX_EDGES 16

int64_t om_grid_edges(int64_t nx, int64_t ny) { return 4 * nx * ny; }

/* The four edges of cell c of the nx x ny grid: East, North, West, South. */
static void grid_cell_edges(int64_t nx, int64_t ny, double dx, double dy, int64_t c,
                            int64_t nbr[4], double ex[4], double ey[4], double len[4]) {
  static const int di[4] = {1, 0, -1, 0};
  static const int dj[4] = {0, 1, 0, -1};
  int64_t i = c % nx, j = c / nx;
  for (int k = 0; k < 4; ++k) {
    int64_t ii = i + di[k], jj = j + dj[k];
    int inside = ii >= 0 && ii < nx && jj >= 0 && jj < ny;
    nbr[k] = inside ? jj * nx + ii : -1;
    ex[k] = (double)di[k];
    ey[k] = (double)dj[k];
    len[k] = (k == 0 || k == 2) ? dy : dx;
  }
}

void om_grid_mesh(int64_t nx, int64_t ny, double dx, double dy, double *area,
                  int64_t *edge_start, int64_t *nbr, double *eta_x,
                  double *eta_y, double *len) {
  for (int64_t c = 0; c < nx * ny; ++c) {
    area[c] = dx * dy;
    edge_start[c] = 4 * c;
    grid_cell_edges(nx, ny, dx, dy, c, nbr + 4 * c, eta_x + 4 * c, eta_y + 4 * c,
                    len + 4 * c);
  }
  edge_start[nx * ny] = 4 * nx * ny;
}

static double sgn(double x) { return (x > 0.0) ? 1.0 : ((x < 0.0) ? -1.0 : 0.0); }

void om_wall_ghost1(const double *Wi, double ex, double ey, double *Wg) {
  /* reflect the discharge about the wall: q - 2 (q . eta) eta */
  double qn = Wi[1] * ex + Wi[2] * ey;
  Wg[0] = Wi[0];
  Wg[1] = Wi[1] - 2.0 * qn * ex;
  Wg[2] = Wi[2] - 2.0 * qn * ey;
  Wg[3] = Wi[3];
}

/* Physical flux F_1 of the rotated 1D system (mass, normal momentum). */
static void flux_1d(double h, double qn, double g, double F[2]) {
  F[0] = qn;
  F[1] = qn * qn / h + 0.5 * g * h * h;
}

void om_flux1(const double *Wi, const double *Wj, double Hi, double Hj,
              double ex, double ey, double g, double *F, double *Dinf) {
  /* Step 1: W_eta = T_eta W.  R_eta maps (qx, qy) to
   * (q . eta, q . eta_perp) with eta_perp = (-ey, ex)  (eq. (2)). */
  double hi = Wi[0], hj = Wj[0];
  double qni = Wi[1] * ex + Wi[2] * ey;
  double qnj = Wj[1] * ex + Wj[2] * ey;
  double qti = -Wi[1] * ey + Wi[2] * ex;
  double qtj = -Wj[1] * ey + Wj[2] * ex;

  /* Step 2: Roe matrix of the 1D system.  Velocities are averaged with
   * sqrt(h) weights per Cartesian component, depths arithmetically. */
  double si = sqrt(hi), sj = sqrt(hj);
  double uxi = Wi[1] / hi, uyi = Wi[2] / hi;
  double uxj = Wj[1] / hj, uyj = Wj[2] / hj;
  double ux = (si * uxi + sj * uxj) / (si + sj);
  double uy = (si * uyi + sj * uyj) / (si + sj);
  double un = ux * ex + uy * ey;
  double hbar = 0.5 * (hi + hj);
  /* A_ij = [[0, 1], [g hbar - un^2, 2 un]]: eigenvalues un -+ sqrt(g hbar),
   * eigenvectors (1, lambda_k). */
  double c = sqrt(g * hbar);
  double lam[2] = {un - c, un + c};
  double K[2][2] = {{1.0, 1.0}, {lam[0], lam[1]}};
  double detK = K[0][0] * K[1][1] - K[0][1] * K[1][0];
  double Kinv[2][2] = {{K[1][1] / detK, -K[0][1] / detK},
                       {-K[1][0] / detK, K[0][0] / detK}};
  /* P^- = 1/2 K (I - sgn D) K^-1 */
  double w[2] = {0.5 * (1.0 - sgn(lam[0])), 0.5 * (1.0 - sgn(lam[1]))};
  double P[2][2];
  for (int r = 0; r < 2; ++r)
    for (int s = 0; s < 2; ++s)
      P[r][s] = K[r][0] * w[0] * Kinv[0][s] + K[r][1] * w[1] * Kinv[1][s];

  /* Fluctuation F_1(W_eta,j) - F_1(W_eta,i) - S_ij (H_j - H_i), with the
   * one-layer source S_ij = (0, g hbar) and no coupling term B. */
  double Fi[2], Fj[2];
  flux_1d(hi, qni, g, Fi);
  flux_1d(hj, qnj, g, Fj);
  double d[2] = {Fj[0] - Fi[0], Fj[1] - Fi[1] - g * hbar * (Hj - Hi)};
  /* Phi^- = P^- d + F_1(W_eta,i) */
  double phi[2];
  for (int r = 0; r < 2; ++r) phi[r] = P[r][0] * d[0] + P[r][1] * d[1] + Fi[r];

  /* Step 3: tangential discharge and pollutant as passive scalars carried
   * by the mass flux, upwinded on its sign. */
  double ut = (phi[0] > 0.0) ? qti / hi : qtj / hj;
  double Cs = (phi[0] > 0.0) ? Wi[3] / hi : Wj[3] / hj;
  double phit = phi[0] * ut;

  /* Step 4: back to Cartesian components with T_eta^-1. */
  F[0] = phi[0];
  F[1] = phi[1] * ex - phit * ey;
  F[2] = phi[1] * ey + phit * ex;
  F[3] = phi[0] * Cs;
  *Dinf = fmax(fabs(lam[0]), fabs(lam[1]));
}

/* pairwise sum of a[0..n) in list order */
static double psum(const double *a, int n) {
  if (n == 1) return a[0];
  if (n == 2) return a[0] + a[1];
  int h = n / 2;
  return psum(a, h) + psum(a + h, n - h);
}

static void cell_state(const double *const *W, int64_t i, double out[4]) {
  for (int k = 0; k < 4; ++k) out[k] = W[k][i];
}

/* A cell-edge source: an explicit polygon mesh, or the implicit Cartesian
 * grid (the same edges as om_grid_mesh, generated per cell). */
typedef struct {
  const om_mesh *m;
  int64_t nx, ny;
  double dx, dy;
} view;

static int64_t view_cells(const view *v) { return v->m ? v->m->n_cells : v->nx * v->ny; }
static double view_area(const view *v, int64_t i) { return v->m ? v->m->area[i] : v->dx * v->dy; }

static int view_edges(const view *v, int64_t i, int64_t nbr[OM_MAX_EDGES],
                      double ex[OM_MAX_EDGES], double ey[OM_MAX_EDGES],
                      double len[OM_MAX_EDGES]) {
  if (!v->m) {
    grid_cell_edges(v->nx, v->ny, v->dx, v->dy, i, nbr, ex, ey, len);
    return 4;
  }
  int64_t e0 = v->m->edge_start[i], e1 = v->m->edge_start[i + 1];
  int n = (int)(e1 - e0);
  if (n > OM_MAX_EDGES) n = OM_MAX_EDGES; /* meshes are checked by the caller */
  for (int k = 0; k < n; ++k) {
    nbr[k] = v->m->nbr[e0 + k];
    ex[k] = v->m->eta_x[e0 + k];
    ey[k] = v->m->eta_y[e0 + k];
    len[k] = v->m->len[e0 + k];
  }
  return n;
}

/* All edge terms of cell i: L_e F_e (4 components) and L_e ||D_e||. */
static int cell_terms(const view *v, const double *const *W, const double *H,
                      double g, int64_t i, double Fl[4][OM_MAX_EDGES],
                      double Dl[OM_MAX_EDGES]) {
  int64_t nbr[OM_MAX_EDGES];
  double exs[OM_MAX_EDGES], eys[OM_MAX_EDGES], lens[OM_MAX_EDGES];
  int n = view_edges(v, i, nbr, exs, eys, lens);
  double Wi[4], Wj[4];
  cell_state(W, i, Wi);
  for (int k = 0; k < n; ++k) {
    double ex = exs[k], ey = eys[k], L = lens[k];
    double Hj;
    if (nbr[k] >= 0) {
      cell_state(W, nbr[k], Wj);
      Hj = H[nbr[k]];
    } else {
      om_wall_ghost1(Wi, ex, ey, Wj);
      Hj = H[i];
    }
    double F[4], D;
    om_flux1(Wi, Wj, H[i], Hj, ex, ey, g, F, &D);
    for (int c = 0; c < 4; ++c) Fl[c][k] = L * F[c];
    Dl[k] = L * D;
  }
  return n;
}

static double dt_view(const view *v, const double *const *W, const double *H,
                      double g, double cfl) {
  double dt = INFINITY;
  double Fl[4][OM_MAX_EDGES], Dl[OM_MAX_EDGES];
  int64_t N = view_cells(v);
  for (int64_t i = 0; i < N; ++i) {
    int n = cell_terms(v, W, H, g, i, Fl, Dl);
    double s = psum(Dl, n);
    double dti = 2.0 * cfl * view_area(v, i) / s;
    if (isnan(dti)) return dti;
    if (dti < dt) dt = dti;
  }
  return dt;
}

static int check_state(const double w[4]) {
  for (int k = 0; k < 4; ++k)
    if (!isfinite(w[k])) return OM_ERR_NONFINITE;
  if (!(w[0] > 0.0)) return OM_ERR_DEPTH;
  return OM_OK;
}

static int update_view(const view *v, double *const *W, const double *H, double g,
                       double dt, double *work) {
  const double *const *Wc = (const double *const *)W;
  double Fl[4][OM_MAX_EDGES], Dl[OM_MAX_EDGES];
  int64_t N = view_cells(v);
  for (int64_t i = 0; i < N; ++i) {
    int n = cell_terms(v, Wc, H, g, i, Fl, Dl);
    for (int c = 0; c < 4; ++c)
      work[c * N + i] = W[c][i] - dt / view_area(v, i) * psum(Fl[c], n);
  }
  int status = OM_OK;
  for (int64_t i = 0; i < N; ++i) {
    double w[4];
    for (int c = 0; c < 4; ++c) {
      w[c] = work[c * N + i];
      W[c][i] = w[c];
    }
    int s = check_state(w);
    if (s != OM_OK && status == OM_OK) status = s;
  }
  return status;
}

static void update_at_view(const view *v, const double *const *W, const double *H,
                           double g, double dt, const int64_t *cells, int64_t n_sel,
                           double *out) {
  double Fl[4][OM_MAX_EDGES], Dl[OM_MAX_EDGES];
  for (int64_t s = 0; s < n_sel; ++s) {
    int64_t i = cells[s];
    int n = cell_terms(v, W, H, g, i, Fl, Dl);
    for (int c = 0; c < 4; ++c)
      out[c * n_sel + s] = W[c][i] - dt / view_area(v, i) * psum(Fl[c], n);
  }
}

static int run_view(const view *v, double *const *W, const double *H, double g,
                    double cfl, int64_t nsteps, double *dts, double *work,
                    int64_t *steps_done) {
  int64_t done = 0;
  int status = OM_OK;
  for (int64_t n = 0; n < nsteps; ++n) {
    double dt = dt_view(v, (const double *const *)W, H, g, cfl);
    if (dts) dts[n] = dt;
    if (!isfinite(dt) || !(dt > 0.0)) {
      status = OM_ERR_NONFINITE;
      break;
    }
    status = update_view(v, W, H, g, dt, work);
    ++done;
    if (status != OM_OK) break;
  }
  if (steps_done) *steps_done = done;
  return status;
}

static view mesh_view(const om_mesh *m) {
  view v = {m, 0, 0, 0.0, 0.0};
  return v;
}
static view grid_view(int64_t nx, int64_t ny, double dx, double dy) {
  view v = {0, nx, ny, dx, dy};
  return v;
}

double om_dt1(const om_mesh *m, const double *const *W, const double *H,
              double g, double cfl) {
  view v = mesh_view(m);
  return dt_view(&v, W, H, g, cfl);
}

int om_update1(const om_mesh *m, double *const *W, const double *H, double g,
               double dt, double *work) {
  view v = mesh_view(m);
  return update_view(&v, W, H, g, dt, work);
}

void om_update1_at(const om_mesh *m, const double *const *W, const double *H,
                   double g, double dt, const int64_t *cells, int64_t n_sel,
                   double *out) {
  view v = mesh_view(m);
  update_at_view(&v, W, H, g, dt, cells, n_sel, out);
}

int om_run1(const om_mesh *m, double *const *W, const double *H, double g,
            double cfl, int64_t nsteps, double *dts, double *work,
            int64_t *steps_done) {
  view v = mesh_view(m);
  return run_view(&v, W, H, g, cfl, nsteps, dts, work, steps_done);
}

double om_grid_dt1(int64_t nx, int64_t ny, double dx, double dy,
                   const double *const *W, const double *H, double g, double cfl) {
  view v = grid_view(nx, ny, dx, dy);
  return dt_view(&v, W, H, g, cfl);
}

int om_grid_update1(int64_t nx, int64_t ny, double dx, double dy, double *const *W,
                    const double *H, double g, double dt, double *work) {
  view v = grid_view(nx, ny, dx, dy);
  return update_view(&v, W, H, g, dt, work);
}

int om_grid_run1(int64_t nx, int64_t ny, double dx, double dy, double *const *W,
                 const double *H, double g, double cfl, int64_t nsteps, double *dts,
                 double *work, int64_t *steps_done) {
  view v = grid_view(nx, ny, dx, dy);
  return run_view(&v, W, H, g, cfl, nsteps, dts, work, steps_done);
}
