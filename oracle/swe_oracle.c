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

/* Optional entropy fix of the flux (off unless switched on; om_flux1 and
 * om_flux2, where lambda_k(W) is the k-th eigenvalue of the two-layer
 * Jacobian of the state W).
 * [P1] Sec. 2.2 remarks that an entropy fix of Harten-Hyman type can be
 * adapted to the scheme but gives no formula; this is the published one:
 * Harten's regularised absolute value |lambda|_d = |lambda| when
 * |lambda| >= delta, (lambda^2 + delta^2) / (2 delta) otherwise, with the
 * Harten-Hyman choice delta_k = max(0, lambda_k - lambda_k(W_i),
 * lambda_k(W_j) - lambda_k), lambda_k(W) being the eigenvalue of the
 * physical Jacobian of the state W itself (u_eta -/+ sqrt(g h)).  Adapted to
 * Phi^- = P^- d + F(W_i) as added numerical viscosity along each wave,
 * measured on the state jump: Phi^- += 1/2 (|lambda_k| - |lambda_k|_d)
 * beta_k K_k with beta = K^-1 (W_j - W_i).  With a flat bottom this is the
 * Roe fluctuation with |lambda| replaced by |lambda|_d; it vanishes wherever
 * |lambda_k| >= delta_k (so water at rest stays at rest). */
static int g_entropy_fix = 0;
void om_set_entropy_fix(int on) { g_entropy_fix = on ? 1 : 0; }

/* Optional wet/dry treatment (one layer; off unless switched on).  The
 * pages give none: they report depths bounded away from zero.  This is the
 * combination of two published techniques for explicit upwind finite-volume
 * schemes:
 *  - dry cells and wet/dry fronts as in Brufau, Vazquez-Cendon and
 *    Garcia-Navarro, "A numerical model for the flooding and drying of
 *    irregular domains" (Int. J. Numer. Meth. Fluids 39, 2002): a cell with
 *    h <= h_dry is dry and carries no velocity and no concentration; an edge
 *    between two dry cells passes nothing; an edge between a wet cell and a
 *    dry cell whose bed (-H) is at or above the wet cell's free surface
 *    (h - H) is a reflective wall for both (the wet side sees its mirror
 *    ghost over its own bed, so water at rest against an emerged bank stays
 *    at rest); any other wet/dry edge takes the Roe flux with the dry side's
 *    velocity and concentration zero;
 *  - positivity by the draining time of Bollermann, Chen, Kurganov and
 *    Noelle, "A well-balanced reconstruction of wet/dry fronts for the
 *    shallow water equations" (J. Sci. Comput. 56, 2013): a cell i whose
 *    edges carry mass out at the total rate M_i = sum_e L_e max(0, phi_e)
 *    empties in tau_i = h_i |V_i| / M_i; every term of an edge (mass,
 *    momentum, pollutant, both sides) is scaled by min(1, tau_d / dt), d the
 *    cell the edge's mass flux leaves, so no cell loses more water than it
 *    holds.
 * After the update a depth is clamped at 0 (rounding only) and a cell that
 * ended dry loses its discharge. */
static int g_wet_dry = 0;
static double g_h_dry = 0.0;
void om_set_wet_dry(int on, double h_dry) {
  g_wet_dry = on ? 1 : 0;
  g_h_dry = on ? h_dry : 0.0;
}
static int is_dry(double h) { return g_wet_dry && h <= g_h_dry; }

static double harten_abs(double lam, double lamL, double lamR) {
  double delta = fmax(0.0, fmax(lam - lamL, lamR - lam));
  double a = fabs(lam);
  return (a < delta) ? (lam * lam + delta * delta) / (2.0 * delta) : a;
}

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
  /* wet/dry (when switched on): two dry sides pass nothing; a dry side
   * whose bed is at or above the wet side's surface is a wall */
  int dry_i = is_dry(Wi[0]), dry_j = is_dry(Wj[0]);
  if (dry_i && dry_j) {
    F[0] = F[1] = F[2] = F[3] = 0.0;
    *Dinf = 0.0;
    return;
  }
  if ((dry_j && -Hj >= Wi[0] - Hi) || (dry_i && -Hi >= Wj[0] - Hj)) {
    if (dry_i) {
      F[0] = F[1] = F[2] = F[3] = 0.0;
      *Dinf = 0.0;
      return;
    }
    double Wg[4];
    om_wall_ghost1(Wi, ex, ey, Wg);
    om_flux1(Wi, Wg, Hi, Hi, ex, ey, g, F, Dinf);
    return;
  }
  /* Step 1: W_eta = T_eta W.  R_eta maps (qx, qy) to
   * (q . eta, q . eta_perp) with eta_perp = (-ey, ex)  (eq. (2)).  A dry
   * side carries no discharge. */
  double hi = Wi[0], hj = Wj[0];
  double qni = dry_i ? 0.0 : Wi[1] * ex + Wi[2] * ey;
  double qnj = dry_j ? 0.0 : Wj[1] * ex + Wj[2] * ey;
  double qti = dry_i ? 0.0 : -Wi[1] * ey + Wi[2] * ex;
  double qtj = dry_j ? 0.0 : -Wj[1] * ey + Wj[2] * ex;

  /* Step 2: Roe matrix of the 1D system.  Velocities are averaged with
   * sqrt(h) weights per Cartesian component, depths arithmetically. */
  double si = sqrt(hi), sj = sqrt(hj);
  double uxi = dry_i ? 0.0 : Wi[1] / hi, uyi = dry_i ? 0.0 : Wi[2] / hi;
  double uxj = dry_j ? 0.0 : Wj[1] / hj, uyj = dry_j ? 0.0 : Wj[2] / hj;
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
  if (dry_i) Fi[1] = 0.5 * g * hi * hi;  /* no q^2 / h on a dry side */
  if (dry_j) Fj[1] = 0.5 * g * hj * hj;
  double d[2] = {Fj[0] - Fi[0], Fj[1] - Fi[1] - g * hbar * (Hj - Hi)};
  /* Phi^- = P^- d + F_1(W_eta,i) */
  double phi[2];
  for (int r = 0; r < 2; ++r) phi[r] = P[r][0] * d[0] + P[r][1] * d[1] + Fi[r];
  if (g_entropy_fix) {
    /* the eigenvalues of each side's own Jacobian, u_eta -/+ sqrt(g h) */
    double uni = dry_i ? 0.0 : qni / hi, unj = dry_j ? 0.0 : qnj / hj;
    double ci = sqrt(g * hi), cj = sqrt(g * hj);
    double lamL[2] = {uni - ci, uni + ci}, lamR[2] = {unj - cj, unj + cj};
    double dW[2] = {hj - hi, qnj - qni};
    for (int k = 0; k < 2; ++k) {
      double beta = Kinv[k][0] * dW[0] + Kinv[k][1] * dW[1];
      double nu = 0.5 * (fabs(lam[k]) - harten_abs(lam[k], lamL[k], lamR[k])) * beta;
      for (int r = 0; r < 2; ++r) phi[r] += nu * K[r][k];
    }
  }

  /* Step 3: tangential discharge and pollutant as passive scalars carried
   * by the mass flux, upwinded on its sign. */
  double ut, Cs;
  if (phi[0] > 0.0) {
    ut = dry_i ? 0.0 : qti / hi;
    Cs = dry_i ? 0.0 : Wi[3] / hi;
  } else {
    ut = dry_j ? 0.0 : qtj / hj;
    Cs = dry_j ? 0.0 : Wj[3] / hj;
  }
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
  if (g_wet_dry ? !(w[0] >= 0.0) : !(w[0] > 0.0)) return OM_ERR_DEPTH;
  return OM_OK;
}

/* Wet/dry only: min(1, tau_i / dt) of cell i, tau_i = h_i |V_i| / M_i its
 * draining time (1 when no mass leaves it). */
static double drain_ratio(const view *v, const double *const *W, const double *H, double g,
                          double dt, int64_t i) {
  double Fl[4][OM_MAX_EDGES], Dl[OM_MAX_EDGES], out[OM_MAX_EDGES];
  int n = cell_terms(v, W, H, g, i, Fl, Dl);
  for (int k = 0; k < n; ++k) out[k] = fmax(Fl[0][k], 0.0);
  double M = psum(out, n);
  if (!(M > 0.0)) return 1.0;
  return fmin(1.0, W[0][i] * view_area(v, i) / M / dt);
}

/* Wet/dry only: scale every term of each edge of cell i by the ratio of the
 * cell its mass flux leaves (ratio_of(j) gives it for any cell j). */
static void drain_scale(const view *v, int64_t i, double Fl[4][OM_MAX_EDGES], int n,
                        double ri, const double *ratios, const double *const *W,
                        const double *H, double g, double dt) {
  int64_t nbr[OM_MAX_EDGES];
  double exs[OM_MAX_EDGES], eys[OM_MAX_EDGES], lens[OM_MAX_EDGES];
  view_edges(v, i, nbr, exs, eys, lens);
  for (int k = 0; k < n; ++k) {
    double theta = 1.0;
    if (Fl[0][k] > 0.0) theta = ri;
    else if (Fl[0][k] < 0.0 && nbr[k] >= 0)
      theta = ratios ? ratios[nbr[k]] : drain_ratio(v, W, H, g, dt, nbr[k]);
    for (int c = 0; c < 4; ++c) Fl[c][k] *= theta;
  }
}

/* Wet/dry only: a depth below zero (rounding) is clamped, and a dry cell
 * keeps no discharge. */
static void dry_cleanup(double w[4]) {
  if (!g_wet_dry) return;
  if (w[0] < 0.0) w[0] = 0.0;
  if (w[0] <= g_h_dry) w[1] = w[2] = 0.0;
}

static int update_view(const view *v, double *const *W, const double *H, double g,
                       double dt, double *work) {
  const double *const *Wc = (const double *const *)W;
  double Fl[4][OM_MAX_EDGES], Dl[OM_MAX_EDGES];
  int64_t N = view_cells(v);
  double *ratios = NULL;
  if (g_wet_dry) {
    ratios = (double *)malloc((size_t)N * sizeof(double));
    if (!ratios) return OM_ERR_ARG;
    for (int64_t i = 0; i < N; ++i) ratios[i] = drain_ratio(v, Wc, H, g, dt, i);
  }
  for (int64_t i = 0; i < N; ++i) {
    int n = cell_terms(v, Wc, H, g, i, Fl, Dl);
    if (ratios) drain_scale(v, i, Fl, n, ratios[i], ratios, Wc, H, g, dt);
    for (int c = 0; c < 4; ++c)
      work[c * N + i] = W[c][i] - dt / view_area(v, i) * psum(Fl[c], n);
  }
  free(ratios);
  int status = OM_OK;
  for (int64_t i = 0; i < N; ++i) {
    double w[4];
    for (int c = 0; c < 4; ++c) w[c] = work[c * N + i];
    dry_cleanup(w);
    for (int c = 0; c < 4; ++c) W[c][i] = w[c];
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
    if (g_wet_dry)
      drain_scale(v, i, Fl, n, drain_ratio(v, W, H, g, dt, i), NULL, W, H, g, dt);
    double w[4];
    for (int c = 0; c < 4; ++c) w[c] = W[c][i] - dt / view_area(v, i) * psum(Fl[c], n);
    dry_cleanup(w);
    for (int c = 0; c < 4; ++c) out[c * n_sel + s] = w[c];
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

/* ======================================================================
 * Two layers ([P1] Sec. 2.1 eq. (1), Sec. 2.2 steps 1-4 with four
 * components in the normal frame).  W = (h1, q1x, q1y, h2, q2x, q2y).
 * Readings: the density ratio r stripped from the garbled text is restored in
 * the coupling of the lower layer (B: -r g h2 dh1) and in A_ij[3][0]; the
 * wall ghost mirrors both layers.
 * ====================================================================== */

void om_wall_ghost2(const double *Wi, double ex, double ey, double *Wg) {
  for (int k = 0; k < 2; ++k) {
    const double *w = Wi + 3 * k;
    double *o = Wg + 3 * k;
    double qn = w[1] * ex + w[2] * ey;
    o[0] = w[0];
    o[1] = w[1] - 2.0 * qn * ex;
    o[2] = w[2] - 2.0 * qn * ey;
  }
}

/* p(l) = Q1(l) Q2(l) - r c1s c2s with Q_k(l) = (l - u_k)^2 - c_ks */
typedef struct {
  double u1, u2, c1s, c2s, r;
} quartic;

static double qk(double l, double u, double cs) { return (l - u) * (l - u) - cs; }
static double pq(const quartic *q, double l) {
  return qk(l, q->u1, q->c1s) * qk(l, q->u2, q->c2s) - q->r * q->c1s * q->c2s;
}
static double dpq(const quartic *q, double l) {
  return 2.0 * (l - q->u1) * qk(l, q->u2, q->c2s) + 2.0 * (l - q->u2) * qk(l, q->u1, q->c1s);
}

/* bisection of f on [lo, hi] with f(lo) and f(hi) of opposite signs (or one
 * of them zero) until the interval is a few ulp wide */
static double bisect(const quartic *q, double (*f)(const quartic *, double), double lo,
                     double hi) {
  double flo = f(q, lo);
  for (int it = 0; it < 200; ++it) {
    double mid = 0.5 * (lo + hi);
    if (!(mid > lo && mid < hi)) break;
    double fm = f(q, mid);
    if (fm == 0.0) return mid;
    if ((fm > 0.0) == (flo > 0.0)) {
      lo = mid;
      flo = fm;
    } else {
      hi = mid;
    }
  }
  return 0.5 * (lo + hi);
}

/* the local maximum of p in [a1, a2]: p has its two local minima in
 * [a0, a1] and [a2, a3] (p < -r c1s c2s where exactly one Q_k is negative)
 * and its local maximum between them, so p' > 0 left of the maximum and
 * p' < 0 right of it; the bisection follows that sign alone (the end values
 * of p' vanish when roots of Q1 and Q2 coincide, e.g. equal layers) */
static double local_max(const quartic *q, double lo, double hi) {
  for (int it = 0; it < 200; ++it) {
    double mid = 0.5 * (lo + hi);
    if (!(mid > lo && mid < hi)) break;
    double fm = dpq(q, mid);
    if (fm == 0.0) return mid;
    if (fm > 0.0) lo = mid;
    else hi = mid;
  }
  return 0.5 * (lo + hi);
}

/* two Newton steps on p, kept inside [lo, hi] */
static double polish(const quartic *q, double l, double lo, double hi) {
  for (int it = 0; it < 2; ++it) {
    double d = dpq(q, l);
    if (d == 0.0) break;
    double n = l - pq(q, l) / d;
    if (n >= lo && n <= hi) l = n;
  }
  return l;
}

int om_roots2(double u1, double u2, double c1s, double c2s, double r, double *lam) {
  quartic q = {u1, u2, c1s, c2s, r};
  double c1 = sqrt(c1s), c2 = sqrt(c2s);
  /* roots of Q1 Q2, sorted: p is -r c1s c2s <= 0 there */
  double a[4] = {u1 - c1, u1 + c1, u2 - c2, u2 + c2};
  for (int i = 1; i < 4; ++i)
    for (int j = i; j > 0 && a[j - 1] > a[j]; --j) {
      double t = a[j];
      a[j] = a[j - 1];
      a[j - 1] = t;
    }
  double step = c1 + c2;
  /* p(a[k]) = -r c1s c2s <= 0; where rounding makes it non-negative (r = 0
   * or a vanishing c_k) the root is a[k] itself */
  /* outer roots: below a[0] and above a[3]; widen the bracket outward until
   * p changes sign */
  if (!(pq(&q, a[0]) < 0.0)) {
    lam[0] = a[0];
  } else {
    double lo = a[0] - step;
    while (pq(&q, lo) <= 0.0) {
      step *= 2.0;
      lo = a[0] - step;
    }
    lam[0] = polish(&q, bisect(&q, pq, lo, a[0]), lo, a[0]);
  }
  step = c1 + c2;
  if (!(pq(&q, a[3]) < 0.0)) {
    lam[3] = a[3];
  } else {
    double hi = a[3] + step;
    while (pq(&q, hi) <= 0.0) {
      step *= 2.0;
      hi = a[3] + step;
    }
    lam[3] = polish(&q, bisect(&q, pq, a[3], hi), a[3], hi);
  }
  /* inner pair: p has its local maximum m in (a[1], a[2]) (p' > 0 at a[1],
   * < 0 at a[2]); real roots need p(m) > 0 */
  if (!(a[2] > a[1])) return OM_ERR_HYPERBOLIC;
  double m = local_max(&q, a[1], a[2]);
  if (!(pq(&q, m) > 0.0)) return OM_ERR_HYPERBOLIC;
  lam[1] = (pq(&q, a[1]) < 0.0) ? polish(&q, bisect(&q, pq, a[1], m), a[1], m) : a[1];
  lam[2] = (pq(&q, a[2]) < 0.0) ? polish(&q, bisect(&q, pq, m, a[2]), m, a[2]) : a[2];
  return OM_OK;
}

/* inverse of a 4x4 matrix by Gauss-Jordan elimination with partial pivoting;
 * returns 0 if singular */
static int inv4(const double Min[4][4], double Inv[4][4]) {
  double M[4][8];
  for (int i = 0; i < 4; ++i)
    for (int j = 0; j < 8; ++j) M[i][j] = j < 4 ? Min[i][j] : (double)(j - 4 == i);
  for (int col = 0; col < 4; ++col) {
    int piv = col;
    for (int i = col + 1; i < 4; ++i)
      if (fabs(M[i][col]) > fabs(M[piv][col])) piv = i;
    if (M[piv][col] == 0.0) return 0;
    if (piv != col)
      for (int j = 0; j < 8; ++j) {
        double t = M[col][j];
        M[col][j] = M[piv][j];
        M[piv][j] = t;
      }
    double d = M[col][col];
    for (int j = 0; j < 8; ++j) M[col][j] /= d;
    for (int i = 0; i < 4; ++i) {
      if (i == col) continue;
      double f = M[i][col];
      for (int j = 0; j < 8; ++j) M[i][j] -= f * M[col][j];
    }
  }
  for (int i = 0; i < 4; ++i)
    for (int j = 0; j < 4; ++j) Inv[i][j] = M[i][j + 4];
  return 1;
}

/* physical flux of one layer in the normal frame (mass, normal momentum) */
static void flux_layer(double h, double qn, double g, double *F) {
  F[0] = qn;
  F[1] = qn * qn / h + 0.5 * g * h * h;
}

int om_flux2(const double *Wi, const double *Wj, double Hi, double Hj,
             double ex, double ey, double g, double r, double *F, double *Dinf) {
  /* step 1: W_eta = T_eta W for both layers */
  double h[2][2], qn[2][2], qt[2][2], ux[2][2], uy[2][2];
  const double *W[2] = {Wi, Wj};
  for (int side = 0; side < 2; ++side)
    for (int k = 0; k < 2; ++k) {
      const double *w = W[side] + 3 * k;
      h[side][k] = w[0];
      qn[side][k] = w[1] * ex + w[2] * ey;
      qt[side][k] = -w[1] * ey + w[2] * ex;
      ux[side][k] = w[1] / w[0];
      uy[side][k] = w[2] / w[0];
    }
  /* step 2: Roe averages per layer and the matrix A_ij */
  double un[2], hb[2], cs[2];
  for (int k = 0; k < 2; ++k) {
    double si = sqrt(h[0][k]), sj = sqrt(h[1][k]);
    double ax = (si * ux[0][k] + sj * ux[1][k]) / (si + sj);
    double ay = (si * uy[0][k] + sj * uy[1][k]) / (si + sj);
    un[k] = ax * ex + ay * ey;
    hb[k] = 0.5 * (h[0][k] + h[1][k]);
    cs[k] = g * hb[k];
  }
  /* A_ij = [[0, 1, 0, 0], [c1^2 - u1^2, 2 u1, c1^2, 0], [0, 0, 0, 1],
   *         [r c2^2, 0, c2^2 - u2^2, 2 u2]] with c_k^2 = g hbar_k */
  double lam[4];
  int st = om_roots2(un[0], un[1], cs[0], cs[1], r, lam);
  if (st != OM_OK) return st;
  /* eigenvectors K_k = (1, l, Q1(l)/c1^2, l Q1(l)/c1^2) */
  double K[4][4], Kinv[4][4];
  for (int k = 0; k < 4; ++k) {
    double mu = qk(lam[k], un[0], cs[0]) / cs[0];
    K[0][k] = 1.0;
    K[1][k] = lam[k];
    K[2][k] = mu;
    K[3][k] = lam[k] * mu;
  }
  if (!inv4(K, Kinv)) return OM_ERR_HYPERBOLIC;
  /* P^- = 1/2 K (I - sgn D) K^-1 */
  double w[4], P[4][4];
  for (int k = 0; k < 4; ++k) w[k] = 0.5 * (1.0 - sgn(lam[k]));
  for (int a = 0; a < 4; ++a)
    for (int b = 0; b < 4; ++b) {
      double acc = 0.0;
      for (int k = 0; k < 4; ++k) acc += K[a][k] * w[k] * Kinv[k][b];
      P[a][b] = acc;
    }
  /* d = F_1(W_j) - F_1(W_i) - B_ij (W_j - W_i) - S_ij (H_j - H_i) in the
   * components [1, 2, 4, 5]: B couples -g h1 dh2 (upper) and -r g h2 dh1
   * (lower); S = (0, g h1, 0, g h2) with Roe-averaged depths */
  double Fi[4], Fj[4];
  flux_layer(h[0][0], qn[0][0], g, Fi);
  flux_layer(h[0][1], qn[0][1], g, Fi + 2);
  flux_layer(h[1][0], qn[1][0], g, Fj);
  flux_layer(h[1][1], qn[1][1], g, Fj + 2);
  double dH = Hj - Hi;
  double dh1 = h[1][0] - h[0][0], dh2 = h[1][1] - h[0][1];
  double d[4];
  d[0] = Fj[0] - Fi[0];
  d[1] = Fj[1] - Fi[1] - (-g * hb[0] * dh2) - g * hb[0] * dH;
  d[2] = Fj[2] - Fi[2];
  d[3] = Fj[3] - Fi[3] - (-r * g * hb[1] * dh1) - g * hb[1] * dH;
  /* Phi^- = P^- d + F_1(W_eta,i) */
  double phi[4];
  for (int a = 0; a < 4; ++a) {
    double acc = 0.0;
    for (int b = 0; b < 4; ++b) acc += P[a][b] * d[b];
    phi[a] = acc + Fi[a];
  }
  if (g_entropy_fix) {
    /* the same Harten-Hyman viscosity as one layer, per wave of A_ij: the
     * k-th speed of each side is the k-th smallest eigenvalue of the side's
     * own Jacobian, i.e. the k-th root of the quartic with that side's
     * normal velocities and c_k^2 = g h_k (an error if that side's own
     * system is not hyperbolic); beta = K^-1 (W_j - W_i) */
    double lamS[2][4];
    for (int side = 0; side < 2; ++side) {
      int st2 = om_roots2(qn[side][0] / h[side][0], qn[side][1] / h[side][1], g * h[side][0],
                          g * h[side][1], r, lamS[side]);
      if (st2 != OM_OK) return st2;
    }
    double dW[4] = {h[1][0] - h[0][0], qn[1][0] - qn[0][0], h[1][1] - h[0][1],
                    qn[1][1] - qn[0][1]};
    for (int k = 0; k < 4; ++k) {
      double beta = 0.0;
      for (int b = 0; b < 4; ++b) beta += Kinv[k][b] * dW[b];
      double nu = 0.5 * (fabs(lam[k]) - harten_abs(lam[k], lamS[0][k], lamS[1][k])) * beta;
      for (int a = 0; a < 4; ++a) phi[a] += nu * K[a][k];
    }
  }
  /* step 3: tangential discharge of each layer upwinded with its mass flux */
  double pt[2];
  for (int k = 0; k < 2; ++k) {
    double m = phi[2 * k];
    double ut = (m > 0.0) ? qt[0][k] / h[0][k] : qt[1][k] / h[1][k];
    pt[k] = m * ut;
  }
  /* step 4: back to Cartesian components */
  for (int k = 0; k < 2; ++k) {
    F[3 * k + 0] = phi[2 * k];
    F[3 * k + 1] = phi[2 * k + 1] * ex - pt[k] * ey;
    F[3 * k + 2] = phi[2 * k + 1] * ey + pt[k] * ex;
  }
  double dm = 0.0;
  for (int k = 0; k < 4; ++k) dm = fmax(dm, fabs(lam[k]));
  *Dinf = dm;
  return OM_OK;
}

static int cell_terms2(const view *v, const double *const *W, const double *H, double g,
                       double r, int64_t i, double Fl[6][OM_MAX_EDGES],
                       double Dl[OM_MAX_EDGES], int *n_out) {
  int64_t nbr[OM_MAX_EDGES];
  double exs[OM_MAX_EDGES], eys[OM_MAX_EDGES], lens[OM_MAX_EDGES];
  int n = view_edges(v, i, nbr, exs, eys, lens);
  double Wi[6], Wj[6];
  for (int k = 0; k < 6; ++k) Wi[k] = W[k][i];
  for (int e = 0; e < n; ++e) {
    double Hj;
    if (nbr[e] >= 0) {
      for (int k = 0; k < 6; ++k) Wj[k] = W[k][nbr[e]];
      Hj = H[nbr[e]];
    } else {
      om_wall_ghost2(Wi, exs[e], eys[e], Wj);
      Hj = H[i];
    }
    double F[6], D;
    int st = om_flux2(Wi, Wj, H[i], Hj, exs[e], eys[e], g, r, F, &D);
    if (st != OM_OK) return st;
    for (int c = 0; c < 6; ++c) Fl[c][e] = lens[e] * F[c];
    Dl[e] = lens[e] * D;
  }
  *n_out = n;
  return OM_OK;
}

static double dt_view2(const view *v, const double *const *W, const double *H, double g,
                       double r, double cfl, int *status) {
  double dt = INFINITY;
  double Fl[6][OM_MAX_EDGES], Dl[OM_MAX_EDGES];
  int64_t N = view_cells(v);
  if (status) *status = OM_OK;
  for (int64_t i = 0; i < N; ++i) {
    int n;
    int st = cell_terms2(v, W, H, g, r, i, Fl, Dl, &n);
    if (st != OM_OK) {
      if (status) *status = st;
      return NAN;
    }
    double dti = 2.0 * cfl * view_area(v, i) / psum(Dl, n);
    if (isnan(dti)) return dti;
    if (dti < dt) dt = dti;
  }
  return dt;
}

static int check_state2(const double w[6]) {
  for (int k = 0; k < 6; ++k)
    if (!isfinite(w[k])) return OM_ERR_NONFINITE;
  if (!(w[0] > 0.0) || !(w[3] > 0.0)) return OM_ERR_DEPTH;
  return OM_OK;
}

static int update_view2(const view *v, double *const *W, const double *H, double g, double r,
                        double dt, double *work) {
  const double *const *Wc = (const double *const *)W;
  double Fl[6][OM_MAX_EDGES], Dl[OM_MAX_EDGES];
  int64_t N = view_cells(v);
  for (int64_t i = 0; i < N; ++i) {
    int n;
    int st = cell_terms2(v, Wc, H, g, r, i, Fl, Dl, &n);
    if (st != OM_OK) return st;
    for (int c = 0; c < 6; ++c)
      work[c * N + i] = W[c][i] - dt / view_area(v, i) * psum(Fl[c], n);
  }
  int status = OM_OK;
  for (int64_t i = 0; i < N; ++i) {
    double w[6];
    for (int c = 0; c < 6; ++c) {
      w[c] = work[c * N + i];
      W[c][i] = w[c];
    }
    int s = check_state2(w);
    if (s != OM_OK && status == OM_OK) status = s;
  }
  return status;
}

static int update_at_view2(const view *v, const double *const *W, const double *H, double g,
                           double r, double dt, const int64_t *cells, int64_t n_sel,
                           double *out) {
  double Fl[6][OM_MAX_EDGES], Dl[OM_MAX_EDGES];
  for (int64_t s = 0; s < n_sel; ++s) {
    int64_t i = cells[s];
    int n;
    int st = cell_terms2(v, W, H, g, r, i, Fl, Dl, &n);
    if (st != OM_OK) return st;
    for (int c = 0; c < 6; ++c)
      out[c * n_sel + s] = W[c][i] - dt / view_area(v, i) * psum(Fl[c], n);
  }
  return OM_OK;
}

static int run_view2(const view *v, double *const *W, const double *H, double g, double r,
                     double cfl, int64_t nsteps, double *dts, double *work,
                     int64_t *steps_done) {
  int64_t done = 0;
  int status = OM_OK;
  for (int64_t n = 0; n < nsteps; ++n) {
    int st = OM_OK;
    double dt = dt_view2(v, (const double *const *)W, H, g, r, cfl, &st);
    if (dts) dts[n] = dt;
    if (st != OM_OK) {
      status = st;
      break;
    }
    if (!isfinite(dt) || !(dt > 0.0)) {
      status = OM_ERR_NONFINITE;
      break;
    }
    status = update_view2(v, W, H, g, r, dt, work);
    ++done;
    if (status != OM_OK) break;
  }
  if (steps_done) *steps_done = done;
  return status;
}

double om_dt2(const om_mesh *m, const double *const *W, const double *H, double g, double r,
              double cfl, int *status) {
  view v = mesh_view(m);
  return dt_view2(&v, W, H, g, r, cfl, status);
}
int om_update2(const om_mesh *m, double *const *W, const double *H, double g, double r,
               double dt, double *work) {
  view v = mesh_view(m);
  return update_view2(&v, W, H, g, r, dt, work);
}
int om_update2_at(const om_mesh *m, const double *const *W, const double *H, double g,
                  double r, double dt, const int64_t *cells, int64_t n_sel, double *out) {
  view v = mesh_view(m);
  return update_at_view2(&v, W, H, g, r, dt, cells, n_sel, out);
}
int om_run2(const om_mesh *m, double *const *W, const double *H, double g, double r,
            double cfl, int64_t nsteps, double *dts, double *work, int64_t *steps_done) {
  view v = mesh_view(m);
  return run_view2(&v, W, H, g, r, cfl, nsteps, dts, work, steps_done);
}
double om_grid_dt2(int64_t nx, int64_t ny, double dx, double dy, const double *const *W,
                   const double *H, double g, double r, double cfl, int *status) {
  view v = grid_view(nx, ny, dx, dy);
  return dt_view2(&v, W, H, g, r, cfl, status);
}
int om_grid_update2(int64_t nx, int64_t ny, double dx, double dy, double *const *W,
                    const double *H, double g, double r, double dt, double *work) {
  view v = grid_view(nx, ny, dx, dy);
  return update_view2(&v, W, H, g, r, dt, work);
}
int om_grid_run2(int64_t nx, int64_t ny, double dx, double dy, double *const *W,
                 const double *H, double g, double r, double cfl, int64_t nsteps,
                 double *dts, double *work, int64_t *steps_done) {
  view v = grid_view(nx, ny, dx, dy);
  return run_view2(&v, W, H, g, r, cfl, nsteps, dts, work, steps_done);
}

/* ======================================================================
 * Triangle meshes: geometry of the finite volumes of [P1] Sec. 2.2 (cells
 * V_i with area |V_i|, edges Gamma_ij with length and unit normal pointing
 * from V_i to V_j).
 * ====================================================================== */

typedef struct {
  int64_t key;   /* min vertex * n_vertices + max vertex */
  int64_t cell;
  int local;     /* 0, 1, 2: edge (v0 v1), (v1 v2), (v2 v0) */
} half_edge;

static int cmp_half_edge(const void *a, const void *b) {
  const half_edge *x = (const half_edge *)a, *y = (const half_edge *)b;
  if (x->key != y->key) return x->key < y->key ? -1 : 1;
  if (x->cell != y->cell) return x->cell < y->cell ? -1 : 1;
  return x->local - y->local;
}

int om_tri_mesh(int64_t n_vertices, const double *xy, int64_t n_cells,
                const int32_t *tri, double *area, int64_t *edge_start,
                int64_t *nbr, double *eta_x, double *eta_y, double *len) {
  for (int64_t c = 0; c < 3 * n_cells; ++c)
    if (tri[c] < 0 || tri[c] >= n_vertices) return OM_ERR_ARG;
  half_edge *he = (half_edge *)malloc((size_t)(3 * n_cells) * sizeof(half_edge));
  if (!he) return OM_ERR_ARG;
  for (int64_t c = 0; c < n_cells; ++c) {
    const int32_t *v = tri + 3 * c;
    double x0 = xy[2 * v[0]], y0 = xy[2 * v[0] + 1];
    double x1 = xy[2 * v[1]], y1 = xy[2 * v[1] + 1];
    double x2 = xy[2 * v[2]], y2 = xy[2 * v[2] + 1];
    /* shoelace area; counter-clockwise triangles have a positive one */
    area[c] = 0.5 * ((x1 - x0) * (y2 - y0) - (x2 - x0) * (y1 - y0));
    if (!(area[c] > 0.0)) {
      free(he);
      return OM_ERR_ARG;
    }
    edge_start[c] = 3 * c;
    for (int k = 0; k < 3; ++k) {
      int64_t a = v[k], b = v[(k + 1) % 3];
      int64_t e = 3 * c + k;
      double ex = xy[2 * b] - xy[2 * a], ey = xy[2 * b + 1] - xy[2 * a + 1];
      double l = sqrt(ex * ex + ey * ey);
      /* outward normal of a counter-clockwise edge a -> b: (ey, -ex) / l */
      eta_x[e] = ey / l;
      eta_y[e] = -ex / l;
      len[e] = l;
      nbr[e] = -1;
      he[e].key = (a < b ? a : b) * n_vertices + (a < b ? b : a);
      he[e].cell = c;
      he[e].local = k;
    }
  }
  edge_start[n_cells] = 3 * n_cells;
  /* pair the half-edges that share their two vertices */
  qsort(he, (size_t)(3 * n_cells), sizeof(half_edge), cmp_half_edge);
  int status = OM_OK;
  for (int64_t s = 0; s < 3 * n_cells;) {
    int64_t t = s + 1;
    while (t < 3 * n_cells && he[t].key == he[s].key) ++t;
    if (t - s > 2) status = OM_ERR_ARG;
    if (t - s == 2) {
      nbr[3 * he[s].cell + he[s].local] = he[s + 1].cell;
      nbr[3 * he[s + 1].cell + he[s + 1].local] = he[s].cell;
    }
    s = t;
  }
  free(he);
  return status;
}
