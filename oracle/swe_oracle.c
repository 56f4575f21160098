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

void om_grid_mesh(int64_t nx, int64_t ny, double dx, double dy, double *area,
                  int64_t *edge_start, int64_t *nbr, double *eta_x,
                  double *eta_y, double *len) {
  /* East, North, West, South */
  static const int di[4] = {1, 0, -1, 0};
  static const int dj[4] = {0, 1, 0, -1};
  int64_t e = 0;
  for (int64_t j = 0; j < ny; ++j) {
    for (int64_t i = 0; i < nx; ++i) {
      int64_t c = j * nx + i;
      area[c] = dx * dy;
      edge_start[c] = e;
      for (int k = 0; k < 4; ++k) {
        int64_t ii = i + di[k], jj = j + dj[k];
        int inside = ii >= 0 && ii < nx && jj >= 0 && jj < ny;
        nbr[e] = inside ? jj * nx + ii : -1;
        eta_x[e] = (double)di[k];
        eta_y[e] = (double)dj[k];
        len[e] = (k == 0 || k == 2) ? dy : dx;
        ++e;
      }
    }
  }
  edge_start[nx * ny] = e;
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

/* All edge terms of cell i: L_e F_e (4 components) and L_e ||D_e||. */
static int cell_terms(const om_mesh *m, const double *const *W, const double *H,
                      double g, int64_t i, double Fl[4][OM_MAX_EDGES],
                      double Dl[OM_MAX_EDGES]) {
  int64_t e0 = m->edge_start[i], e1 = m->edge_start[i + 1];
  int n = (int)(e1 - e0);
  double Wi[4], Wj[4];
  cell_state(W, i, Wi);
  for (int k = 0; k < n; ++k) {
    int64_t e = e0 + k;
    double ex = m->eta_x[e], ey = m->eta_y[e], L = m->len[e];
    double Hj;
    if (m->nbr[e] >= 0) {
      cell_state(W, m->nbr[e], Wj);
      Hj = H[m->nbr[e]];
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

double om_dt1(const om_mesh *m, const double *const *W, const double *H,
              double g, double cfl) {
  double dt = INFINITY;
  double Fl[4][OM_MAX_EDGES], Dl[OM_MAX_EDGES];
  for (int64_t i = 0; i < m->n_cells; ++i) {
    int n = cell_terms(m, W, H, g, i, Fl, Dl);
    double s = psum(Dl, n);
    double dti = 2.0 * cfl * m->area[i] / s;
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

int om_update1(const om_mesh *m, double *const *W, const double *H, double g,
               double dt, double *work) {
  const double *const *Wc = (const double *const *)W;
  double Fl[4][OM_MAX_EDGES], Dl[OM_MAX_EDGES];
  int64_t N = m->n_cells;
  for (int64_t i = 0; i < N; ++i) {
    int n = cell_terms(m, Wc, H, g, i, Fl, Dl);
    for (int c = 0; c < 4; ++c)
      work[c * N + i] = W[c][i] - dt / m->area[i] * psum(Fl[c], n);
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

void om_update1_at(const om_mesh *m, const double *const *W, const double *H,
                   double g, double dt, const int64_t *cells, int64_t n_sel,
                   double *out) {
  double Fl[4][OM_MAX_EDGES], Dl[OM_MAX_EDGES];
  for (int64_t s = 0; s < n_sel; ++s) {
    int64_t i = cells[s];
    int n = cell_terms(m, W, H, g, i, Fl, Dl);
    for (int c = 0; c < 4; ++c)
      out[c * n_sel + s] = W[c][i] - dt / m->area[i] * psum(Fl[c], n);
  }
}

int om_run1(const om_mesh *m, double *const *W, const double *H, double g,
            double cfl, int64_t nsteps, double *dts, double *work,
            int64_t *steps_done) {
  int64_t done = 0;
  int status = OM_OK;
  for (int64_t n = 0; n < nsteps; ++n) {
    double dt = om_dt1(m, (const double *const *)W, H, g, cfl);
    if (dts) dts[n] = dt;
    if (!isfinite(dt) || !(dt > 0.0)) {
      status = OM_ERR_NONFINITE;
      break;
    }
    status = om_update1(m, W, H, g, dt, work);
    ++done;
    if (status != OM_OK) break;
  }
  if (steps_done) *steps_done = done;
  return status;
}
