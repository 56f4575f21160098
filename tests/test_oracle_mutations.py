"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (on the CPU,
in a temporary directory), compiles it, and runs the pin suite against that
copy; the suite must fail.  The committed oracle is never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "swe_oracle.c")
HDR = os.path.join(ROOT, "oracle", "swe_oracle.h")

MUTANTS = {
    # the entropy fix: anti-diffusion, delta from the wrong sides, beta from
    # the jump with its components swapped
    "efix_sign": ("0.5 * (fabs(lam[k]) - harten_abs(lam[k], lamL[k], lamR[k])) * beta",
                  "0.5 * (harten_abs(lam[k], lamL[k], lamR[k]) - fabs(lam[k])) * beta"),
    "efix_delta": ("fmax(lam - lamL, lamR - lam)", "fmax(lamL - lam, lam - lamR)"),
    "efix_beta": ("Kinv[k][0] * dW[0] + Kinv[k][1] * dW[1]", "Kinv[k][0] * dW[1] + Kinv[k][1] * dW[0]"),
    # two layers: the same three, and each side's speeds from the quartic
    # with the layers' depths swapped
    "efix2_sign": ("0.5 * (fabs(lam[k]) - harten_abs(lam[k], lamS[0][k], lamS[1][k])) * beta",
                   "0.5 * (harten_abs(lam[k], lamS[0][k], lamS[1][k]) - fabs(lam[k])) * beta"),
    "efix2_sides": ("harten_abs(lam[k], lamS[0][k], lamS[1][k])",
                    "harten_abs(lam[k], lamS[1][k], lamS[0][k])"),
    "efix2_beta": ("double dW[4] = {h[1][0] - h[0][0], qn[1][0] - qn[0][0], h[1][1] - h[0][1],\n"
                   "                    qn[1][1] - qn[0][1]};",
                   "double dW[4] = {h[1][1] - h[0][1], qn[1][1] - qn[0][1], h[1][0] - h[0][0],\n"
                   "                    qn[1][0] - qn[0][0]};"),
    "efix2_layer_speeds": ("g * h[side][0],\n                          g * h[side][1], r",
                           "g * h[side][1],\n                          g * h[side][0], r"),
    # bathymetry source with the wrong sign
    "source_sign": ("- g * hbar * (Hj - Hi)", "+ g * hbar * (Hj - Hi)"),
    # source term dropped
    "source_dropped": ("- g * hbar * (Hj - Hi)", "- 0.0 * (Hj - Hi)"),
    # arithmetic instead of sqrt(h)-weighted velocity average
    "plain_average": ("double ux = (si * uxi + sj * uxj) / (si + sj);",
                      "double ux = 0.5 * (uxi + uxj);"),
    # P^+ instead of P^-
    "p_plus": ("0.5 * (1.0 - sgn(lam[0])), 0.5 * (1.0 - sgn(lam[1]))",
               "0.5 * (1.0 + sgn(lam[0])), 0.5 * (1.0 + sgn(lam[1]))"),
    # tangential velocity upwinded from the wrong side
    "tangential_downwind": ("    ut = dry_i ? 0.0 : qti / hi;\n    Cs = dry_i ? 0.0 : Wi[3] / hi;\n"
                            "  } else {\n    ut = dry_j ? 0.0 : qtj / hj;",
                            "    ut = dry_j ? 0.0 : qtj / hj;\n    Cs = dry_i ? 0.0 : Wi[3] / hi;\n"
                            "  } else {\n    ut = dry_i ? 0.0 : qti / hi;"),
    # pollutant upwinded from the wrong side
    "pollutant_downwind": ("    Cs = dry_i ? 0.0 : Wi[3] / hi;\n  } else {\n"
                           "    ut = dry_j ? 0.0 : qtj / hj;\n    Cs = dry_j ? 0.0 : Wj[3] / hj;",
                           "    Cs = dry_j ? 0.0 : Wj[3] / hj;\n  } else {\n"
                           "    ut = dry_j ? 0.0 : qtj / hj;\n    Cs = dry_i ? 0.0 : Wi[3] / hi;"),
    # wet/dry: the emerged-bank rule reversed (flooded cells become walls,
    # banks pass water), the draining limit taken from the receiving cell,
    # no draining limit at all, the draining time without the cell's area
    "wd_bank_rule": ("(dry_j && -Hj >= Wi[0] - Hi) || (dry_i && -Hi >= Wj[0] - Hj)",
                     "(dry_j && -Hj <= Wi[0] - Hi) || (dry_i && -Hi <= Wj[0] - Hj)"),
    "wd_theta_receiver": ("if (Fl[0][k] > 0.0) theta = ri;\n    else if (Fl[0][k] < 0.0 && nbr[k] >= 0)",
                          "if (Fl[0][k] < 0.0) theta = ri;\n    else if (Fl[0][k] > 0.0 && nbr[k] >= 0)"),
    "wd_no_drain": ("for (int c = 0; c < 4; ++c) Fl[c][k] *= theta;",
                    "for (int c = 0; c < 4; ++c) Fl[c][k] *= 1.0 + 0.0 * theta;"),
    "wd_tau_area": ("return fmin(1.0, W[0][i] * view_area(v, i) / M / dt);",
                    "return fmin(1.0, W[0][i] / M / dt);"),
    # back-rotation with a transposed operator
    "back_rotation": ("F[1] = phi[1] * ex - phit * ey;", "F[1] = phi[1] * ex + phit * ey;"),
    # hydrostatic pressure without its factor 1/2 (one layer, two layers)
    "pressure_half": ("qn * qn / h + 0.5 * g * h * h", "qn * qn / h + g * h * h", 0),
    "pressure_half_2": ("qn * qn / h + 0.5 * g * h * h", "qn * qn / h + g * h * h", 1),
    # CFL without the factor 2 of eq. (5)
    "cfl_factor": ("double dti = 2.0 * cfl * view_area(v, i) / s;",
                   "double dti = cfl * view_area(v, i) / s;"),
    # edge lengths of the two directions swapped
    "edge_length": ("len[k] = (k == 0 || k == 2) ? dy : dx;",
                    "len[k] = (k == 0 || k == 2) ? dx : dy;"),
    # wrong neighbour index (North points South)
    "neighbour_index": ("static const int dj[4] = {0, 1, 0, -1};",
                        "static const int dj[4] = {0, -1, 0, -1};"),
    # update with the wrong sign (one layer, then two layers)
    "update_sign": ("work[c * N + i] = W[c][i] - dt / view_area(v, i)",
                    "work[c * N + i] = W[c][i] + dt / view_area(v, i)", 0),
    "update_sign_2": ("work[c * N + i] = W[c][i] - dt / view_area(v, i)",
                      "work[c * N + i] = W[c][i] + dt / view_area(v, i)", 1),
    # wall ghost that does not reflect the normal discharge
    "wall_no_reflect": ("Wg[1] = Wi[1] - 2.0 * qn * ex;", "Wg[1] = Wi[1];"),
    # two layers: coupling term of the upper layer with the wrong sign
    "coupling_sign": ("d[1] = Fj[1] - Fi[1] - (-g * hb[0] * dh2) - g * hb[0] * dH;",
                      "d[1] = Fj[1] - Fi[1] + (-g * hb[0] * dh2) - g * hb[0] * dH;"),
    # two layers: density ratio dropped from the lower layer's coupling
    "coupling_no_r": ("d[3] = Fj[3] - Fi[3] - (-r * g * hb[1] * dh1) - g * hb[1] * dH;",
                      "d[3] = Fj[3] - Fi[3] - (-g * hb[1] * dh1) - g * hb[1] * dH;"),
    # two layers: eigenvectors built with the lower layer's Q
    "eigvec_wrong_layer": ("double mu = qk(lam[k], un[0], cs[0]) / cs[0];",
                           "double mu = qk(lam[k], un[1], cs[1]) / cs[0];"),
    # two layers: P^+ instead of P^-
    "p_plus_2": ("for (int k = 0; k < 4; ++k) w[k] = 0.5 * (1.0 - sgn(lam[k]));",
                 "for (int k = 0; k < 4; ++k) w[k] = 0.5 * (1.0 + sgn(lam[k]));"),
    # two layers: tangential velocity upwinded with the other layer's mass flux
    "tangential_other_layer": ("double m = phi[2 * k];", "double m = phi[2 * (1 - k)];"),
    # two layers: characteristic polynomial without the density ratio
    "charpoly_no_r": ("- q->r * q->c1s * q->c2s;", "- q->c1s * q->c2s;"),
    # two layers: the inner pair's bracket taken from the end signs of p'
    # (fails when roots of Q1 and Q2 coincide)
    "inner_max_by_end_signs": ("double m = local_max(&q, a[1], a[2]);",
                               "double m = bisect(&q, dpq, a[1], a[2]);"),
    # triangle meshes: inward instead of outward normals
    "tri_normal_inward": ("eta_x[e] = ey / l;\n      eta_y[e] = -ex / l;",
                          "eta_x[e] = -ey / l;\n      eta_y[e] = ex / l;"),
    # triangle meshes: shoelace area without its factor 1/2
    "tri_area_half": ("area[c] = 0.5 * ((x1 - x0)", "area[c] = ((x1 - x0)"),
    # triangle meshes: a half-edge paired with its own cell
    "tri_pair_self": ("nbr[3 * he[s].cell + he[s].local] = he[s + 1].cell;",
                      "nbr[3 * he[s].cell + he[s].local] = he[s].cell;"),
    # triangle meshes: unit edge lengths
    "tri_len_unit": ("len[e] = l;", "len[e] = 1.0;"),
}


@pytest.fixture(scope="module")
def workdir(tmp_path_factory):
    return tmp_path_factory.mktemp("mutants")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, workdir):
    old, new, *which = MUTANTS[name]
    src = open(SRC).read()
    if which:   # the k-th of several identical sites
        k = which[0]
        pos = -1
        for _ in range(k + 1):
            pos = src.index(old, pos + 1)
        mutated = src[:pos] + new + src[pos + len(old):]
    else:
        assert src.count(old) == 1, f"mutation site of {name} not found exactly once"
        mutated = src.replace(old, new)
    d = workdir / name
    d.mkdir()
    (d / "swe_oracle.c").write_text(mutated)
    shutil.copy(HDR, d / "swe_oracle.h")
    so = d / "liboracle.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", str(so), str(d / "swe_oracle.c"), "-lm"], check=True)
    env = dict(os.environ, SWE_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_oracle_pins.py"),
                        os.path.join(HERE, "test_oracle_pins2.py"),
                        os.path.join(HERE, "test_oracle_pins_tri.py"),
                        os.path.join(HERE, "test_oracle_pins_wetdry.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
