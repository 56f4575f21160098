"""The boundary is a C ABI: include/swe.h and include/swe_probe.h compile as C99
(and as C++), and a
C program links against libswe and gets its argument checks and status
strings without a GPU (no compute call)."""
import os
import shutil
import subprocess

import pytest

from finite_volume_shallow_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "swe.h"
#include "swe_probe.h"

int main(void) {
  swe_grid grid;
  swe_params params;
  swe_state *s = (swe_state *)0x1;
  double H[4] = {0, 0, 0, 0};
  double h[4] = {1, 1, 1, 1}, z[4] = {0, 0, 0, 0};
  const void *W[4];
  int bad = 0;
  memset(&params, 0, sizeof params);
  grid.nx = 2; grid.ny = 2; grid.dx = 1.0; grid.dy = 1.0;
  params.n_layers = 1; params.precision = 64; params.pollutant = 1;
  params.g = 9.81; params.r = 0.0; params.cfl = 0.9; params.stream = NULL;
  W[0] = h; W[1] = z; W[2] = z; W[3] = z;
  params.cfl = 1.5;                     /* outside (0, 1] */
  if (swe_create_grid(&grid, H, W, &params, &s) != SWE_ERR_ARG || s != NULL) bad |= 1;
  params.cfl = 0.9;
  params.entropy_fix = 7;               /* only 0 or 1 */
  if (swe_create_grid(&grid, H, W, &params, &s) != SWE_ERR_ARG) bad |= 2;
  params.entropy_fix = 0;
  grid.nx = 0;
  if (swe_create_grid(&grid, H, W, &params, &s) != SWE_ERR_ARG) bad |= 4;
  if (swe_step(NULL, 0.9, NULL) != SWE_ERR_ARG) bad |= 8;
  swe_destroy(NULL);
  if (strcmp(swe_status_str(SWE_OK), swe_status_str(SWE_ERR_ARG)) == 0) bad |= 16;
  {
    double rate = 0.0;
    if (swe_probe_fma_rate(9, 10.0, NULL, &rate, NULL) != SWE_ERR_ARG) bad |= 32;
    if (swe_probe_fma_rate(SWE_PROBE_DFMA, 0.5, NULL, &rate, NULL) != SWE_ERR_ARG) bad |= 64;
    if (swe_probe_fma_rate(SWE_PROBE_FFMA, 10.0, NULL, NULL, NULL) != SWE_ERR_ARG) bad |= 128;
  }
  printf("%d\n", bad);
  return bad;
}
"""


@pytest.fixture(scope="module")
def libdir():
    B.build()
    return os.path.dirname(B.LIB)


@pytest.mark.parametrize("lang,compiler,flags", [("c", "gcc", ["-std=c99", "-Wall", "-Werror"]),
                                                 ("cpp", "g++", ["-std=c++17", "-Wall"])])
def test_header_compiles_and_a_program_links(tmp_path, libdir, lang, compiler, flags):
    cc = shutil.which(compiler)
    if cc is None:
        pytest.skip(f"{compiler} not found")
    src = tmp_path / f"use_swe.{lang}"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_swe"
    subprocess.run([cc, *flags, "-I", INCLUDE, str(src), "-o", str(exe), "-L", libdir,
                    "-lswe", f"-Wl,-rpath,{libdir}"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
