"""Host logic of the one-layer step's launch plan (csrc/swe_plan.h), compiled
on the CPU with g++: every plan keeps one wave when the bands fit, never cuts
a segment below its minimum length, gives the wall bands at least as many
segments as the others, and counts its warps consistently; the 8192 x 8192
fp32 grid on 152 SMs x 16 warp slots gets 17 segments per band and 22 in the
two wall bands (2339 warps)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "finite_volume_shallow_gb300", "csrc")

HARNESS = r"""
#include <stdio.h>
#include "swe_plan.h"
int main() {
  long long slots, nbands, ny;
  while (scanf("%lld %lld %lld", &slots, &nbands, &ny) == 3) {
    swe::StepPlan p = swe::plan_step(slots, nbands, ny);
    printf("%d %d %d %d\n", p.nbands, p.nsegs, p.nsegs_wall, p.units);
  }
  return 0;
}
"""


@pytest.fixture(scope="module")
def planner(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not found")
    d = tmp_path_factory.mktemp("plan")
    src = d / "plan.cpp"
    src.write_text(HARNESS)
    exe = d / "plan"
    subprocess.run([gxx, "-std=c++17", "-O1", "-I", CSRC, "-o", str(exe), str(src)], check=True)

    def run(cases):
        inp = "".join(f"{s} {b} {n}\n" for s, b, n in cases)
        out = subprocess.run([str(exe)], input=inp, capture_output=True, text=True, check=True)
        return [tuple(int(v) for v in line.split()) for line in out.stdout.splitlines()]
    return run


def bands_of(nx, own=60):
    return (nx + own - 1) // own


def test_the_8192_grid_plan(planner):
    slots = 152 * 4 * 4          # SMs x resident blocks x warps per block
    (nb, s, sw, units), = planner([(slots, bands_of(8192), 8192)])
    assert (nb, s, sw, units) == (137, 17, 22, 2339)


def test_plan_invariants(planner):
    cases = []
    for slots in (64, 608, 2432, 4864):
        for nx in (1, 7, 60, 61, 300, 2048, 8192, 20000):
            for ny in (1, 2, 9, 31, 33, 150, 1000, 2048, 8192):
                cases.append((slots, bands_of(nx), ny))
    for (slots, nbands, ny), (nb, s, sw, units) in zip(cases, planner(cases)):
        nw = 2 if nbands > 1 else 1
        assert nb == nbands
        assert 1 <= s <= sw, (slots, nbands, ny, s, sw)
        assert units == nbands * s + nw * (sw - s)
        # one wave whenever every band fits in the warp slots
        if nbands * 1 + nw * 0 <= slots:
            assert units <= slots or sw == s == 1, (slots, nbands, ny, units)
        # segment length: at least the minimum (8 rows on grids too small to
        # fill a quarter of the slots, else 32; half of it in wall bands)
        min_rows = 8 if nbands * (ny // 32) * 4 <= slots else 32
        if s > 1:
            assert ny // s >= min_rows, (slots, nbands, ny, s)
        if sw > 1 and sw > s:
            assert ny // sw >= min_rows // 2, (slots, nbands, ny, sw)
