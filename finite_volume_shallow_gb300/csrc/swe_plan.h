// swe_plan.h -- host-side launch planning of the one-layer step kernel,
// shared by the simulation handle and the allocation-free entry point.
#pragma once

#include <stdint.h>

namespace swe {

// Launch shape of the one-layer step: one warp per (band, row segment),
// every band cut into nsegs segments, the first and the last band (whose
// warps also handle the side walls, a slower code path) into nsegs_wall
// shorter ones, so that all warps of the single wave finish together.  No
// segment is shorter than 32 rows, 16 in the wall bands (each segment
// re-reads four halo rows), unless the grid is so small that even then it
// would fill less than a quarter of the warp slots: then 8 rows.
#ifndef SWE_WALL_EXTRA_PCT
#define SWE_WALL_EXTRA_PCT 25
#endif
#ifndef SWE_MIN_SEG_ROWS
#define SWE_MIN_SEG_ROWS 32
#endif
struct StepPlan {
  int nbands, nsegs, nsegs_wall, units;
};
inline StepPlan plan_step(int64_t slots, int64_t nbands, int64_t ny) {
  StepPlan p;
  p.nbands = (int)nbands;
  const int64_t min_rows =
      nbands * (ny / SWE_MIN_SEG_ROWS) * 4 <= slots ? 8 : SWE_MIN_SEG_ROWS;
  const int64_t most = ny / min_rows > 1 ? ny / min_rows : 1;
  int64_t S = slots / nbands;
  if (S > most) S = most;
  if (S < 1) S = 1;
  const int64_t nw = nbands > 1 ? 2 : 1;
  int64_t Sw = (S * (100 + SWE_WALL_EXTRA_PCT) + 99) / 100;
  int64_t most_wall = ny / (min_rows / 2) > 1 ? ny / (min_rows / 2) : 1;  // half as long
  if (most_wall < most) most_wall = most;
  if (Sw > most_wall) Sw = most_wall;
  while (Sw > S && nbands * S + nw * (Sw - S) > slots) --Sw;
  if (Sw < S) Sw = S;
  p.nsegs = (int)S;
  p.nsegs_wall = (int)Sw;
  p.units = (int)(nbands * S + nw * (Sw - S));
  return p;
}

}  // namespace swe
