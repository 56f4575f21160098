// swe_mesh_prep.cpp -- host preparation of a triangle mesh for the edge and
// cell kernels of swe_mesh.cu.
//
// Geometry of An MPI-CUDA implementation of an improved Roe method for
// two-layer shallow water systems, Sec. 2.2: per volume V_i its area |V_i|;
// per edge Gamma_ij its length and the unit normal eta_ij pointing from V_i
// to V_j; an edge owned by one triangle only is a wall.  All of it is
// computed here in double precision from the vertex coordinates.
//
// Cell order: the Hilbert curve through the cell centroids (on a 2^16 x 2^16
// lattice over the bounding square), so that any run of consecutive cells is
// a compact patch of the mesh.  The order is then cut into tiles (runs of
// consecutive cells, see swe_internal.h) whose edges, cells and halo fit the
// tile kernel's shared memory; a compact patch keeps its border, and so the
// edges evaluated twice and the halo cells loaded, short.
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <new>
#include <utility>
#include <vector>

#include "swe_internal.h"

namespace swe {
namespace {

// Position of lattice point (x, y), 0 <= x, y < 2^16, along the Hilbert
// curve of order 16: at each level the quadrant of (x, y) adds its rank
// times the quadrant size, then (x, y) is taken into that quadrant's own
// frame (the lower quadrants are transposed, the lower-right one also
// mirrored), so the next level sees the standard curve again.
uint64_t hilbert_rank(uint32_t x, uint32_t y) {
  uint64_t d = 0;
  for (uint32_t s = 1u << 15; s > 0; s >>= 1) {
    const uint32_t rx = (x & s) ? 1u : 0u;
    const uint32_t ry = (y & s) ? 1u : 0u;
    d += (uint64_t)s * s * ((3u * rx) ^ ry);
    if (ry == 0) {
      if (rx == 1) {
        x = ~x;
        y = ~y;
      }
      const uint32_t t = x;
      x = y;
      y = t;
    }
    x &= s - 1;
    y &= s - 1;
  }
  return d;
}

// Cells sorted by the Hilbert rank of their centroid (ties by caller index).
void hilbert_order(const double* xy, const int32_t* tri, int64_t nc, std::vector<int32_t>& order) {
  std::vector<double> cx((size_t)nc), cy((size_t)nc);
  double x0 = INFINITY, x1 = -INFINITY, y0 = INFINITY, y1 = -INFINITY;
  for (int64_t c = 0; c < nc; ++c) {
    const int32_t* v = tri + 3 * c;
    cx[c] = (xy[2 * v[0]] + xy[2 * v[1]] + xy[2 * v[2]]) / 3.0;
    cy[c] = (xy[2 * v[0] + 1] + xy[2 * v[1] + 1] + xy[2 * v[2] + 1]) / 3.0;
    x0 = std::min(x0, cx[c]);
    x1 = std::max(x1, cx[c]);
    y0 = std::min(y0, cy[c]);
    y1 = std::max(y1, cy[c]);
  }
  double span = std::max(x1 - x0, y1 - y0);
  if (!(span > 0.0)) span = 1.0;
  const double q = 65535.0 / span;
  auto lat = [&](double v) {
    const double t = floor(v * q);
    return (uint32_t)(t < 0.0 ? 0.0 : (t > 65535.0 ? 65535.0 : t));
  };
  std::vector<std::pair<uint64_t, int32_t>> key((size_t)nc);
  for (int64_t c = 0; c < nc; ++c)
    key[c] = {hilbert_rank(lat(cx[c] - x0), lat(cy[c] - y0)), (int32_t)c};
  std::sort(key.begin(), key.end());
  order.resize((size_t)nc);
  for (int64_t c = 0; c < nc; ++c) order[c] = key[c].second;
}

// Cuts the internal order into tiles and lays out their slots, halo lists
// and per-cell slot references.  Cells are taken greedily: a cell joins the
// current tile unless the tile would then exceed kTileSlots - 1 slots (one
// is kept for the even padding), kTileCells cells, kTileHalo halo cells or
// kTileCap cells plus halo cells.
void build_tiles(MeshPrep* out) {
  const int64_t nc = out->ncells;
  const std::vector<int32_t>& ref = out->ref;
  auto other = [&](int64_t c, int k) {  // the cell across edge k of c, -1 on a wall
    const int32_t r = ref[(size_t)k * nc + c];
    const int32_t e = r >> 1;
    return (r & 1) ? out->ea[e] : out->eb[e];
  };
  // pass 1: tile boundaries
  std::vector<int32_t> in_halo((size_t)nc, -1);  // tile that has the cell in its halo
  out->tile_cell.clear();
  out->tile_cell.push_back(0);
  int32_t tile = 0;
  int64_t c0 = 0, ns = 0, nh = 0;
  for (int64_t c = 0; c < nc; ++c) {
    for (int attempt = 0; attempt < 2; ++attempt) {
      int64_t ds = 0, dh = (in_halo[c] == tile) ? -1 : 0;
      int32_t seen[3];
      int nseen = 0;
      for (int k = 0; k < 3; ++k) {
        const int32_t j = other(c, k);
        if (j >= c0 && j < c) continue;  // inside the tile: slot already counted
        ++ds;
        if (j < 0 || in_halo[j] == tile) continue;
        bool dup = false;
        for (int i = 0; i < nseen; ++i) dup |= seen[i] == j;
        if (!dup) {
          seen[nseen++] = j;
          ++dh;
        }
      }
      const bool fits = ns + ds <= kTileSlots - 1 && nh + dh <= kTileHalo &&
                        c - c0 + 1 <= kTileCells && (c - c0 + 1) + nh + dh <= kTileCap;
      if (!fits && attempt == 0 && c > c0) {  // close the tile, retry c in a new one
        out->tile_cell.push_back((int32_t)c);
        ++tile;
        c0 = c;
        ns = 0;
        nh = 0;
        continue;
      }
      ns += ds;
      nh += dh;
      for (int i = 0; i < nseen; ++i) in_halo[seen[i]] = tile;
      break;
    }
  }
  out->tile_cell.push_back((int32_t)nc);
  const int64_t nt = (int64_t)out->tile_cell.size() - 1;
  out->ntiles = nt;

  // pass 2: halo lists, slots (tile-major, even starts) and cell references
  out->tile_halo.assign((size_t)nt + 1, 0);
  out->tile_slot.assign((size_t)nt + 1, 0);
  out->halo.clear();
  out->slot_ab.clear();
  out->slot_nx.clear();
  out->slot_ny.clear();
  out->slot_len.clear();
  out->cref.assign((size_t)(2 * nc), 0u);
  out->edge_evals = 0;
  std::vector<int32_t> hpos((size_t)nc, -1), hstamp((size_t)nc, -1);
  std::vector<int32_t> slot_of_edge((size_t)out->nedges, -1);
  for (int64_t t = 0; t < nt; ++t) {
    const int64_t a0 = out->tile_cell[t], a1 = out->tile_cell[t + 1];
    const int64_t nct = a1 - a0;
    out->tile_halo[t] = (int32_t)out->halo.size();
    out->tile_slot[t] = (int32_t)out->slot_ab.size();
    const int64_t sbase = (int64_t)out->slot_ab.size();
    auto local = [&](int32_t x) -> int32_t {
      if (x >= a0 && x < a1) return (int32_t)(x - a0);
      if (hstamp[x] != (int32_t)t) {
        hstamp[x] = (int32_t)t;
        hpos[x] = (int32_t)(out->halo.size() - out->tile_halo[t]);
        out->halo.push_back(x);
      }
      return (int32_t)(nct + hpos[x]);
    };
    uint16_t cr[3];
    for (int64_t c = a0; c < a1; ++c) {
      for (int k = 0; k < 3; ++k) {
        const int32_t r = ref[(size_t)k * nc + c];
        const int32_t e = r >> 1, side = r & 1;
        const int32_t j = side ? out->ea[e] : out->eb[e];
        int32_t s;
        if (j >= a0 && j < c) {
          s = slot_of_edge[e];  // made by j, earlier in this tile
        } else {
          s = (int32_t)((int64_t)out->slot_ab.size() - sbase);
          slot_of_edge[e] = s;
          const int32_t la = local(out->ea[e]);
          const int32_t lb = out->eb[e] < 0 ? kTileWall : local(out->eb[e]);
          out->slot_ab.push_back(la | (lb << 16));
          out->slot_nx.push_back(out->enx[e]);
          out->slot_ny.push_back(out->eny[e]);
          out->slot_len.push_back(out->elen[e]);
        }
        cr[k] = (uint16_t)(s | (side << 15));
      }
      out->cref[2 * c] = (uint32_t)cr[0] | ((uint32_t)cr[1] << 16);
      out->cref[2 * c + 1] = (uint32_t)cr[2];
    }
    const int64_t n = (int64_t)out->slot_ab.size() - sbase;
    out->edge_evals += n;
    if (n & 1) {  // even padding: a copy of the last slot, referenced by no cell
      out->slot_ab.push_back(out->slot_ab.back());
      out->slot_nx.push_back(out->slot_nx.back());
      out->slot_ny.push_back(out->slot_ny.back());
      out->slot_len.push_back(out->slot_len.back());
    }
  }
  out->tile_halo[nt] = (int32_t)out->halo.size();
  out->tile_slot[nt] = (int32_t)out->slot_ab.size();
}

// Consistency of the tiles with the edges they were cut from: every cell's
// three references name a slot of its own tile whose side is the cell and
// whose other side is the neighbour across that edge (or a wall), with the
// edge's normal and length; the limits of the tile kernel hold.  O(n).
bool tiles_consistent(const MeshPrep& m) {
  const int64_t nc = m.ncells, nt = m.ntiles;
  if (nt < 1 || (int64_t)m.tile_cell.size() != nt + 1 || m.tile_cell[0] != 0 ||
      m.tile_cell[nt] != nc)
    return false;
  for (int64_t t = 0; t < nt; ++t) {
    const int64_t c0 = m.tile_cell[t], c1 = m.tile_cell[t + 1];
    const int64_t h0 = m.tile_halo[t], nh = m.tile_halo[t + 1] - h0;
    const int64_t s0 = m.tile_slot[t], ns = m.tile_slot[t + 1] - s0;
    const int64_t nct = c1 - c0;
    if (nct < 1 || nct > kTileCells || nh < 0 || nh > kTileHalo || nct + nh > kTileCap ||
        (s0 & 1) || (ns & 1) || ns < 2 ||
        ns > kTileSlots)
      return false;
    auto global = [&](int32_t l) -> int64_t {
      if (l < nct) return c0 + l;
      if (l - nct >= nh) return -2;
      return m.halo[h0 + l - nct];
    };
    for (int64_t c = c0; c < c1; ++c) {
      for (int k = 0; k < 3; ++k) {
        const uint32_t w = k < 2 ? (m.cref[2 * c] >> (16 * k)) & 0xffffu : m.cref[2 * c + 1];
        const int64_t sl = w & 0x7fffu;
        const int side = (int)(w >> 15);
        const int32_t r = m.ref[(size_t)k * nc + c];
        const int32_t e = r >> 1;
        if (sl >= ns || side != (r & 1)) return false;
        const int32_t ab = m.slot_ab[s0 + sl];
        const int32_t la = ab & 0xffff, lb = (ab >> 16) & 0xffff;
        if (global(la) != m.ea[e]) return false;
        if (m.eb[e] < 0 ? lb != kTileWall : global(lb) != m.eb[e]) return false;
        if ((side ? global(lb) : global(la)) != c) return false;
        if (m.slot_nx[s0 + sl] != m.enx[e] || m.slot_ny[s0 + sl] != m.eny[e] ||
            m.slot_len[s0 + sl] != m.elen[e])
          return false;
      }
    }
  }
  return true;
}

}  // namespace

int prepare_mesh(int64_t nv, const double* xy, int64_t nc, const int32_t* tri, bool reorder,
                 MeshPrep* out) {
  try {
    for (int64_t i = 0; i < 2 * nv; ++i)
      if (!isfinite(xy[i])) return -1;
    for (int64_t i = 0; i < 3 * nc; ++i)
      if (tri[i] < 0 || tri[i] >= nv) return -1;
    auto head = [&](int64_t he) { return tri[he]; };
    auto tail = [&](int64_t he) { return tri[he - he % 3 + (he % 3 + 1) % 3]; };

    // areas (shoelace; counter-clockwise triangles are positive)
    std::vector<double> area((size_t)nc);
    for (int64_t c = 0; c < nc; ++c) {
      const int32_t* v = tri + 3 * c;
      const double x0 = xy[2 * v[0]], y0 = xy[2 * v[0] + 1];
      const double x1 = xy[2 * v[1]], y1 = xy[2 * v[1] + 1];
      const double x2 = xy[2 * v[2]], y2 = xy[2 * v[2] + 1];
      area[c] = 0.5 * ((x1 - x0) * (y2 - y0) - (x2 - x0) * (y1 - y0));
      if (!(area[c] > 0.0) || !isfinite(area[c])) return -1;
    }

    // half-edges leaving each vertex (CSR), then each half-edge's twin
    const int64_t nh = 3 * nc;
    std::vector<int64_t> start((size_t)nv + 1, 0);
    for (int64_t h = 0; h < nh; ++h) ++start[head(h) + 1];
    for (int64_t v = 0; v < nv; ++v) start[v + 1] += start[v];
    std::vector<int64_t> fill(start.begin(), start.end() - 1);
    std::vector<int64_t> out_he((size_t)nh);
    for (int64_t h = 0; h < nh; ++h) out_he[fill[head(h)]++] = h;
    std::vector<int32_t> nbr((size_t)nh, -1);  // neighbour cell across half-edge h (old ids)
    std::vector<int64_t> twin((size_t)nh, -1);
    for (int64_t h = 0; h < nh; ++h) {
      const int32_t u = head(h), v = tail(h);
      for (int64_t s = start[u]; s < start[u + 1]; ++s)
        if (out_he[s] != h && tail(out_he[s]) == v) return -1;  // u -> v used twice
      for (int64_t s = start[v]; s < start[v + 1]; ++s)
        if (tail(out_he[s]) == u) {
          twin[h] = out_he[s];
          break;
        }
      if (twin[h] >= 0) nbr[h] = (int32_t)(twin[h] / 3);
    }

    // cell order
    out->ncells = nc;
    out->new_of_old.assign((size_t)nc, 0);
    out->old_of_new.assign((size_t)nc, 0);
    if (reorder) {
      hilbert_order(xy, tri, nc, out->old_of_new);
    } else {
      for (int64_t c = 0; c < nc; ++c) out->old_of_new[c] = (int32_t)c;
    }
    for (int64_t c = 0; c < nc; ++c) out->new_of_old[out->old_of_new[c]] = (int32_t)c;

    // edges in order of their first cell a (internal numbering)
    int64_t nb = 0;
    for (int64_t h = 0; h < nh; ++h) nb += twin[h] < 0;
    const int64_t ne = (nh + nb) / 2;
    out->nedges = ne;
    out->ea.resize((size_t)ne);
    out->eb.resize((size_t)ne);
    out->enx.resize((size_t)ne);
    out->eny.resize((size_t)ne);
    out->elen.resize((size_t)ne);
    out->ref.assign((size_t)(3 * nc), -1);
    out->inv_area.resize((size_t)nc);
    int64_t e = 0;
    for (int64_t c = 0; c < nc; ++c) {
      const int64_t o = out->old_of_new[c];
      out->inv_area[c] = 1.0 / area[o];
      for (int k = 0; k < 3; ++k) {
        const int64_t h = 3 * o + k;
        int32_t j = -1;
        if (twin[h] >= 0) {
          j = out->new_of_old[nbr[h]];
          if (j < c) continue;  // stored by cell j
        }
        const int32_t u = head(h), v = tail(h);
        const double ex = xy[2 * v] - xy[2 * u], ey = xy[2 * v + 1] - xy[2 * u + 1];
        const double l = sqrt(ex * ex + ey * ey);
        out->ea[e] = (int32_t)c;
        out->eb[e] = j;
        out->enx[e] = ey / l;  // outward normal of a counter-clockwise edge
        out->eny[e] = -ex / l;
        out->elen[e] = l;
        out->ref[(size_t)k * nc + c] = (int32_t)(2 * e);
        if (j >= 0) out->ref[(size_t)(twin[h] % 3) * nc + j] = (int32_t)(2 * e + 1);
        ++e;
      }
    }
    if (e != ne) return -1;
    for (int64_t i = 0; i < 3 * nc; ++i)
      if (out->ref[i] < 0) return -1;
    build_tiles(out);
    if (!tiles_consistent(*out)) return -2;
    return 0;
  } catch (const std::bad_alloc&) {
    return -3;
  }
}

}  // namespace swe
