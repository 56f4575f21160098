// swe_mesh_prep.cpp -- host preparation of a triangle mesh for the edge and
// cell kernels of swe_mesh.cu.
//
// Geometry of An MPI-CUDA implementation of an improved Roe method for
// two-layer shallow water systems, Sec. 2.2: per volume V_i its area |V_i|;
// per edge Gamma_ij its length and the unit normal eta_ij pointing from V_i
// to V_j; an edge owned by one triangle only is a wall.  All of it is
// computed here in double precision from the vertex coordinates.
//
// Cell order: reverse Cuthill-McKee on the cell adjacency graph (breadth-
// first from a pseudo-peripheral cell, neighbours visited by increasing
// degree, then reversed), so that the two cells of an edge, and the edges of
// a cell, sit close together in memory; the gathers of the edge and cell
// kernels then mostly hit in L2.
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <new>
#include <vector>

#include "swe_internal.h"

namespace swe {
namespace {

struct Graph {
  const std::vector<int32_t>* nbr;  // 3 per cell, -1 on walls
  std::vector<uint8_t> deg;
};

// Breadth-first levels from r over the cell adjacency; returns the
// eccentricity of r and leaves the last level in `last`.
int bfs_levels(const Graph& G, int32_t r, std::vector<int32_t>& level, std::vector<int32_t>& queue,
               std::vector<int32_t>& last) {
  const std::vector<int32_t>& nbr = *G.nbr;
  queue.clear();
  queue.push_back(r);
  level[r] = 0;
  int ecc = 0;
  for (size_t head = 0; head < queue.size(); ++head) {
    const int32_t u = queue[head];
    for (int k = 0; k < 3; ++k) {
      const int32_t v = nbr[3 * (size_t)u + k];
      if (v >= 0 && level[v] < 0) {
        level[v] = level[u] + 1;
        ecc = std::max(ecc, level[v]);
        queue.push_back(v);
      }
    }
  }
  last.clear();
  for (int32_t u : queue)
    if (level[u] == ecc) last.push_back(u);
  for (int32_t u : queue) level[u] = -1;  // reset for the next search
  return ecc;
}

// George-Liu style pseudo-peripheral cell of the component of seed.
int32_t pseudo_peripheral(const Graph& G, int32_t seed, std::vector<int32_t>& level,
                          std::vector<int32_t>& queue) {
  std::vector<int32_t> last;
  int32_t r = seed;
  int ecc = bfs_levels(G, r, level, queue, last);
  for (int it = 0; it < 16; ++it) {
    int32_t x = last[0];
    for (int32_t u : last)
      if (G.deg[u] < G.deg[x] || (G.deg[u] == G.deg[x] && u < x)) x = u;
    std::vector<int32_t> last2;
    const int e2 = bfs_levels(G, x, level, queue, last2);
    if (e2 <= ecc) break;
    r = x;
    ecc = e2;
    last.swap(last2);
  }
  return r;
}

// Cuthill-McKee order of every component, concatenated, then reversed.
void rcm_order(const std::vector<int32_t>& nbr, int64_t nc, std::vector<int32_t>& order) {
  Graph G{&nbr, std::vector<uint8_t>((size_t)nc)};
  for (int64_t c = 0; c < nc; ++c) {
    int d = 0;
    for (int k = 0; k < 3; ++k) d += nbr[3 * c + k] >= 0;
    G.deg[c] = (uint8_t)d;
  }
  std::vector<int32_t> level((size_t)nc, -1), queue;
  queue.reserve((size_t)nc);
  std::vector<uint8_t> seen((size_t)nc, 0);
  order.clear();
  order.reserve((size_t)nc);
  for (int d = 0; d <= 3; ++d)
    for (int64_t c0 = 0; c0 < nc; ++c0) {
      if (G.deg[c0] != d || seen[c0]) continue;
      const int32_t start = pseudo_peripheral(G, (int32_t)c0, level, queue);
      size_t head = order.size();
      order.push_back(start);
      seen[start] = 1;
      for (; head < order.size(); ++head) {
        const int32_t u = order[head];
        int32_t nb[3];
        int n = 0;
        for (int k = 0; k < 3; ++k) {
          const int32_t v = nbr[3 * (size_t)u + k];
          if (v >= 0 && !seen[v]) {
            seen[v] = 1;
            nb[n++] = v;
          }
        }
        std::sort(nb, nb + n, [&](int32_t x, int32_t y) {
          return G.deg[x] != G.deg[y] ? G.deg[x] < G.deg[y] : x < y;
        });
        for (int i = 0; i < n; ++i) order.push_back(nb[i]);
      }
    }
  std::reverse(order.begin(), order.end());
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
      rcm_order(nbr, nc, out->old_of_new);
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
    return 0;
  } catch (const std::bad_alloc&) {
    return -3;
  }
}

}  // namespace swe
