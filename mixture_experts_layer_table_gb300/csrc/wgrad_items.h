// Work-item arithmetic of the weight-gradient pair kernel (wgrad_pair.cuh): which output tiles an
// item covers and in which order the pairs take the items.  Plain C++ so that the host tests can
// check it (every output tile of every expert covered exactly once, the merged order a
// permutation with the long experts' items spread evenly).
#pragma once

#ifdef __CUDACC__
#define MOK_WI_HD __host__ __device__ __forceinline__
#else
#define MOK_WI_HD inline
#endif

namespace mok {

// The items of one launch over E experts, of which the first n_long in the expert list (s_list)
// have more rows than the stationary region holds.  Output tiles are 256 x 256: per_e stationary
// strips per expert, strip_len tiles along a strip.
//  * a long expert's item: two neighbouring tiles (i, i + 1) of one strip (the last item of a
//    strip of odd length has one), pairs_f items per strip, tiles_e per expert;
//  * another expert's item: one whole strip.
struct WgpItems {
  int per_e, strip_len, n_long, E;
  int pairs_f, tiles_e, n_tile_items, total;
};

MOK_WI_HD WgpItems wgp_items(int per_e, int strip_len, int n_long, int E) {
  WgpItems w;
  w.per_e = per_e;
  w.strip_len = strip_len;
  w.n_long = n_long;
  w.E = E;
  w.pairs_f = (strip_len + 1) / 2;
  w.tiles_e = per_e * w.pairs_f;
  w.n_tile_items = n_long * w.tiles_e;
  w.total = w.n_tile_items + (E - n_long) * per_e;
  return w;
}

// Item n (long items first, then the strips, each list in expert-list order) -> the index le of
// its expert in s_list, its strip f and its tiles [i0, i1).
MOK_WI_HD void wgp_item(const WgpItems& w, int n, int& le, int& f, int& i0, int& i1) {
  if (n < w.n_tile_items) {
    le = n / w.tiles_e;
    const int local = n - le * w.tiles_e;
    f = local / w.pairs_f;
    i0 = 2 * (local - f * w.pairs_f);
    i1 = i0 + 2 < w.strip_len ? i0 + 2 : w.strip_len;
  } else {
    const int b = n - w.n_tile_items;
    const int se = b / w.per_e;
    le = w.n_long + se;
    f = b - se * w.per_e;
    i0 = 0;
    i1 = w.strip_len;
  }
}

// Position pos of the order the pairs take items in: the two lists merged with the long items
// spread evenly among the strips (position pos is the k-th long item when floor(pos * L / total)
// steps up to k + 1 there, L = n_tile_items), each list keeping its own order.
MOK_WI_HD int wgp_item_at(const WgpItems& w, int pos) {
  const long long nl0 = (long long)pos * w.n_tile_items / w.total;
  const long long nl1 = (long long)(pos + 1) * w.n_tile_items / w.total;
  return nl1 > nl0 ? (int)nl0 : w.n_tile_items + (pos - (int)nl0);
}

}  // namespace mok
