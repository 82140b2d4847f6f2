// Tile arithmetic of the narrow-segment grouped GEMM (gemm_narrow.cuh): how an expert's rows are
// cut into chunks (the MMA's N) and which TMA boxes bring one CTA's half of a chunk.  Plain C++ so
// that the host tests can check it (every row of every expert covered once per weight tile, N a
// multiple of 16 within the chunk limit, the boxes inside the row buffer).
#pragma once

#ifdef __CUDACC__
#define MOK_HD __host__ __device__ __forceinline__
#else
#define MOK_HD inline
#endif

namespace mok {

// One CTA's rows of X arrive as 64-row TMA boxes (8 KB) and at most one 32-row box (the last box
// may run into the next expert's rows, which only feed accumulator columns that are not stored).
// The copies cost per box, not only per byte: with 16-row boxes (up to 17 boxes per stage) GEMM2
// and dX_g at the DSV3 layer took 1.81 and 3.71 ms, with 32-row boxes 1.64 and 3.10 ms, and a
// 16-row box for an odd tail made them slower again (1.68 and 3.31 ms).
constexpr int NARROW_XBOX = 64;
constexpr int NARROW_XBOX_S = 32;

// Boxes for `half` rows: n64 boxes of 64 rows, then one of 32 if `with32`; returns the rows loaded.
MOK_HD int narrow_x_boxes(int half, int& n64, bool& with32) {
  n64 = half >> 6;
  int rem = half & 63;
  if (rem > NARROW_XBOX_S) {
    ++n64;
    rem = 0;
  }
  with32 = rem > 0;
  return n64 * NARROW_XBOX + (with32 ? NARROW_XBOX_S : 0);
}

struct NarrowTile {
  int e, c, m;
  int nc;    // row chunks of this expert (they share each weight tile)
  int row0;  // first row of the chunk
  int rows;  // rows of the chunk (1..nmax)
  int n;     // MMA N: rows rounded up to 16
};

// Rows per chunk of an expert with `cnt` rows cut into `nc` chunks of at most `nmax`: the equal
// share rounded up to 16 (so only the last chunk pads), or nmax where that would leave the last
// chunk empty.
MOK_HD int narrow_chunk(int cnt, int nc, int nmax) {
  int ch = ((cnt + nc - 1) / nc + 15) & ~15;
  if ((nc - 1) * ch >= cnt) ch = nmax;
  return ch;
}

// Expert e owns tiles [s_coff[e]*MT, s_coff[e+1]*MT) with s_coff the prefix of ceil(rows/nmax);
// inside an expert the chunks of one weight tile are neighbours, so the pairs that run them at
// the same time read that weight tile from HBM once.
template <typename CoffT>
MOK_HD NarrowTile decode_narrow_tile(int g, int MT, int E, int nmax, const int* s_off, const CoffT* s_coff) {
  int lo = 0, hi = E;  // largest e with s_coff[e]*MT <= g (the last of equal starts owns tiles)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int)s_coff[mid] * MT <= g) lo = mid; else hi = mid;
  }
  NarrowTile t;
  t.e = lo;
  const int nc = (int)s_coff[lo + 1] - (int)s_coff[lo];
  const int cnt = s_off[lo + 1] - s_off[lo];
  const int local = g - (int)s_coff[lo] * MT;
  t.nc = nc;
  t.m = local / nc;
  t.c = local - t.m * nc;
  const int ch = narrow_chunk(cnt, nc, nmax);
  t.row0 = s_off[lo] + t.c * ch;
  t.rows = (ch < cnt - t.c * ch ? ch : cnt - t.c * ch);
  t.n = (t.rows + 15) & ~15;
  return t;
}

}  // namespace mok
