// Tile and layout arithmetic of the block-scaled MXFP8 grouped GEMMs (gemm_mx.cuh) and of the
// kernels that prepare their operands.  Plain C++ so that the host tests can check it.
//
// Row operands (the dispatched rows, the SwiGLU output) are E4M3 in a padded row space: expert e
// owns rows [32 blk_off[e], 32 blk_off[e+1]) with blk_off the prefix of ceil(rows / 32), its rows in
// schedule order followed by zero rows.  Their scales (one E8M0 byte per row and 32 K-elements)
// are kept in the order tcgen05.cp 32x128b.warpx4 copies into TMEM: a 512-byte block holds 128
// rows x 4 K-blocks, row 32 j + l and K-block b at byte 16 l + 4 j + b, so that in TMEM row n of
// the block sits in column n / 32, lane n % 32 (of every lane quarter) and K-block b in byte b.
// A weight matrix [Nw][K] has one such block per 128-row tile and 128-element K stage.  For the
// row operands, whose chunks start at any multiple of 32 rows, block (g, s) holds rows
// 32 g .. 32 g + 127 (so every row's scales are stored in the four blocks g = row / 32 - 3 .. row / 32)
// and a chunk starting at row 32 g0 reads blocks g0, g0 + 4, ...
#pragma once

#include "narrow_tiles.h"  // MOK_HD

namespace mok {

constexpr int MX_ROW_ALIGN = 32;   // expert rows padded to a multiple of this
constexpr int MX_BK = 128;         // K elements (bytes of E4M3) per pipeline stage
constexpr int MX_SF_BLOCK = 512;   // scale block: 128 rows x 4 K-blocks of 32

// Byte of (row r, K-block kb) inside its scale block; r is the row within the block (0..127) and
// kb the K-block within the stage (0..3).
MOK_HD int mx_sf_byte(int r, int kb) { return (r & 31) * 16 + ((r >> 5) & 3) * 4 + (kb & 3); }

// Upper bound of the padded rows of R rows in E experts, and of the row groups of their scales
// (a chunk at the last group reads up to four groups further).
MOK_HD long long mx_rows_padded_bound(long long R, int E) { return 32LL * ((R + 31) / 32 + E); }
MOK_HD long long mx_row_groups(long long R, int E) { return mx_rows_padded_bound(R, E) / 32 + 4; }

struct MxTile {
  int e, m, c;
  int nc;     // row chunks of this expert (they share each weight tile)
  int row0;   // first (schedule-order) row of the chunk
  int prow0;  // its padded row (a multiple of 32)
  int rows;   // rows of the chunk (1..nmax)
  int nload;  // rows loaded: rows rounded up to 32 (zero rows past the expert's end)
  int n;      // MMA N: rows rounded up to 16
};

// Rows per chunk of an expert with `cnt` rows cut into `nc` chunks of at most `nmax` (a multiple
// of 32): the equal share rounded up to 32, so that every chunk starts on a 32-row boundary of the
// padded space and only the last one is short.
MOK_HD int mx_chunk(int cnt, int nc, int nmax) {
  int ch = ((cnt + nc - 1) / nc + 31) & ~31;
  if ((nc - 1) * ch >= cnt) ch = nmax;
  return ch;
}

// Expert e owns tiles [s_coff[e]*MT, s_coff[e+1]*MT), s_coff the prefix of ceil(rows / nmax);
// chunks of one weight tile are neighbours (c fastest, then the weight tile m).
MOK_HD MxTile decode_mx_tile(int g, int MT, int E, int nmax, const int* s_off, const int* s_boff, const int* s_coff) {
  int lo = 0, hi = E;  // largest e with s_coff[e]*MT <= g (the last of equal starts owns tiles)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_coff[mid] * MT <= g) lo = mid; else hi = mid;
  }
  MxTile t;
  t.e = lo;
  const int nc = s_coff[lo + 1] - s_coff[lo];
  const int cnt = s_off[lo + 1] - s_off[lo];
  const int local = g - s_coff[lo] * MT;
  t.nc = nc;
  t.m = local / nc;
  t.c = local - t.m * nc;
  const int ch = mx_chunk(cnt, nc, nmax);
  t.row0 = s_off[lo] + t.c * ch;
  t.prow0 = MX_ROW_ALIGN * s_boff[lo] + t.c * ch;
  t.rows = (ch < cnt - t.c * ch ? ch : cnt - t.c * ch);
  t.nload = (t.rows + 31) & ~31;
  t.n = (t.rows + 15) & ~15;
  return t;
}

}  // namespace mok
