"""Host checks of the MXFP8 grouped GEMM's tile and layout arithmetic (csrc/mx_tiles.h), compiled
with g++ against the same header the kernels include.

For random expert row counts (empty experts, ragged and long segments, one expert, many experts)
and every chunk limit: decoding every tile index must cover each row of each expert exactly once
per weight tile, with chunks of 1..nmax rows that start on a 32-row boundary of the padded row
space, load whole 32-row groups inside the expert's padded rows, and have the MMA's N the row count
rounded up to 16; the padded rows and the scale row-groups a chunk reads stay inside the bounds the
workspace is sized by.  The scale-block byte map is a bijection, and the row-group form the
writers use (row p stored in the four blocks p/32 - 3 .. p/32) reads back through it.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "mixture_experts_layer_table_gb300", "csrc")

HARNESS = r"""
#include <cstdio>
#include <random>
#include <vector>
#include "mx_tiles.h"
using namespace mok;

static int fail(const char* what, int a, int b) {
  std::printf("FAIL %s %d %d\n", what, a, b);
  return 1;
}

static int check(const std::vector<int>& counts, int MT, int nmax) {
  const int E = (int)counts.size();
  std::vector<int> off(E + 1, 0), boff(E + 1, 0), coff(E + 1, 0);
  for (int e = 0; e < E; ++e) {
    off[e + 1] = off[e] + counts[e];
    boff[e + 1] = boff[e] + (counts[e] + 31) / 32;          // as mx_block_offsets computes it
    coff[e + 1] = coff[e] + (counts[e] + nmax - 1) / nmax;  // as the kernel builds s_coff
  }
  const int R = off[E];
  if (32LL * boff[E] > mx_rows_padded_bound(R, E)) return fail("padded bound", R, boff[E]);
  const long long G = mx_row_groups(R, E);
  const int total = coff[E] * MT;
  std::vector<int> seen((size_t)R * MT, 0);
  int prev_e = -1, prev_m = -1, prev_c = -1;
  for (int g = 0; g < total; ++g) {
    const MxTile t = decode_mx_tile(g, MT, E, nmax, off.data(), boff.data(), coff.data());
    if (t.e < 0 || t.e >= E || counts[t.e] == 0) return fail("expert", g, t.e);
    if (t.m < 0 || t.m >= MT || t.c < 0 || t.c >= t.nc) return fail("indices", g, t.m);
    if (t.rows < 1 || t.rows > nmax) return fail("rows", g, t.rows);
    if (t.n % 16 != 0 || t.n < t.rows || t.n - t.rows >= 16) return fail("n", g, t.n);
    if (t.nload % 32 != 0 || t.nload < t.n || t.nload - t.rows >= 32 || t.nload > nmax) return fail("nload", g, t.nload);
    if (t.row0 < off[t.e] || t.row0 + t.rows > off[t.e + 1]) return fail("segment", g, t.row0);
    if (t.prow0 % 32 != 0 || t.prow0 - 32 * boff[t.e] != t.row0 - off[t.e]) return fail("padded row", g, t.prow0);
    if (t.prow0 + t.nload > 32 * boff[t.e + 1]) return fail("padded segment", g, t.prow0 + t.nload);
    const int nsfb = (t.nload + 127) / 128;
    if (t.prow0 / 32 + 4 * (nsfb - 1) >= G) return fail("scale groups", g, t.prow0);
    if (t.c + 1 < t.nc && t.rows % 32 != 0) return fail("chunk padding", g, t.rows);
    if (t.e == prev_e) {
      const bool next_chunk = t.m == prev_m && t.c == prev_c + 1;
      const bool next_tile = t.m == prev_m + 1 && t.c == 0 && prev_c == t.nc - 1;
      if (!next_chunk && !next_tile) return fail("order", g, t.c);
    } else if (t.m != 0 || t.c != 0) {
      return fail("expert start", g, t.m);
    }
    prev_e = t.e;
    prev_m = t.m;
    prev_c = t.c;
    for (int r = t.row0; r < t.row0 + t.rows; ++r) ++seen[(size_t)r * MT + t.m];
  }
  for (size_t i = 0; i < seen.size(); ++i)
    if (seen[i] != 1) return fail("coverage", (int)(i / MT), seen[i]);
  return 0;
}

int main() {
  // the scale-block byte map: a bijection of 128 rows x 4 K-blocks onto 512 bytes
  std::vector<int> hit(MX_SF_BLOCK, 0);
  for (int r = 0; r < 128; ++r)
    for (int kb = 0; kb < 4; ++kb) ++hit[mx_sf_byte(r, kb)];
  for (int b = 0; b < MX_SF_BLOCK; ++b)
    if (hit[b] != 1) return fail("sf bijection", b, hit[b]);
  // row p of the padded space sits in block p/32 - jj at local row 32 jj + p % 32, which is where the
  // writers put it, byte 16 (p % 32) + 4 jj + kb; a chunk starting at group g0 finds row n of the
  // chunk in its block b = n / 128 at local row n % 128
  for (int p = 0; p < 4096; ++p)
    for (int jj = 0; jj < 4; ++jj)
      for (int kb = 0; kb < 4; ++kb)
        if (mx_sf_byte(32 * jj + p % 32, kb) != 16 * (p % 32) + 4 * jj + kb) return fail("row groups", p, jj);
  for (int g0 = 0; g0 < 64; ++g0)
    for (int n = 0; n < 256; ++n) {
      const int p = 32 * g0 + n, b = n / 128, jj = p / 32 - (g0 + 4 * b);
      if (jj < 0 || jj > 3 || mx_sf_byte(n % 128, 0) != 16 * (p % 32) + 4 * jj) return fail("chunk read", g0, n);
    }
  std::mt19937 rng(2468);
  const int nmaxes[3] = {128, 192, 256};
  int checked = 0;
  for (int trial = 0; trial < 400; ++trial) {
    const int E = 1 + (int)(rng() % 300);
    const int scale = (int)std::vector<int>{3, 40, 140, 300, 700, 3000}[rng() % 6];
    std::vector<int> counts(E);
    for (int& c : counts) c = (int)(rng() % (scale + 1));
    if (rng() % 3 == 0)
      for (int z = 0; z < E / 2; ++z) counts[rng() % E] = 0;
    const int MT = 1 + (int)(rng() % 30);
    for (int nm : nmaxes) {
      if (check(counts, MT, nm)) return 1;
      ++checked;
    }
  }
  for (int cnt = 0; cnt <= 5000; ++cnt)
    for (int nm : nmaxes) {
      if (check(std::vector<int>{cnt}, 3, nm)) return 1;
      ++checked;
    }
  std::printf("OK %d\n", checked);
  return 0;
}
"""


def test_mx_tile_arithmetic(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    src = tmp_path / "mx_tiles_check.cpp"
    exe = tmp_path / "mx_tiles_check"
    src.write_text(HARNESS)
    subprocess.run([gxx, "-O2", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True,
                   capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.startswith("OK"), r.stdout + r.stderr
