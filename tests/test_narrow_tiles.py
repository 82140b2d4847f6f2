"""Host checks of the narrow-segment GEMM's tile arithmetic (csrc/narrow_tiles.h), compiled with
g++ against the same header the kernel includes.

For random expert row counts (empty experts, ragged and long segments, one expert, many experts)
and every chunk limit the kernel instantiates, decoding every tile index must give: each row of
each expert covered exactly once per weight tile, chunks of 1..nmax rows with the MMA's N the row
count rounded up to 16 (only an expert's last chunk padded), the chunks of one weight tile
adjacent in the tile order, and TMA boxes that bring at least the CTA's rows and stay inside its
row buffer (nmax / 2 rows).
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "mixture_experts_layer_table_gb300", "csrc")

HARNESS = r"""
#include <cstdio>
#include <cstdlib>
#include <random>
#include <vector>
#include "narrow_tiles.h"
using namespace mok;

static int fail(const char* what, int a, int b) {
  std::printf("FAIL %s %d %d\n", what, a, b);
  return 1;
}

static int check(const std::vector<int>& counts, int MT, int nmax) {
  const int E = (int)counts.size();
  std::vector<int> off(E + 1, 0), coff(E + 1, 0);
  for (int e = 0; e < E; ++e) {
    off[e + 1] = off[e] + counts[e];
    coff[e + 1] = coff[e] + (counts[e] + nmax - 1) / nmax;  // as the kernel builds s_coff
  }
  const int R = off[E];
  const int total = coff[E] * MT;
  std::vector<int> seen((size_t)R * MT, 0);
  int prev_e = -1, prev_m = -1, prev_c = -1;
  for (int g = 0; g < total; ++g) {
    const NarrowTile t = decode_narrow_tile(g, MT, E, nmax, off.data(), coff.data());
    if (t.e < 0 || t.e >= E || counts[t.e] == 0) return fail("expert", g, t.e);
    if (t.m < 0 || t.m >= MT || t.c < 0 || t.c >= t.nc) return fail("indices", g, t.m);
    if (t.rows < 1 || t.rows > nmax) return fail("rows", g, t.rows);
    if (t.n % 16 != 0 || t.n < t.rows || t.n - t.rows >= 16 || t.n > nmax) return fail("n", g, t.n);
    if (t.row0 < off[t.e] || t.row0 + t.rows > off[t.e + 1]) return fail("segment", g, t.row0);
    // only an expert's last chunk pads: the others hold a multiple of 16 rows
    if (t.c + 1 < t.nc && t.rows % 16 != 0) return fail("chunk padding", g, t.rows);
    // tile order: expert, then weight tile, then chunk (chunks of one weight tile adjacent)
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
    // each CTA of the pair stages n / 2 rows; its boxes bring at least those and fit its buffer
    int n64 = 0;
    bool with32 = false;
    const int half = t.n / 2;
    const int loaded = narrow_x_boxes(half, n64, with32);
    if (loaded < half || loaded > nmax / 2 || loaded != n64 * NARROW_XBOX + (with32 ? NARROW_XBOX_S : 0))
      return fail("boxes", g, loaded);
  }
  for (size_t i = 0; i < seen.size(); ++i)
    if (seen[i] != 1) return fail("coverage", (int)(i / MT), seen[i]);
  return 0;
}

int main() {
  std::mt19937 rng(12345);
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


def test_narrow_tile_arithmetic(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    src = tmp_path / "narrow_tiles_check.cpp"
    exe = tmp_path / "narrow_tiles_check"
    src.write_text(HARNESS)
    subprocess.run([gxx, "-O2", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True,
                   capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.startswith("OK"), r.stdout + r.stderr
