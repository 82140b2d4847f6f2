"""Host checks of the weight-gradient pair kernel's work items (csrc/wgrad_items.h), compiled with
g++ against the same header the kernel includes.

For random launches (expert counts, strips per expert, strip lengths odd and even, any number of
long experts) the order in which the pairs take items must be a permutation of the items; every
output tile of every expert must be covered by exactly one item (a long expert's items are one
or two neighbouring tiles of one strip, another expert's items whole strips); each of the two
lists keeps its own order in the merged one, and after any number of positions the long items
taken are exactly their even share (floor(p * L / total)).
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
#include "wgrad_items.h"
using namespace mok;

static int fail(const char* what, long a, long b) {
  std::printf("FAIL %s %ld %ld\n", what, a, b);
  return 1;
}

static int check(int per_e, int strip_len, int n_long, int E) {
  const WgpItems w = wgp_items(per_e, strip_len, n_long, E);
  const int L = w.n_tile_items;
  if (w.total != n_long * per_e * ((strip_len + 1) / 2) + (E - n_long) * per_e) return fail("total", w.total, 0);
  std::vector<int> taken(w.total, 0);
  std::vector<int> tiles((size_t)E * per_e * strip_len, 0);
  int last_long = -1, last_short = -1, longs = 0;
  for (int pos = 0; pos < w.total; ++pos) {
    const int n = wgp_item_at(w, pos);
    if (n < 0 || n >= w.total) return fail("range", pos, n);
    if (taken[n]++) return fail("twice", pos, n);
    if (n < L) {
      if (n != last_long + 1) return fail("long order", pos, n);
      last_long = n;
      ++longs;
    } else {
      if (n != last_short + 1 && !(last_short < 0 && n == L)) return fail("short order", pos, n);
      last_short = n;
    }
    if ((long long)longs != (long long)(pos + 1) * L / w.total) return fail("spread", pos, longs);
    int le, f, i0, i1;
    wgp_item(w, n, le, f, i0, i1);
    if (le < 0 || le >= E || f < 0 || f >= per_e) return fail("item", n, le);
    if (n < L) {
      if (le >= n_long || i0 % 2 != 0 || i1 - i0 < 1 || i1 - i0 > 2 || i1 > strip_len) return fail("long item", n, i0);
      if (i1 - i0 == 1 && i1 != strip_len) return fail("single tile inside a strip", n, i0);
    } else {
      if (le < n_long || i0 != 0 || i1 != strip_len) return fail("strip item", n, le);
    }
    for (int i = i0; i < i1; ++i) ++tiles[((size_t)le * per_e + f) * strip_len + i];
  }
  for (size_t t = 0; t < tiles.size(); ++t)
    if (tiles[t] != 1) return fail("coverage", (long)t, tiles[t]);
  return 0;
}

int main() {
  std::mt19937 rng(2024);
  int checked = 0;
  // the DSV3 layer's shapes: dW13 (16 strips of 28 tiles), dW2 (8 strips of 28)
  const int shapes[][2] = {{16, 28}, {28, 16}, {8, 28}, {28, 8}, {1, 1}, {3, 5}, {2, 3}, {5, 1}};
  for (auto& s : shapes)
    for (int E : {1, 2, 16, 47, 256, 300})
      for (int n_long : {0, 1, E / 5, E / 2, E - 1, E}) {
        if (n_long < 0 || n_long > E) continue;
        if (check(s[0], s[1], n_long, E)) return 1;
        ++checked;
      }
  for (int trial = 0; trial < 2000; ++trial) {
    const int E = 1 + (int)(rng() % 400);
    const int per_e = 1 + (int)(rng() % 30);
    const int strip_len = 1 + (int)(rng() % 30);
    const int n_long = (int)(rng() % (E + 1));
    if (check(per_e, strip_len, n_long, E)) return 1;
    ++checked;
  }
  std::printf("OK %d\n", checked);
  return 0;
}
"""


def test_wgrad_item_arithmetic(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    src = tmp_path / "wgrad_items_check.cpp"
    exe = tmp_path / "wgrad_items_check"
    src.write_text(HARNESS)
    subprocess.run([gxx, "-O2", "-std=c++17", "-I", CSRC, str(src), "-o", str(exe)], check=True,
                   capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.startswith("OK"), r.stdout + r.stderr
