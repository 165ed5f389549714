"""Host build of the tile geometry the kernels and the work-list builder share
(csrc/common.cuh), checked by a small C++ program compiled with g++. CPU only.

  * full_tiles (the kernels' count of leading key tiles that need no mask) equals the
    number of leading tiles for which tile_all_valid holds, and those tiles are a prefix
    (no mask-free tile after the first masked one), for random lengths, context and
    target counts, group sizes and both mask types;
  * tile_all_valid is conservative: a tile it calls all valid has every (i, j) valid under
    the per-row predicate (row_range / valid_in_range), checked element by element;
  * kv_end_for_rows bounds the keys: no row of the tile sees a key at or beyond it.
"""
import os
import subprocess

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "hstu_dense_forward_gb300", "csrc")

PROGRAM = r'''
#include <cstdio>
#include <cstdlib>
#include "common.cuh"
using namespace hstu;
int main() {
  long bad = 0, n = 0, tiles = 0;
  unsigned s = 12345u;
  auto rnd = [&](int m) { s = s * 1103515245u + 12345u; return (int)((s >> 8) % (unsigned)m); };
  for (int it = 0; it < 30000; ++it) {
    const int L = rnd(700), nc = rnd(200) - 10, nt = rnd(260) - 10, g = rnd(20) - 2;
    const int mt = rnd(2) ? kMaskCausal : kMaskNone;
    const SeqGeom geo = make_geom(L, nc, nt, g, mt);
    for (int m0 = 0; m0 < L; m0 += kTileM) {
      int nf = 0;
      while (tile_all_valid(geo, m0, kTileM, nf * kTileN, kTileN, mt)) ++nf;
      const int kv_end = kv_end_for_rows(geo, m0, kTileM, mt);
      for (int j = 0; j * kTileN < L + kTileN; ++j) {
        const bool all = tile_all_valid(geo, m0, kTileM, j * kTileN, kTileN, mt);
        if (all != (j < nf)) { ++bad; printf("prefix broken L=%d m0=%d j=%d\n", L, m0, j); }
        if (all) {  // element by element, the tile really is all valid
          ++tiles;
          for (int i = m0; i < m0 + kTileM; ++i) {
            const RowRange r = row_range(geo, i, mt);
            for (int c = j * kTileN; c < (j + 1) * kTileN; ++c)
              if (i < L && !valid_in_range(r, c)) { ++bad; break; }
          }
        }
      }
      for (int i = m0; i < m0 + kTileM && i < L; ++i) {  // no key beyond kv_end is visible
        const RowRange r = row_range(geo, i, mt);
        for (int c = kv_end; c < L; ++c)
          if (valid_in_range(r, c)) { ++bad; break; }
      }
      if (full_tiles(geo, m0, kTileM, kTileN, mt) != nf) {
        ++bad;
        if (bad < 5) printf("full_tiles L=%d nc=%d H=%d g=%d mt=%d m0=%d: %d vs %d\n", L, geo.nc,
                            geo.H, geo.g, mt, m0, full_tiles(geo, m0, kTileM, kTileN, mt), nf);
      }
      ++n;
    }
  }
  printf("checked %ld item geometries, %ld mask-free tiles, mismatches %ld\n", n, tiles, bad);
  return bad != 0;
}
'''


def test_tile_geometry_host_build(tmp_path):
    src = tmp_path / "geometry.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "geometry"
    subprocess.check_call(["g++", "-std=c++17", "-O2", "-I", CSRC, "-o", str(exe), str(src)])
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches 0" in r.stdout
