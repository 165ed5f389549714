// Per-sequence geometry and the mask predicate shared by the host planner and
// the device kernels of the HSTU forward.
//
// Mask ("RecOps Running Case Documentation", feature table "Support causal mask"
// and the Inputs and Outputs table rows num_context / num_target / mask_type /
// target_group_size): causal over the history, context rows see the whole
// history, target rows see the history plus the earlier targets of their own
// group of target_group_size, and target_group_size 0 builds no target mask.
// Written out, with H = (g > 0) ? max(L - nt, 0) : L:
//   valid(i, j) = (j <= i && j < H) || (i < nc && j < H)
//              || (g > 0 && i >= H && j >= H && j <= i && (i - H) / g == (j - H) / g)
//              || (g == 0 && j <= i)
// For one row this is the union of a prefix [0, hist_end) and a range
// [grp_lo, i] (the row's own target group), which is how the kernels test it.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define HSTU_HD __host__ __device__ __forceinline__
#else
#define HSTU_HD inline
#endif

namespace hstu {

constexpr int kMaskCausal = 0;
constexpr int kMaskNone = 2;
constexpr int kTileM = 128;  // query rows per work item (tensor-core path)
constexpr int kTileN = 128;  // key/value rows per pipeline step (tensor-core path)
constexpr int kMaxMTiles = 1024;  // work-list packing: m-tile index in 10 bits

// One sequence as the kernels see it.
struct SeqGeom {
  int L;   // length
  int nc;  // num_context clamped to [0, L]
  int H;   // history end: targets occupy [H, L)
  int g;   // target group size (0 = no target mask)
};

HSTU_HD SeqGeom make_geom(int L, long long nc_raw, long long nt_raw, int g, int mask_type) {
  SeqGeom s;
  s.L = L;
  if (mask_type == kMaskNone) {
    s.nc = 0;
    s.H = L;
    s.g = 0;
    return s;
  }
  long long nc = nc_raw < 0 ? 0 : (nc_raw > L ? L : nc_raw);
  long long nt = nt_raw < 0 ? 0 : (nt_raw > L ? L : nt_raw);
  s.nc = (int)nc;
  s.g = g > 0 ? g : 0;
  s.H = s.g > 0 ? (int)(L - nt) : L;
  return s;
}

// Valid columns of row i: [0, hist_end) U [grp_lo, grp_hi], all < L.
struct RowRange {
  int hist_end;
  int grp_lo;
  int grp_hi;  // grp_lo > grp_hi means no group range
};

HSTU_HD RowRange row_range(const SeqGeom& s, int i, int mask_type) {
  RowRange r;
  if (mask_type == kMaskNone) {
    r.hist_end = s.L;
    r.grp_lo = 1;
    r.grp_hi = 0;
    return r;
  }
  int he = (i < s.nc) ? s.H : (i + 1 < s.H ? i + 1 : s.H);
  if (s.g == 0 && i + 1 > he) he = i + 1;  // no target mask: plain causal (H = L here)
  r.hist_end = he < s.L ? he : s.L;
  if (s.g > 0 && i >= s.H && i < s.L) {
    r.grp_lo = s.H + ((i - s.H) / s.g) * s.g;
    r.grp_hi = i;
  } else {
    r.grp_lo = 1;
    r.grp_hi = 0;
  }
  return r;
}

HSTU_HD bool valid_in_range(const RowRange& r, int j) {
  return j < r.hist_end || (j >= r.grp_lo && j <= r.grp_hi);
}

// End (exclusive) of the key range any row in [m0, m0 + rows) of the sequence
// may attend. Keys at or beyond it are masked for every such row.
HSTU_HD int kv_end_for_rows(const SeqGeom& s, int m0, int rows, int mask_type) {
  if (mask_type == kMaskNone) return s.L;
  int last = m0 + rows;  // exclusive
  if (last > s.L) last = s.L;
  int e = last;  // causal part: row i sees at most j <= i
  if (m0 < s.nc && s.H > e) e = s.H;  // context rows see the whole history
  return e < s.L ? e : s.L;
}

// True when every (i, j) with i in [m0, m0 + rows), j in [n0, n0 + cols) is valid
// (so the tile needs no per-element mask). Conservative: false is always safe.
HSTU_HD bool tile_all_valid(const SeqGeom& s, int m0, int rows, int n0, int cols,
                            int mask_type) {
  const int jmax = n0 + cols - 1;
  if (jmax >= s.L) return false;
  if (mask_type == kMaskNone) return true;
  if (jmax < s.H && jmax <= m0) return true;       // causal history block below the diagonal
  if (m0 + rows - 1 < s.nc && jmax < s.H) return true;  // context rows
  return false;
}

// Number of leading key tiles of cols columns (from key 0) for which tile_all_valid holds
// for the rows [m0, m0 + rows): those tiles form a prefix. Tile n is all valid when its last
// key n*cols + cols - 1 lies below L and, with a causal mask, below H and at or below m0
// (or, for context rows only, below H): that is n*cols + cols <= E for the E below.
HSTU_HD int full_tiles(const SeqGeom& s, int m0, int rows, int cols, int mask_type) {
  int e = s.L;
  if (mask_type != kMaskNone) {
    if (s.H < e) e = s.H;
    if (!(m0 + rows - 1 < s.nc) && m0 + 1 < e) e = m0 + 1;
  }
  return e > 0 ? e / cols : 0;
}

HSTU_HD int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Key tiles of one work item when the keys are a cached history of `hist` positions
// followed by new rows. Key tile x covers positions [128x, 128x + 128). A tile in which
// the history ends and new rows begin is visited twice, first with its cached rows
// (columns [0, hist % 128)), then with its new rows (columns [hist % 128, 128)), so that
// every visit loads one run of rows of one tensor. split_tile is that tile, or -1.
HSTU_HD int split_tile(int hist, int Lk) {
  return (hist % kTileN != 0 && hist < Lk) ? hist / kTileN : -1;
}

// Visits of an item whose keys end (for its rows) at kv_end.
HSTU_HD int key_visits(int kv_end, int split) {
  const int n = ceil_div(kv_end, kTileN);
  return n + ((split >= 0 && split < n) ? 1 : 0);
}

struct KeyTile {
  int x;         // key tile: positions [128x, 128x + 128)
  int clo, chi;  // columns of the tile this visit covers
  bool cached;   // rows come from the cache (else from k / v)
};

HSTU_HD KeyTile key_tile(int j, int split, int hist) {
  KeyTile t;
  const bool second = split >= 0 && j == split + 1;  // new-row part of the split tile
  t.x = (split >= 0 && j > split) ? j - 1 : j;
  t.clo = second ? hist % kTileN : 0;
  t.chi = j == split ? hist % kTileN : kTileN;
  t.cached = !second && t.x * kTileN < hist;
  return t;
}

HSTU_HD uint32_t pack_item(int b, int mt) { return ((uint32_t)b << 10) | (uint32_t)mt; }
HSTU_HD int item_b(uint32_t e) { return (int)(e >> 10); }
HSTU_HD int item_mt(uint32_t e) { return (int)(e & 1023u); }

}  // namespace hstu
