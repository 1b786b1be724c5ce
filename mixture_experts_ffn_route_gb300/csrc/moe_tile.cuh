// Tile walk of the persistent grouped GEMMs: which group, row tile and column
// tile a linear tile index names.
#pragma once

#include "moe_internal.h"

namespace moe {

struct TileInfo {
  int group, m, n;
  int row0, row_end;  // output rows [row0, row_end) of this tile's group
  int a_row0;         // first A row fetched for this tile
  bool second;        // uses the second (shared-expert) tensor maps
};

// Tile order: group by group; inside a group, column tile by column tile, and
// the 128-row tiles of one column tile consecutively.  CTAs running at the
// same time then share one weight column block through L2 while the group's
// rows (the smaller operand) stay resident, so each weight byte is read from
// HBM about once even when a group spans many row tiles.
__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, int tile) {
  TileInfo t;
  if (p.row_off == nullptr) {
    const int mt = (p.dense_rows + kBM - 1) / kBM;
    t.group = 0;
    t.n = tile / mt;
    t.m = tile - t.n * mt;
    t.row0 = t.m * kBM;
    t.row_end = p.dense_rows;
  } else {
    // largest g with tile_off[g] * n_tiles <= tile (groups without tiles share
    // their start with the next group)
    int lo = 0, hi = p.num_groups - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(p.tile_off + mid) * p.n_tiles <= tile) lo = mid; else hi = mid - 1;
    }
    const int t0 = __ldg(p.tile_off + lo);
    const int mt = __ldg(p.tile_off + lo + 1) - t0;
    const int local = tile - t0 * p.n_tiles;
    t.group = lo;
    t.n = local / mt;
    t.m = local - t.n * mt;
    t.row0 = __ldg(p.row_off + lo) + t.m * kBM;
    t.row_end = __ldg(p.row_off + lo + 1);
  }
  t.second = (t.group == p.shared_group);
  t.a_row0 = (t.second && p.a2_shared) ? t.m * kBM : t.row0;
  return t;
}

}  // namespace moe
