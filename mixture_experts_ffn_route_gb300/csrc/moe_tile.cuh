// Tile walk of the persistent grouped GEMMs: which group, row tile and column
// tile a linear tile index names.  Host-callable as well, so that the walk can
// be checked on the CPU against the tile counts it is given.
#pragma once

#include "moe_internal.h"

namespace moe {

// Read-only load: through the non-coherent cache on the device.
__host__ __device__ __forceinline__ int ld_ro(const int* p) {
#ifdef __CUDA_ARCH__
  return __ldg(p);
#else
  return *p;
#endif
}

struct TileInfo {
  int group, m, n;
  int row0, row_end;  // output rows [row0, row_end) of this tile's group
  int a_row0;         // first A row fetched for this tile
  bool second;        // uses the second (shared-expert) tensor maps
  bool stream;        // a sparse group's tile in the interleaved order
};

// Largest g in [0, G) with off[g] * n_tiles <= j (groups without tiles share
// their start with the next group, so the search lands on the one holding j).
__host__ __device__ __forceinline__ int find_group(const int* off, int G, int n_tiles, long long j) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<long long>(ld_ro(off + mid)) * n_tiles <= j) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Tile order: group by group; inside a group, column tile by column tile, and
// the 128-row tiles of one column tile consecutively.  CTAs running at the
// same time then share one weight column block through L2 while the group's
// rows (the smaller operand) stay resident, so each weight byte is read from
// HBM about once even when a group spans many row tiles.
//
// Interleaved order (tile_doff set): the same walk is taken separately over the
// dense groups (a list of nd tiles) and over the others, and linear index i is
// the dense list's floor(i nd / total)-th tile when that floor steps up at i,
// else the sparse list's (i - floor(i nd / total))-th.  Every window of
// consecutive indices, hence every set of CTAs running at the same time, then
// holds the two lists in the ratio nd : total - nd, so the dense groups'
// tensor-bound tiles overlap the sparse groups' HBM-bound weight stream
// instead of running in phases of their own.
__host__ __device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, int tile) {
  TileInfo t;
  t.stream = false;
  if (p.row_off == nullptr) {
    const int mt = (p.dense_rows + kBM - 1) / kBM;
    t.group = 0;
    t.n = tile / mt;
    t.m = tile - t.n * mt;
    t.row0 = t.m * kBM;
    t.row_end = p.dense_rows;
  } else {
    const int G = p.num_groups;
    const int* off = p.tile_off;
    long long j = tile;
    if (p.tile_doff != nullptr) {
      const int mt_all = ld_ro(p.tile_off + G), mt_dense = ld_ro(p.tile_doff + G);
      if (mt_dense == 0) {
        t.stream = true;  // all sparse: the plain walk, every tile streamed
      } else if (mt_dense < mt_all) {
        const long long total = static_cast<long long>(mt_all) * p.n_tiles;
        const long long nd = static_cast<long long>(mt_dense) * p.n_tiles;
        const long long d0 = j * nd / total;
        if ((j + 1) * nd / total > d0) {
          off = p.tile_doff;
          j = d0;
        } else {
          off = p.tile_soff;
          j -= d0;
          t.stream = true;
        }
      }  // all dense: the plain walk
    }
    const int g = find_group(off, G, p.n_tiles, j);
    const int t0 = ld_ro(off + g);
    const int mt = ld_ro(off + g + 1) - t0;
    const int local = static_cast<int>(j - static_cast<long long>(t0) * p.n_tiles);
    t.group = g;
    t.n = local / mt;
    t.m = local - t.n * mt;
    t.row0 = ld_ro(p.row_off + g) + t.m * kBM;
    t.row_end = ld_ro(p.row_off + g + 1);
  }
  t.second = (t.group == p.shared_group);
  t.a_row0 = (t.second && p.a2_shared) ? t.m * kBM : t.row0;
  return t;
}

}  // namespace moe
