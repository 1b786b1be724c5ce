// Host check of the grouped GEMMs' tile walk (decode_tile in csrc/moe_tile.cuh,
// compiled here for the CPU): for random group sizes, with and without the
// shared group, in the plain and the interleaved order, every (group, row
// tile, column tile) is named by exactly one linear tile index; the
// interleaved order marks exactly the sparse groups' tiles as streamed and
// keeps the dense : sparse ratio in every window of consecutive indices.
// The prefix arrays are built from their definition (the dispatch scan's):
// tile_off counts 128-row tiles over all groups, tile_doff over the groups of
// at least dense_mt row tiles, tile_soff over the others.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <random>
#include <vector>

#include "moe_tile.cuh"

using moe::GemmParams;
using moe::TileInfo;

static int fails = 0;
#define CHECK(c, ...)                              \
  do {                                             \
    if (!(c)) {                                    \
      if (fails < 20) std::printf(__VA_ARGS__);    \
      ++fails;                                     \
    }                                              \
  } while (0)

static void run_case(const std::vector<int>& counts, int T_shared, int n_tiles, int dense_mt,
                     bool interleave, int window) {
  const int E = static_cast<int>(counts.size());
  const int G = E + (T_shared > 0 ? 1 : 0);
  std::vector<int> rows(counts);
  if (T_shared > 0) rows.push_back(T_shared);
  std::vector<int> row_off(G + 1, 0), toff(G + 1, 0), doff(G + 1, 0), soff(G + 1, 0), mt(G);
  for (int g = 0; g < G; ++g) {
    mt[g] = (rows[g] + moe::kBM - 1) / moe::kBM;
    row_off[g + 1] = row_off[g] + rows[g];
    toff[g + 1] = toff[g] + mt[g];
    doff[g + 1] = doff[g] + (mt[g] >= dense_mt ? mt[g] : 0);
    soff[g + 1] = toff[g + 1] - doff[g + 1];
  }
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.row_off = row_off.data();
  p.tile_off = toff.data();
  p.num_groups = G;
  p.shared_group = T_shared > 0 ? E : -1;
  p.n_tiles = n_tiles;
  if (interleave) {
    p.tile_doff = doff.data();
    p.tile_soff = soff.data();
  }
  const long long total = static_cast<long long>(toff[G]) * n_tiles;
  const long long nd = static_cast<long long>(doff[G]) * n_tiles;
  std::vector<std::vector<int>> seen(G);
  for (int g = 0; g < G; ++g) seen[g].assign(static_cast<size_t>(mt[g]) * n_tiles, 0);
  std::vector<int> dense_at(static_cast<size_t>(total), 0);
  int prev_g = -1, prev_m = -1, prev_n = -1;
  for (long long i = 0; i < total; ++i) {
    const TileInfo t = moe::decode_tile(p, static_cast<int>(i));
    CHECK(t.group >= 0 && t.group < G, "tile %lld: group %d of %d\n", i, t.group, G);
    if (t.group < 0 || t.group >= G) continue;
    const int g = t.group;
    CHECK(t.m >= 0 && t.m < mt[g] && t.n >= 0 && t.n < n_tiles, "tile %lld: m %d n %d (group %d: %d x %d)\n",
          i, t.m, t.n, g, mt[g], n_tiles);
    if (t.m < 0 || t.m >= mt[g] || t.n < 0 || t.n >= n_tiles) continue;
    ++seen[g][static_cast<size_t>(t.n) * mt[g] + t.m];
    CHECK(t.row0 == row_off[g] + t.m * moe::kBM && t.row_end == row_off[g + 1] && t.row0 < t.row_end,
          "tile %lld: rows [%d, %d)\n", i, t.row0, t.row_end);
    CHECK(t.second == (g == p.shared_group), "tile %lld: shared flag\n", i);
    const bool dense = mt[g] >= dense_mt;
    if (interleave) {
      // streamed = the sparse list's tiles (all tiles when no group is dense)
      CHECK(t.stream == (!dense || doff[G] == 0) && !(doff[G] == toff[G] && t.stream),
            "tile %lld: stream %d for a group of %d row tiles\n", i, t.stream, mt[g]);
    } else {
      CHECK(!t.stream, "tile %lld: streamed in the plain walk\n", i);
      // plain walk: inside a group, row tiles fastest, then column tiles
      if (g == prev_g) {
        const bool next = (t.n == prev_n && t.m == prev_m + 1) || (t.n == prev_n + 1 && t.m == 0 && prev_m == mt[g] - 1);
        CHECK(next, "tile %lld: (%d, %d) after (%d, %d)\n", i, t.m, t.n, prev_m, prev_n);
      } else {
        CHECK(g > prev_g && t.m == 0 && t.n == 0, "tile %lld: group %d starts at (%d, %d)\n", i, g, t.m, t.n);
      }
    }
    prev_g = g;
    prev_m = t.m;
    prev_n = t.n;
    dense_at[static_cast<size_t>(i)] = dense ? 1 : 0;
  }
  for (int g = 0; g < G; ++g)
    for (size_t j = 0; j < seen[g].size(); ++j)
      CHECK(seen[g][j] == 1, "group %d tile %zu named %d times\n", g, j, seen[g][j]);
  if (interleave && nd > 0 && nd < total) {
    // every window of `window` consecutive indices holds floor or ceil of its share
    long long run = 0;
    for (long long i = 0; i < total; ++i) {
      run += dense_at[static_cast<size_t>(i)];
      if (i >= window) run -= dense_at[static_cast<size_t>(i - window)];
      if (i + 1 >= window) {
        const double share = static_cast<double>(window) * nd / total;
        CHECK(run >= static_cast<long long>(share) - 1 && run <= static_cast<long long>(share) + 2,
              "window ending at %lld: %lld dense, share %.2f\n", i, run, share);
      }
    }
  }
}

int main() {
  std::mt19937 rng(20240611u);
  int cases = 0;
  for (int trial = 0; trial < 600; ++trial) {
    const int E = 1 + static_cast<int>(rng() % 48);
    std::vector<int> counts(E);
    const int mode = trial % 4;  // mixed, all single-tile, all multi-tile, with empty groups
    for (int e = 0; e < E; ++e) {
      int n = static_cast<int>(rng() % 700);
      if (mode == 1) n = 1 + static_cast<int>(rng() % 128);
      if (mode == 2) n = 129 + static_cast<int>(rng() % 600);
      if (mode == 3 && rng() % 3 == 0) n = 0;
      counts[e] = n;
    }
    const int T_shared = (trial % 3 == 0) ? static_cast<int>(rng() % 600) : 0;
    const int n_tiles = 1 + static_cast<int>(rng() % 24);
    const int dense_mt = 1 + static_cast<int>(rng() % 4);
    long long rows = T_shared;
    for (int n : counts) rows += n;
    if (rows == 0) continue;
    run_case(counts, T_shared, n_tiles, dense_mt, false, 152);
    run_case(counts, T_shared, n_tiles, dense_mt, true, 152);
    cases += 2;
  }
  std::printf("%d cases, %d failures\n", cases, fails);
  return fails == 0 ? 0 : 1;
}
