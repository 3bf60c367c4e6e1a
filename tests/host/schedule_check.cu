// Host-side check of the persistent GEMMs' work schedule (no GPU needed):
//   * tile_coords maps the tile indices 0 .. num_m*num_n-1 one-to-one onto
//     the (row tile, column tile) grid for every raster setting in use;
//   * chunk_span splits Nk kept rows into chunks that cover [0, Nk) in order,
//     each at most chunk_rows long;
//   * work_schedule / SegIter, walked for every worker as the kernels walk
//     them, cover every (tile, K block) once: the tiles of the whole waves in
//     one unit each, the tiles of a split tail in `split` parts (2 ..
//     max_split) whose slots run 0 .. split-1 in K order; a split tail takes
//     fewer tile-times than the unsplit one, and nothing but dHidden splits;
//   * the 512-column tiles of the CTA-pair kernel (raster over wide tiles,
//     then their two 256-column blocks) cover every 256-column tile once --
//     a block past the last one only when their count is odd;
//     dh_reduce_kernel, which counts the tiles as row tiles x ceil(H / 512)
//     and walks them row-major, sees the kernel's tiles.
// Prints "ok" and exits 0, or names the first failing case and exits 1.
#include <cstdio>
#include <vector>

#include "../../sft_keep_mask_gb300/csrc/tc_common.cuh"

using namespace lmhead;

static int check_raster(int num_m, int num_n, int group_m, int group_n) {
  std::vector<int> seen(static_cast<size_t>(num_m) * num_n, 0);
  for (int t = 0; t < num_m * num_n; ++t) {
    int mt = -1, nt = -1;
    tile_coords(t, num_m, num_n, group_m, group_n, mt, nt);
    if (mt < 0 || mt >= num_m || nt < 0 || nt >= num_n) {
      std::printf("raster out of range: M=%d N=%d gm=%d gn=%d t=%d -> (%d,%d)\n", num_m, num_n,
                  group_m, group_n, t, mt, nt);
      return 1;
    }
    if (seen[static_cast<size_t>(mt) * num_n + nt]++) {
      std::printf("raster repeats a tile: M=%d N=%d gm=%d gn=%d t=%d\n", num_m, num_n, group_m,
                  group_n, t);
      return 1;
    }
  }
  return 0;
}

// Every worker's units, walked as the kernels walk them.
static int check_schedule(int tiles, int workers, int num_kb, bool may_split, int max_split,
                          int fill_pct) {
  const WorkSched s = work_schedule(tiles, workers, num_kb, may_split, max_split, fill_pct);
  char name[160];
  std::snprintf(name, sizeof name, "schedule(T=%d W=%d Kb=%d split=%d S=%d fill=%d)", tiles,
                workers, num_kb, may_split ? 1 : 0, max_split, fill_pct);
  const int rem = tiles - s.full;
  if (s.workers != workers || s.full < 0 || s.full > tiles || s.split < 1 ||
      (s.split == 1) != (rem == 0) || (s.split > 1 && (!may_split || s.split > max_split ||
                                                        s.split > num_kb || rem >= workers))) {
    std::printf("%s: full %d split %d\n", name, s.full, s.split);
    return 1;
  }
  if (s.split > 1) {
    // the split tail: ceil(rem * split / W) rounds of 1/split of a tile-time
    const long long rounds = (static_cast<long long>(rem) * s.split + workers - 1) / workers;
    if (rounds >= s.split) {
      std::printf("%s: a tail of %d tiles in %d parts takes %lld rounds\n", name, rem, s.split,
                  rounds);
      return 1;
    }
  }
  const size_t cells = static_cast<size_t>(tiles) * (num_kb > 0 ? num_kb : 1);
  std::vector<int> cover(cells, 0);
  std::vector<int> seen(static_cast<size_t>(tiles), 0), last_kb(static_cast<size_t>(tiles), -1);
  int units = 0;
  for (int w = 0; w < workers; ++w) {
    SegIter it(s, w);
    int nseg = 0;
    for (WorkSeg g; it.next(g); ++nseg, ++units) {
      const bool bad_range = num_kb > 0 ? (g.kb0 < 0 || g.kb0 >= g.kb1 || g.kb1 > num_kb)
                                        : (g.kb0 != 0 || g.kb1 != 0);
      if (g.tile < 0 || g.tile >= tiles || bad_range || g.slots != s.tile_slots(g.tile) ||
          g.slot < 0 || g.slot >= g.slots || (g.slots == 1 && (g.kb0 != 0 || g.kb1 != num_kb))) {
        std::printf("%s: worker %d unit %d: tile %d K [%d, %d) slot %d of %d\n", name, w, nseg,
                    g.tile, g.kb0, g.kb1, g.slot, g.slots);
        return 1;
      }
      const size_t t = static_cast<size_t>(g.tile);
      seen[t] |= 1 << g.slot;
      for (int kb = g.kb0; kb < (num_kb > 0 ? g.kb1 : 1); ++kb)
        ++cover[t * (num_kb > 0 ? num_kb : 1) + kb];
      // slot p covers the p-th part of the K range
      if (num_kb > 0 && g.kb0 != static_cast<int>(static_cast<long long>(g.slot) * num_kb / g.slots)) {
        std::printf("%s: tile %d slot %d starts at K block %d\n", name, g.tile, g.slot, g.kb0);
        return 1;
      }
    }
  }
  if (units != s.units()) {
    std::printf("%s: %d units walked, %d scheduled\n", name, units, s.units());
    return 1;
  }
  for (size_t i = 0; i < cells; ++i)
    if (cover[i] != 1) {
      std::printf("%s: (tile, K block) %zu covered %d times\n", name, i, cover[i]);
      return 1;
    }
  for (int t = 0; t < tiles; ++t)
    if (seen[static_cast<size_t>(t)] != (1 << s.tile_slots(t)) - 1) {
      std::printf("%s: tile %d parts do not run 0 .. %d\n", name, t, s.tile_slots(t) - 1);
      return 1;
    }
  return 0;
}

// The 512-column tiles of the CTA-pair kernel, walked as it walks them.
static int check_wide_tiles(int num_m, int num_n, int group_m, int group_n) {
  const int num_nw = (num_n + 1) / 2;   // 512-column tiles over num_n 256-column tiles
  const int num_tiles = num_m * num_nw;
  std::vector<int> seen(static_cast<size_t>(num_m) * num_n, 0);
  for (int u = 0; u < num_tiles; ++u) {
    int mt = -1, ntw = -1;
    tile_coords(u, num_m, num_nw, group_m, group_n, mt, ntw);
    for (int h = 0; h < 2; ++h) {
      const int nt = 2 * ntw + h;
      if (nt >= num_n) {
        if (h == 0 || nt > num_n) {  // only the odd last block may lie past the grid
          std::printf("wide: tile %d -> column tile %d of %d\n", u, nt, num_n);
          return 1;
        }
        continue;
      }
      if (mt < 0 || mt >= num_m || seen[static_cast<size_t>(mt) * num_n + nt]++) {
        std::printf("wide: M=%d N=%d gm=%d gn=%d tile %d repeats or leaves the grid\n", num_m,
                    num_n, group_m, group_n, u);
        return 1;
      }
    }
  }
  for (int v : seen)
    if (v != 1) {
      std::printf("wide: M=%d N=%d gm=%d gn=%d misses a tile\n", num_m, num_n, group_m, group_n);
      return 1;
    }
  return 0;
}

int main() {
  const int ms[] = {1, 2, 3, 15, 16, 17, 29, 32, 33, 64, 257};
  const int ns[] = {1, 2, 5, 16, 17, 40, 594};
  const int gms[] = {0, 1, 3, 8, 16, 32};
  const int gns[] = {1, 4, 16, 64};
  for (int m : ms)
    for (int n : ns)
      for (int gm : gms)
        for (int gn : gns)
          if (check_raster(m, n, gm, gn)) return 1;

  const int nks[] = {0, 1, 255, 256, 257, 8191, 8192, 8193, 36258, 65536, 100000};
  const int cs[] = {256, 2048, 8192};
  for (int nk : nks)
    for (int c : cs) {
      const int slots = (nk + c - 1) / c + 1;
      int next = 0;
      for (int i = 0; i < slots + 2; ++i) {
        int start = -1, rows = -1;
        chunk_span(nk, c, i, start, rows);
        if (rows < 0 || rows > c || (rows > 0 && start != next)) {
          std::printf("chunk_span: Nk=%d C=%d chunk %d -> start %d rows %d (expected start %d)\n",
                      nk, c, i, start, rows, next);
          return 1;
        }
        next += rows;
      }
      if (next != nk) {
        std::printf("chunk_span: Nk=%d C=%d covers %d rows\n", nk, c, next);
        return 1;
      }
    }

  for (int tiles : {1, 2, 3, 5, 8, 31, 75, 76, 77, 151, 152, 153, 232, 256, 320, 699, 1280})
    for (int workers : {1, 2, 38, 76, 152})
      for (int kb : {0, 1, 2, 3, 4, 7, 47, 64, 2374, 4096})
        for (int S : {1, 2, 3, 4})
          for (int fill : {85, 100})
            for (bool may : {false, true})
              if (check_schedule(tiles, workers, kb, may, S, fill)) return 1;
  // the half-kept 30B-MoE head's dHidden (8192-row chunks, H = 4096 on wide
  // tiles, V = 151936: 256 tiles on 76 CTA pairs) runs 3 whole waves and a
  // tail of 28 tiles in halves; the long-context head's (H = 5120: 320 tiles)
  // 4 whole waves and a tail of 16 tiles in quarters
  {
    const WorkSched a = work_schedule(32 * 8, 76, 2374, true, 4, 85);
    const WorkSched b = work_schedule(32 * 10, 76, 2374, true, 4, 85);
    if (a.full != 228 || a.split != 2 || b.full != 304 || b.split != 4) {
      std::printf("bench heads: full %d split %d / full %d split %d\n", a.full, a.split, b.full,
                  b.split);
      return 1;
    }
  }
  for (int m : {1, 2, 15, 29, 33})
    for (int n : {1, 2, 3, 10, 16, 17, 20})
      for (int gm : {0, 16})
        for (int gn : {1, 4, 16})
          if (check_wide_tiles(m, n, gm, gn)) return 1;
  // dh_reduce_kernel walks the dHidden tiles row-major: tile_coords with
  // group_m = 0 and all column tiles in one group
  for (int m : {1, 3, 32, 33})
    for (int n : {1, 2, 8, 20})
      for (int t = 0; t < m * n; ++t) {
        int mt = -1, nt = -1;
        tile_coords(t, m, n, 0, n, mt, nt);
        if (mt != t / n || nt != t % n) {
          std::printf("dHidden raster is not row-major: M=%d N=%d t=%d\n", m, n, t);
          return 1;
        }
      }

  // dh_reduce_kernel's tile count (tile_m = 256, tile_n = 512) equals the
  // wide kernel's for every H, so both compute the same schedule
  for (int H = 8; H <= 16384; H += 8) {
    const int num_n = (H + kBN - 1) / kBN;
    if ((num_n + 1) / 2 != (H + 2 * kBN - 1) / (2 * kBN)) {
      std::printf("wide tile count differs from the reduction's at H=%d\n", H);
      return 1;
    }
  }
  std::printf("ok\n");
  return 0;
}
