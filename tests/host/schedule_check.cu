// Host-side check of the persistent GEMMs' work schedule (no GPU needed):
//   * tile_coords maps the tile indices 0 .. num_m*num_n-1 one-to-one onto
//     the (row tile, column tile) grid for every raster setting in use;
//   * chunk_span splits Nk kept rows into chunks that cover [0, Nk) in order,
//     each at most chunk_rows long;
//   * dh_split_count never splits past the K blocks or the partial buffers;
//   * the 512-column tiles of the CTA-pair kernel, walked as the kernel walks
//     them (raster over wide tiles, then their two 256-column blocks), cover
//     every (row tile, 256-column tile, K part) once -- a block past the last
//     256-column tile only when that count is odd -- and the K parts
//     partition the K blocks; dh_reduce_kernel, which counts the tiles as
//     row tiles x ceil(H / 512), sees the kernel's unit count.
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

// Units of the CTA-pair kernel with 512-column tiles, walked as it walks them.
static int check_wide_units(int num_m, int num_n, int group_m, int group_n, int splits,
                            int num_kb) {
  const int num_nw = (num_n + 1) / 2;   // 512-column tiles over num_n 256-column tiles
  const int num_tiles = num_m * num_nw;
  std::vector<int> seen(static_cast<size_t>(num_m) * num_n * splits, 0);
  std::vector<int> kcover(static_cast<size_t>(num_kb), 0);
  for (int u = 0; u < num_tiles * splits; ++u) {
    const int sidx = u / num_tiles;
    const int kb0 = static_cast<int>(static_cast<long long>(sidx) * num_kb / splits);
    const int kb1 = static_cast<int>(static_cast<long long>(sidx + 1) * num_kb / splits);
    if (kb1 <= kb0) {
      std::printf("wide: empty K part %d of %d over %d blocks\n", sidx, splits, num_kb);
      return 1;
    }
    int mt = -1, ntw = -1;
    tile_coords(u % num_tiles, num_m, num_nw, group_m, group_n, mt, ntw);
    if (u % num_tiles == 0)
      for (int kb = kb0; kb < kb1; ++kb) ++kcover[static_cast<size_t>(kb)];
    for (int h = 0; h < 2; ++h) {
      const int nt = 2 * ntw + h;
      if (nt >= num_n) {
        if (h == 0 || nt > num_n) {  // only the odd last block may lie past the grid
          std::printf("wide: unit %d -> column tile %d of %d\n", u, nt, num_n);
          return 1;
        }
        continue;
      }
      if (mt < 0 || mt >= num_m || seen[(static_cast<size_t>(sidx) * num_m + mt) * num_n + nt]++) {
        std::printf("wide: M=%d N=%d gm=%d gn=%d S=%d unit %d repeats or leaves the grid\n",
                    num_m, num_n, group_m, group_n, splits, u);
        return 1;
      }
    }
  }
  for (int v : seen)
    if (v != 1) {
      std::printf("wide: M=%d N=%d gm=%d gn=%d S=%d misses a tile\n", num_m, num_n, group_m,
                  group_n, splits);
      return 1;
    }
  for (int v : kcover)
    if (v != 1) {
      std::printf("wide: K parts of %d blocks in %d parts do not partition\n", num_kb, splits);
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

  for (int tiles = 1; tiles < 700; tiles += 7)
    for (int workers : {1, 38, 76, 152})
      for (int kb : {1, 2, 3, 64, 2374}) {
        const int s = dh_split_count(tiles, workers, kb, 4, 85);
        if (s < 1 || s > 4 || s > kb) {
          std::printf("dh_split_count(%d, %d, %d) = %d\n", tiles, workers, kb, s);
          return 1;
        }
      }
  for (int m : {1, 2, 15, 29, 33})
    for (int n : {1, 2, 3, 10, 16, 17, 20})
      for (int gm : {0, 16})
        for (int gn : {1, 4, 16})
          for (int s : {1, 2, 3, 4})
            for (int kb : {4, 7, 2374})
              if (check_wide_units(m, n, gm, gn, s, kb)) return 1;

  // dh_reduce_kernel's tile count (tile_m = 256, tile_n = 512) equals the
  // wide kernel's for every H, so both take the same K split
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
