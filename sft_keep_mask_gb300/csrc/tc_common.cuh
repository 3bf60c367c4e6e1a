// Pieces shared by the one-CTA and the CTA-pair tcgen05 GEMMs: the tile
// raster, the drain wait and the fused epilogues of the four contractions.
//
// The epilogues read one accumulator row per thread (TMEM lane = row) in
// slices of 32 fp32 columns:
//   kFwd  per-row online softmax over the 256-column vocab tile: running max
//         m (log2 units), s = sum 2^(z2 - m), u = sum 2^(z2 - m) (z2 - m), and
//         the target logit; written as (m ln2, s, u ln2, t) partials.  This is
//         the single fused projection for log-prob and entropy of SkyRL pull
//         request #2374 ("How it works"), with the entropy -(p log p) of its
//         gemini-code-assist review kept in max-shifted form.
//   kDz   dz = g_lp (1[v=y] - p) - g_ent p (log p + H) from the recomputed
//         logit, p = exp(z - lse) (the backward of the same page; logits
//         recomputed rather than saved, twinkle pull request #283, section 1),
//         rounded to bf16 and written by TMA stores from shared memory.
//   kDh   bf16 rows scattered to dhidden[idx[row]] (fp32 partial rows when
//         the tile's K range is split into parts, see work_schedule).
//   kDw   fp32 dW tile, written by TMA stores (first chunk) or added to dW by
//         TMA reduce-adds at L2.
#pragma once

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace lmhead {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Tile t -> (row tile, column tile).
//
// group_m > 0 (the vocabulary projections): the row tiles form blocks of
// group_m; inside a block the tiles walk the block's row tiles for every
// column tile.  The block's A rows (group_m x 256 rows of Hc) stay in L2 while
// the column operand (W) streams past once per block.
//
// group_m == 0: tiles walk `group_n` column tiles for every row tile before
// the next group, so the CTAs in flight share the group's column operand
// through L2 (dHidden, dW: group_n = all of H).
__host__ __device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int group_m,
                                                     int group_n, int& mt, int& nt) {
  if (group_m > 0) {
    const int per_block = group_m * num_n;
    const int b = t / per_block;
    const int local = t - b * per_block;
    const int left = num_m - b * group_m;
    const int rows = left < group_m ? left : group_m;
    nt = local / rows;
    mt = b * group_m + (local - nt * rows);
    return;
  }
  const int per_group = num_m * group_n;
  const int g = t / per_group;
  const int local = t - g * per_group;
  const int rem = num_n - g * group_n;
  const int gn = rem < group_n ? rem : group_n;
  mt = local / gn;
  nt = g * group_n + (local - (local / gn) * gn);
}

// Wait without the abort check: used only to drain copies / MMAs in flight
// before the CTA releases its shared and tensor memory.  Running out of time
// here is recorded like any other timeout.
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity, int* status,
                                                int site) {
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) {
      record_timeout(status, site);
      return;
    }
  }
}

// Staged TMA output of one epilogue warp (kDz, kDw).  The warp's 32 rows of
// a 128-byte-wide box go to one of its two 4 KB buffers in the 128-byte
// swizzled layout the tensor map expects (16-byte chunk c of row r at chunk
// position c ^ (r & 7); the buffers are 1024-byte aligned), then lane 0 has
// the TMA write the box.  A buffer is refilled only after the store issued
// from it two boxes earlier has read it.
struct OutStage {
  const CUtensorMap* map;  // output tensor map (box: 32 rows x 128 bytes)
  uint8_t* buf;            // this warp's two buffers (8 KB, 1024-byte aligned)
  uint32_t issued;         // boxes issued by this warp so far
};

// Buffer for the next box; waits until the store issued from it has read it.
__device__ __forceinline__ uint8_t* out_buffer(OutStage& os, int lane) {
  if (lane == 0) bulk_wait_read_all_but_one();
  __syncwarp();
  return os.buf + (os.issued & 1u) * kOutBoxBytes;
}

// 16-byte chunk c (0..7) of this lane's 128-byte row in the buffer.
__device__ __forceinline__ void out_put(uint8_t* b, int lane, int c, uint4 v) {
  *reinterpret_cast<uint4*>(b + lane * 128 + ((c ^ (lane & 7)) << 4)) = v;
}

// Makes the buffer visible to the TMA and writes (or, with `add`, adds) the
// box whose top-left element is (x, y) of the output map.
__device__ __forceinline__ void out_issue(OutStage& os, uint8_t* b, int lane, int x, int y,
                                          bool add) {
  fence_proxy_async_shared();
  __syncwarp();
  if (lane == 0) {
    if (add)
      tma_reduce_add_2d(os.map, b, x, y);
    else
      tma_store_2d(os.map, b, x, y);
    bulk_commit();
  }
  ++os.issued;
}

// Epilogue of one 256-column accumulator tile for this thread's row.
//   tbase      TMEM address of (this warp's lane quarter, column 0 of the tile)
//   row        kFwd/kDz/kDh: row within the chunk; kDw: vocabulary row
//   nt         column tile
//   cstart     first compact row of the chunk
//   rows_valid rows of the chunk that hold kept tokens
//   have_acc   false only for kDw with an empty K range (writes zeros)
//   slot, slots  kDh: part `slot` of the `slots` K parts of the tile
//              (work_schedule); with slots > 1 write fp32 partial sums to
//              partial buffer `slot`
//   release    called once, right after the last TMEM load of the tile
//   os         the warp's output staging (kDz, kDw)
template <int MODE, typename Release>
__device__ __forceinline__ void epilogue_tile(const TcGemmParams& p, uint32_t tbase, int row,
                                              int nt, int cstart, int rows_valid, bool have_acc,
                                              int slot, int slots, OutStage& os,
                                              Release&& release) {
  constexpr int kSlices = kBN / 32;
  const int col_tile = nt * kBN;

  if (MODE == kFwd) {
    const bool row_ok = row < rows_valid;
    const int y = row_ok ? p.targets_c[cstart + row] : -1;
    const bool tail = col_tile + kBN > p.V;
    float m2 = -INFINITY, s = 0.f, u2 = 0.f, tz = -INFINITY;
#pragma unroll 1
    for (int c = 0; c < kSlices; ++c) {
      uint32_t r[32];
      __syncwarp();
      tmem_ld32(tbase + c * 32, r);
      tmem_ld_wait();
      if (c == kSlices - 1) release();
      const int col = col_tile + c * 32;
      float z[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) z[j] = __uint_as_float(r[j]);
      if (tail) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (col + j >= p.V) z[j] = -INFINITY;
      }
      if (static_cast<unsigned>(y - col) < 32u) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j == y - col) tz = z[j];
      }
      float cmax = z[0];
#pragma unroll
      for (int j = 1; j < 32; ++j) cmax = fmaxf(cmax, z[j]);
      if (cmax == -INFINITY) continue;  // slice wholly past the vocabulary
      const float cm2 = cmax * kLog2e;
      if (cm2 > m2) {
        if (m2 != -INFINITY) {
          const float sc = fast_exp2(m2 - cm2);
          u2 = sc * (u2 + s * (m2 - cm2));
          s *= sc;
        }
        m2 = cm2;
      }
      if (!tail) {
        if (p.want_entropy) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float d = fmaf(z[j], kLog2e, -m2);
            const float e = fast_exp2(d);
            s += e;
            u2 = fmaf(e, d, u2);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) s += fast_exp2(fmaf(z[j], kLog2e, -m2));
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (col + j < p.V) {
            const float d = fmaf(z[j], kLog2e, -m2);
            const float e = fast_exp2(d);
            s += e;
            u2 = fmaf(e, d, u2);
          }
        }
      }
    }
    // (a column tile past V -- the second pair's tile of a cluster when the
    // number of vocabulary tiles is odd -- has no partials to write)
    if (row_ok && col_tile < p.V && LM_DCHECK(row < p.chunk_rows, p.status))
      p.part[static_cast<int64_t>(nt) * p.chunk_rows + row] =
          make_float4(m2 * kLn2, s, u2 * kLn2, tz);
  } else if (MODE == kDz) {
    // (block-sparse: rows of an active tile that are not kept get dz = 0)
    const bool row_ok = row < rows_valid && (p.lvalid == nullptr || p.lvalid[cstart + row] != 0);
    float lse2 = 0.f, ca = 0.f, cb = 0.f, glp = 0.f;
    int y = -1;
    if (row_ok) {
      const int cr = cstart + row;
      lse2 = p.lse_c[cr] * kLog2e;
      glp = p.glp_c[cr];
      y = p.targets_c[cr];
      if (p.gent_c != nullptr) {
        const float ge = p.gent_c[cr];
        ca = ge * kLn2;
        cb = glp + ge * p.ent_c[cr];
      } else {
        cb = glp;
      }
    }
    // The warp's rows [row0, row0 + 32) of dZ leave in boxes of 64 columns:
    // two 32-column slices fill one box (chunks 0-3, then 4-7).
    const int lane = threadIdx.x & 31;
    const int row0 = row - lane;
    uint8_t* b = nullptr;
#pragma unroll 1
    for (int c = 0; c < kSlices; ++c) {
      uint32_t r[32];
      __syncwarp();
      tmem_ld32(tbase + c * 32, r);
      tmem_ld_wait();
      if (c == kSlices - 1) release();
      const int col = col_tile + c * 32;
      const int box_col = col_tile + (c & ~1) * 32;
      if (box_col >= p.V) continue;  // warp-uniform: the box lies past the vocabulary
      uint32_t packed[16];
      if (row_ok) {
        float g[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float d = fmaf(__uint_as_float(r[j]), kLog2e, -lse2);
          const float pe = fast_exp2(d);
          g[j] = -pe * fmaf(ca, d, cb);
        }
        if (static_cast<unsigned>(y - col) < 32u) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j == y - col) g[j] += glp;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) packed[j] = pack_bf16x2(g[2 * j], g[2 * j + 1]);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) packed[j] = 0u;
      }
      if ((c & 1) == 0) b = out_buffer(os, lane);
#pragma unroll
      for (int v = 0; v < 4; ++v)
        out_put(b, lane, (c & 1) * 4 + v,
                make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2],
                           packed[4 * v + 3]));
      if (c & 1) out_issue(os, b, lane, box_col, row0, false);
    }
  } else if (MODE == kDh) {
    const bool kept = row < rows_valid && (p.lvalid == nullptr || p.lvalid[cstart + row] != 0);
    const int64_t orow = kept ? p.idx[cstart + row] : 0;
    const bool row_ok = kept && LM_DCHECK(orow >= 0 && orow < p.n_rows, p.status);
    __nv_bfloat16* hrow = p.dhidden + orow * p.H;
    float* prow = p.dh_part +
                  (static_cast<int64_t>(slot) * p.chunk_rows + (row_ok ? row : 0)) * p.H;
#pragma unroll 1
    for (int c = 0; c < kSlices; ++c) {
      uint32_t r[32];
      __syncwarp();
      tmem_ld32(tbase + c * 32, r);
      tmem_ld_wait();
      if (c == kSlices - 1) release();
      const int col = col_tile + c * 32;
      if (!row_ok || col >= p.H) continue;
      if (slots > 1) {
        float4* dst = reinterpret_cast<float4*>(prow + col);
#pragma unroll
        for (int v = 0; v < 8; ++v)
          if (col + 4 * v < p.H)
            dst[v] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                 __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
        continue;
      }
      uint4* dst = reinterpret_cast<uint4*>(hrow + col);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        if (col + 8 * v < p.H) {
          dst[v] = make_uint4(
              pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1])),
              pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3])),
              pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5])),
              pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7])));
        }
      }
    }
  } else {  // kDw
    // The warp's rows [row0, row0 + 32) of dW (vocabulary rows; rows past V
    // are clipped by the map) leave in boxes of 32 fp32 columns, added to dW
    // at L2 when accumulating, stored otherwise.
    const int lane = threadIdx.x & 31;
    const int row0 = row - lane;
#pragma unroll 1
    for (int c = 0; c < kSlices; ++c) {
      uint32_t r[32];
      if (have_acc) {
        __syncwarp();
        tmem_ld32(tbase + c * 32, r);
        tmem_ld_wait();
        if (c == kSlices - 1) release();
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = 0u;
      }
      const int col = col_tile + c * 32;
      // warp-uniform: no box starts past the matrix (rows past V inside a
      // box are clipped by the map)
      if (col >= p.H || row0 >= p.V) continue;
      uint8_t* b = out_buffer(os, lane);
#pragma unroll
      for (int v = 0; v < 8; ++v)
        out_put(b, lane, v, make_uint4(r[4 * v], r[4 * v + 1], r[4 * v + 2], r[4 * v + 3]));
      out_issue(os, b, lane, col, row0, p.beta != 0);
    }
  }
}

// Problem extents of a contraction for this chunk (the number of kept rows
// lives on the device).  Returns false when the launch has nothing to do.
template <int MODE>
__device__ __forceinline__ bool gemm_extents(const TcGemmParams& p, int& cstart, int& rows_valid,
                                             int& M, int& N, int& K) {
  chunk_span(*p.d_nk, p.chunk_rows, p.chunk_index, cstart, rows_valid);
  if (MODE == kDw) {
    M = p.V; N = p.H; K = rows_valid;
    // An empty first chunk still has to clear dW when it is not accumulated.
    return !(rows_valid == 0 && (p.beta || p.chunk_index > 0));
  }
  if (MODE == kDh) {
    M = rows_valid; N = p.H; K = p.V;
  } else {
    M = rows_valid; N = p.V; K = p.H;
  }
  return rows_valid > 0;
}

}  // namespace lmhead
