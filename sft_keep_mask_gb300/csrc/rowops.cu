// Row kernels of the fused LM-head path: keep-mask construction, stable
// compaction of the kept rows, gathers into compact buffers, the split-V
// partial merge and the expansion back to every row.  All of them are
// memory-bound and sized by the device-resident number of kept rows, so no
// host synchronisation is needed between the steps.
//
// Source for the steps: prime-rl pull request #3326, "Don't compute the
// logprobs and their gradients for tokens no loss component reads",
// "Overview" (keep mask after the next-token shift; compact -> chunked
// logprob/entropy -> expand back with zeros).
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace lmhead {

namespace {

constexpr int kScanThreads = 256;
constexpr int kScanPerThread = 16;
constexpr int kScanTile = kScanThreads * kScanPerThread;  // rows per block
static_assert(kScanTile == kCompactRowsPerBlock, "scan block size");

// ---------------------------------------------------------------- keep mask
__global__ void build_keep_kernel(const float* __restrict__ c0, const float* __restrict__ c1,
                                  const float* __restrict__ c2,
                                  const int32_t* __restrict__ offsets, int n_seq, int64_t N,
                                  uint8_t* __restrict__ keep) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= N) return;
  const int64_t nxt = i + 1;
  uint8_t k = 0;
  if (nxt < N) {
    // Is token i+1 the first token of a packed sequence?  (binary search)
    int lo = 0, hi = n_seq;  // offsets[0..n_seq]
    bool starts = false;
    while (lo <= hi) {
      const int mid = (lo + hi) >> 1;
      const int64_t v = offsets[mid];
      if (v == nxt) { starts = true; break; }
      if (v < nxt) lo = mid + 1; else hi = mid - 1;
    }
    if (!starts) {
      const bool read = (c0 != nullptr && c0[nxt] != 0.f) || (c1 != nullptr && c1[nxt] != 0.f) ||
                        (c2 != nullptr && c2[nxt] != 0.f);
      k = read ? 1 : 0;
    }
  }
  keep[i] = k;
}

// --------------------------------------------------------------- compaction
__device__ __forceinline__ int block_sum(int v, int* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) red[w] = v;
  __syncthreads();
  int tot = 0;
  for (int j = 0; j < (int)(blockDim.x >> 5); ++j) tot += red[j];
  return tot;
}

// Per block of kScanTile rows: the number of kept rows.
__global__ void count_kernel(const uint8_t* __restrict__ keep, int64_t N, int32_t* counts) {
  __shared__ int red[kScanThreads / 32];
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kScanTile;
  int c = 0;
  for (int j = 0; j < kScanPerThread; ++j) {
    const int64_t r = base + threadIdx.x + static_cast<int64_t>(j) * kScanThreads;
    if (r < N) c += (keep == nullptr || keep[r] != 0) ? 1 : 0;
  }
  const int tot = block_sum(c, red);
  if (threadIdx.x == 0) counts[blockIdx.x] = tot;
}

// Writes the kept rows of block b, in order, after the kept rows of blocks
// 0..b-1; the last block also writes Nk.
// Targets are checked against [0, V_valid) and stored relative to t_offset
// (the first vocabulary row of a shard; 0 for the whole vocabulary).
__global__ void scatter_kernel(const uint8_t* __restrict__ keep,
                               const int64_t* __restrict__ targets, int64_t N, int64_t V_valid,
                               int64_t t_offset, const int32_t* __restrict__ counts,
                               int32_t* __restrict__ idx, int32_t* __restrict__ targets_c,
                               int32_t* d_nk, int* status) {
  __shared__ int red[kScanThreads / 32];
  __shared__ int warp_tot[kScanThreads / 32];
  // offset of this block = sum of the counts of the blocks before it
  int pre = 0;
  for (int j = threadIdx.x; j < static_cast<int>(blockIdx.x); j += kScanThreads) pre += counts[j];
  const int offset = block_sum(pre, red);

  const int64_t base = static_cast<int64_t>(blockIdx.x) * kScanTile +
                       static_cast<int64_t>(threadIdx.x) * kScanPerThread;
  uint32_t bits = 0;
  for (int j = 0; j < kScanPerThread; ++j) {
    const int64_t r = base + j;
    if (r < N && (keep == nullptr || keep[r] != 0)) bits |= 1u << j;
  }
  const int mine = __popc(bits);
  // exclusive scan of `mine` over the block
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  int incl = mine;
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (l >= o) incl += v;
  }
  if (l == 31) warp_tot[w] = incl;
  __syncthreads();
  int wpre = 0;
  for (int j = 0; j < w; ++j) wpre += warp_tot[j];
  int pos = offset + wpre + incl - mine;
  for (int j = 0; j < kScanPerThread; ++j) {
    if (bits & (1u << j)) {
      const int64_t r = base + j;
      idx[pos] = static_cast<int32_t>(r);
      if (targets != nullptr) {  // (null when compacting tiles rather than rows)
        int64_t y = targets[r];
        if (y < 0 || y >= V_valid) {
          atomicCAS(status, 0, kStatusTarget);
          y = 0;
        }
        targets_c[pos] = static_cast<int32_t>(y - t_offset);
      }
      ++pos;
    }
  }
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x == kScanThreads - 1) {
    int tot = 0;
    for (int j = 0; j < kScanThreads / 32; ++j) tot += warp_tot[j];
    *d_nk = offset + tot;
  }
}

// ------------------------------------------------------ block-sparse tiles
// tile_flags[t] = 1 iff some row of rows [256 t, 256 t + 256) is kept.
__global__ void tile_flags_kernel(const uint8_t* __restrict__ keep, int64_t N,
                                  uint8_t* __restrict__ flags) {
  const int64_t t = blockIdx.x;
  const int64_t r = t * 256 + threadIdx.x;
  const int k = (r < N && (keep == nullptr || keep[r] != 0)) ? 1 : 0;
  const int any = __syncthreads_or(k);
  if (threadIdx.x == 0) flags[t] = any ? 1 : 0;
}

// Per compact row l of the active tiles: the batch row behind it, its target
// and whether it is kept.  Rows past N (last tile) are not kept and point at
// row N-1 so that nothing reads out of bounds.
__global__ void tile_rows_kernel(const uint8_t* __restrict__ keep,
                                 const int64_t* __restrict__ targets, int64_t N, int64_t V_valid,
                                 int64_t t_offset, const int32_t* __restrict__ tile_list,
                                 const int32_t* d_na, int32_t* __restrict__ idx,
                                 int32_t* __restrict__ targets_c, uint8_t* __restrict__ lvalid,
                                 int32_t* d_nk, int* status) {
  const int na = *d_na;
  const int64_t l = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (l == 0) *d_nk = na * 256;
  if (l >= static_cast<int64_t>(na) * 256) return;
  const int64_t tile = tile_list[l >> 8];
  if (!LM_DCHECK(tile >= 0 && tile * 256 < N, status)) return;
  const int64_t r = tile * 256 + (l & 255);
  const bool kept = r < N && (keep == nullptr || keep[r] != 0);
  int64_t y = 0;
  if (kept) {
    y = targets[r];
    if (y < 0 || y >= V_valid) {
      atomicCAS(status, 0, kStatusTarget);
      y = 0;
    }
  }
  idx[l] = static_cast<int32_t>(r < N ? r : N - 1);
  targets_c[l] = static_cast<int32_t>(y - t_offset);
  lvalid[l] = kept ? 1 : 0;
}

// ------------------------------------------------------------------ gathers
// h_c[r] = hidden[idx[chunk_start + r]] for r < rows in chunk; rows up to the
// next multiple of 256 are zero-filled (they enter the weight-gradient
// contraction as zero K rows).  One warp per row, 16-byte vectors.
__global__ void gather_rows_kernel(const uint4* __restrict__ hidden,
                                   const int32_t* __restrict__ idx, const int32_t* d_nk,
                                   int chunk_index, int chunk_rows, int vec_per_row,
                                   uint4* __restrict__ hc, int64_t N, int* status) {
  int chunk_start, rows;
  chunk_span(*d_nk, chunk_rows, chunk_index, chunk_start, rows);
  const int padded = (rows + 255) & ~255;
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int l = threadIdx.x & 31;
  if (r >= padded || rows == 0) return;
  uint4* dst = hc + static_cast<int64_t>(r) * vec_per_row;
  if (r < rows) {
    const int32_t row = idx[chunk_start + r];
    if (!LM_DCHECK(row >= 0 && row < N, status)) return;
    const uint4* src = hidden + static_cast<int64_t>(row) * vec_per_row;
    for (int v = l; v < vec_per_row; v += 32) dst[v] = src[v];
  } else {
    for (int v = l; v < vec_per_row; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
  }
}

__global__ void gather_vec_kernel(const int32_t* __restrict__ idx, const int32_t* d_nk,
                                  const float* a, const float* b, const float* c, const float* d,
                                  float* a_c, float* b_c, float* c_c, float* d_c, int64_t N,
                                  int* status) {
  const int k = blockIdx.x * blockDim.x + threadIdx.x;
  if (k >= *d_nk) return;
  const int r = idx[k];
  if (!LM_DCHECK(r >= 0 && r < N, status)) return;
  if (a) a_c[k] = a[r];
  if (b) b_c[k] = b[r];
  if (c) c_c[k] = c[r];
  if (d) d_c[k] = d[r];
}

// -------------------------------------------------------------------- merge
// Split-V merge of the per-tile (m, s, u, t) partials of one chunk:
//   M = max m_i, S = sum s_i e^(m_i - M), U = sum e^(m_i - M)(u_i + s_i (m_i - M))
//   lse = M + log S, logprob = t - lse, entropy = log S - U / S.
// A block takes kMergeRows consecutive rows; its 256 threads form 32 groups
// of one thread per row, group j taking the vocab tiles j, j + 32, ... with
// a running max-shifted (M, S, U), so each load instruction of a warp reads 4
// vocab tiles x 8 consecutive rows: four whole 128-byte lines.  The 32
// partial reductions of a row are combined in a fixed order: the 4 groups of
// a warp by shuffles, then the 8 warps through shared memory.
constexpr int kMergeRows = 8;
constexpr int kMergeGroups = 256 / kMergeRows;

__device__ __forceinline__ void merge_pair(float& M, float& S, float& U, float m2, float s2,
                                           float u2) {
  if (m2 == -INFINITY) return;
  if (M == -INFINITY) {
    M = m2; S = s2; U = u2;
    return;
  }
  const float N = fmaxf(M, m2);
  const float a = expf(M - N), b = expf(m2 - N);
  U = a * (U + S * (M - N)) + b * (u2 + s2 * (m2 - N));
  S = a * S + b * s2;
  M = N;
}

__global__ void __launch_bounds__(256) merge_kernel(const float4* __restrict__ part, int num_vt,
                                                    const int32_t* d_nk, int chunk_index,
                                                    int chunk_rows, int want_entropy,
                                                    float* __restrict__ lp_c,
                                                    float* __restrict__ ent_c,
                                                    float* __restrict__ lse_c,
                                                    float4* __restrict__ raw_c) {
  int chunk_start, rows;
  chunk_span(*d_nk, chunk_rows, chunk_index, chunk_start, rows);
  const int r0 = static_cast<int>(blockIdx.x) * kMergeRows;
  if (r0 >= rows) return;  // whole block
  const int ri = threadIdx.x & (kMergeRows - 1);
  const int grp = threadIdx.x / kMergeRows;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int r = r0 + ri;
  float M = -INFINITY, S = 0.f, U = 0.f, T = -INFINITY;
  if (r < rows) {
    int v = grp;
    for (; v + 3 * kMergeGroups < num_vt; v += 4 * kMergeGroups) {
      float4 q[4];
#pragma unroll
      for (int k = 0; k < 4; ++k)
        q[k] = part[static_cast<int64_t>(v + k * kMergeGroups) * chunk_rows + r];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        merge_pair(M, S, U, q[k].x, q[k].y, q[k].z);
        T = fmaxf(T, q[k].w);
      }
    }
    for (; v < num_vt; v += kMergeGroups) {
      const float4 q = part[static_cast<int64_t>(v) * chunk_rows + r];
      merge_pair(M, S, U, q.x, q.y, q.z);
      T = fmaxf(T, q.w);
    }
  }
  // the 4 groups of this warp: lanes ri, ri + 8, ri + 16, ri + 24
#pragma unroll
  for (int off = kMergeRows; off < 32; off <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, M, off);
    const float s2 = __shfl_xor_sync(0xffffffffu, S, off);
    const float u2 = __shfl_xor_sync(0xffffffffu, U, off);
    const float t2 = __shfl_xor_sync(0xffffffffu, T, off);
    // the lower lane's value first, so both lanes of a pair hold the same sum
    if ((lane & off) == 0) {
      merge_pair(M, S, U, m2, s2, u2);
    } else {
      float m1 = m2, s1 = s2, u1 = u2;
      merge_pair(m1, s1, u1, M, S, U);
      M = m1; S = s1; U = u1;
    }
    T = fmaxf(T, t2);
  }
  __shared__ float4 warp_part[256 / 32][kMergeRows];
  if (lane < kMergeRows) warp_part[warp][lane] = make_float4(M, S, U, T);
  __syncthreads();
  if (threadIdx.x >= kMergeRows || r >= rows) return;
  // thread ri (warp 0, lane ri) adds the warps' reductions of its row in order
  M = -INFINITY; S = 0.f; U = 0.f; T = -INFINITY;
#pragma unroll
  for (int w = 0; w < 256 / 32; ++w) {
    const float4 q = warp_part[w][ri];
    merge_pair(M, S, U, q.x, q.y, q.z);
    T = fmaxf(T, q.w);
  }
  if (raw_c != nullptr) {  // a vocabulary shard: keep the unnormalised reduction
    raw_c[chunk_start + r] = make_float4(M, S, U, T);
    return;
  }
  const float logS = logf(S);
  const float lse = M + logS;
  lp_c[chunk_start + r] = T - lse;
  lse_c[chunk_start + r] = lse;
  if (want_entropy) ent_c[chunk_start + r] = logS - U / S;
}

// Merge of the vocabulary shards' (m, s, u, t) partials, [S][N] float4, into
// logprob, entropy and lse of every row (skipped rows get +0.0).
__global__ void merge_shards_kernel(const float4* __restrict__ partials, int num_shards,
                                    const uint8_t* __restrict__ keep, int64_t N,
                                    int want_entropy, float* __restrict__ lp,
                                    float* __restrict__ ent, float* __restrict__ lse) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= N) return;
  if (keep != nullptr && keep[i] == 0) {
    lp[i] = 0.f;
    lse[i] = 0.f;
    if (ent) ent[i] = 0.f;
    return;
  }
  float M = -INFINITY;
  for (int r = 0; r < num_shards; ++r) M = fmaxf(M, partials[r * N + i].x);
  float S = 0.f, U = 0.f, T = -INFINITY;
  for (int r = 0; r < num_shards; ++r) {
    const float4 q = partials[r * N + i];
    const float sc = expf(q.x - M);
    S = fmaf(q.y, sc, S);
    U = fmaf(sc, fmaf(q.y, q.x - M, q.z), U);
    T = fmaxf(T, q.w);
  }
  const float logS = logf(S);
  lse[i] = M + logS;
  lp[i] = T - (M + logS);
  if (want_entropy) ent[i] = logS - U / S;
}

// Expand compact float4 rows to all rows; skipped rows get (-inf, 0, 0, -inf).
__global__ void expand4_kernel(const uint8_t* __restrict__ keep, const int32_t* __restrict__ idx,
                               const int32_t* d_nk, int64_t N, const float4* __restrict__ src,
                               float4* __restrict__ dst, int* status) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= N) return;
  if (keep != nullptr && keep[i] == 0) dst[i] = make_float4(-INFINITY, 0.f, 0.f, -INFINITY);
  if (i < *d_nk) {
    const int32_t r = idx[i];
    if (LM_DCHECK(r >= 0 && r < N, status)) dst[r] = src[i];
  }
}

// ------------------------------------------------------------------- expand
// Disjoint writes: skipped rows get +0.0, kept row idx[k] gets value k (in
// block-sparse mode only the compact rows with lvalid set are kept rows).
__global__ void expand3_kernel(const uint8_t* __restrict__ keep, const int32_t* __restrict__ idx,
                               const int32_t* d_nk, int64_t N, const float* a_c,
                               const float* b_c, const float* c_c, float* a, float* b,
                               float* c, const uint8_t* __restrict__ lvalid, int* status) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < N && keep != nullptr && keep[i] == 0) {
    if (a) a[i] = 0.f;
    if (b) b[i] = 0.f;
    if (c) c[i] = 0.f;
  }
  if (i < *d_nk && (lvalid == nullptr || lvalid[i] != 0)) {
    const int r = idx[i];
    if (!LM_DCHECK(r >= 0 && r < N, status)) return;
    if (a) a[r] = a_c[i];
    if (b) b[r] = b_c[i];
    if (c) c[r] = c_c[i];
  }
}

// The public expansion: idx and Nk come from the caller, so an index outside
// [0, N) (or Nk > N) is skipped and reported instead of written.
__global__ void scatter_vals_kernel(const float* __restrict__ src, const int32_t* __restrict__ idx,
                                    const int32_t* d_nk, int64_t N, float* __restrict__ dst,
                                    int* status) {
  const int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nk = *d_nk;
  if (k == 0 && nk > N && status != nullptr) atomicCAS(status, 0, kStatusBounds);
  if (k >= nk || k >= N) return;
  const int32_t r = idx[k];
  if (r < 0 || r >= N) {
    if (status != nullptr) atomicCAS(status, 0, kStatusBounds);
    return;
  }
  dst[r] = src[k];
}

// One block per (tile, 32-row slice) of the chunk's dHidden tile grid.  Only
// the tiles of the split tail (work_schedule) hold partial sums; the blocks
// of the tiles taken whole return at once.  The partials are added in slot
// (K) order, so the sum is the same on every run.
__global__ void dh_reduce_kernel(const float4* __restrict__ part, const int32_t* d_nk,
                                 int chunk_index, int chunk_rows, int H, int tile_m, int tile_n,
                                 int workers, int num_kb, int max_split, int fill_pct,
                                 const int32_t* __restrict__ idx,
                                 const uint8_t* __restrict__ lvalid, uint2* __restrict__ dhidden,
                                 int64_t N, int* status) {
  int chunk_start, rows;
  chunk_span(*d_nk, chunk_rows, chunk_index, chunk_start, rows);
  if (rows == 0) return;
  const int num_m = (rows + tile_m - 1) / tile_m;
  const int num_n = (H + tile_n - 1) / tile_n;
  const int t = static_cast<int>(blockIdx.x);
  if (t >= num_m * num_n) return;
  const WorkSched sched = work_schedule(num_m * num_n, workers, num_kb, true, max_split, fill_pct);
  const int slots = sched.tile_slots(t);
  if (slots < 2) return;
  // dHidden walks its tiles row-major (tile_coords with group_m = 0 and all
  // column tiles in one group)
  const int mt = t / num_n;
  const int nt = t - mt * num_n;
  const int q = H / 4;  // float4 columns per row
  const int c0 = nt * (tile_n / 4);
  const int cn = q - c0 < tile_n / 4 ? q - c0 : tile_n / 4;
  const int r0 = mt * tile_m + static_cast<int>(blockIdx.y) * 32;
  const int64_t plane = static_cast<int64_t>(chunk_rows) * q;
  for (int e = threadIdx.x; e < 32 * cn; e += blockDim.x) {
    const int r = r0 + e / cn;
    const int c = c0 + e % cn;
    if (r >= rows) continue;
    if (lvalid != nullptr && lvalid[chunk_start + r] == 0) continue;  // not a kept row
    const int64_t at = static_cast<int64_t>(r) * q + c;
    // all partial loads in flight before the (fixed-order) sum
    float4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      v[k] = k < slots ? __ldcs(part + k * plane + at) : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 acc = v[0];
#pragma unroll
    for (int k = 1; k < 4; ++k) {
      if (k < slots) {
        acc.x += v[k].x; acc.y += v[k].y; acc.z += v[k].z; acc.w += v[k].w;
      }
    }
    const int64_t orow = idx[chunk_start + r];
    if (!LM_DCHECK(orow >= 0 && orow < N, status)) continue;
    dhidden[orow * q + c] = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
  }
}

// Rows of skipped tokens of dhidden are written as zeros (warp per row).
__global__ void zero_skipped_rows_kernel(const uint8_t* __restrict__ keep, int64_t N,
                                         int vec_per_row, uint4* __restrict__ dh) {
  const int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= N || keep[r] != 0) return;
  uint4* dst = dh + r * vec_per_row;
  for (int v = threadIdx.x & 31; v < vec_per_row; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
}

inline unsigned blocks_for(int64_t n, int per) {
  return static_cast<unsigned>((n + per - 1) / per);
}

}  // namespace

cudaError_t launch_build_keep(const float* c0, const float* c1, const float* c2,
                              const int32_t* offsets, int n_seq, int64_t N, uint8_t* keep,
                              cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  build_keep_kernel<<<blocks_for(N, 256), 256, 0, s>>>(c0, c1, c2, offsets, n_seq, N, keep);
  return cudaGetLastError();
}

cudaError_t launch_compact(const uint8_t* keep, const int64_t* targets, int64_t N,
                           int64_t V_valid, int64_t t_offset, int32_t* idx, int32_t* targets_c,
                           int32_t* d_nk, int32_t* counts, int* status, cudaStream_t s) {
  const unsigned nb = blocks_for(N, kScanTile);
  count_kernel<<<nb, kScanThreads, 0, s>>>(keep, N, counts);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  scatter_kernel<<<nb, kScanThreads, 0, s>>>(keep, targets, N, V_valid, t_offset, counts, idx,
                                             targets_c, d_nk, status);
  return cudaGetLastError();
}

cudaError_t launch_tile_scan(const uint8_t* keep, const int64_t* targets, int64_t N,
                             int64_t V_valid, int64_t t_offset, uint8_t* tile_flags,
                             int32_t* tile_list, int32_t* d_na, int32_t* counts, int32_t* idx,
                             int32_t* targets_c, uint8_t* lvalid, int32_t* d_nk, int* status,
                             cudaStream_t s) {
  const int64_t T = (N + 255) / 256;
  tile_flags_kernel<<<static_cast<unsigned>(T), 256, 0, s>>>(keep, N, tile_flags);
  cudaError_t e = launch_compact(tile_flags, nullptr, T, 1, 0, tile_list, nullptr, d_na, counts,
                                 status, s);
  if (e != cudaSuccess) return e;
  tile_rows_kernel<<<static_cast<unsigned>(T), 256, 0, s>>>(keep, targets, N, V_valid, t_offset,
                                                             tile_list, d_na, idx, targets_c,
                                                             lvalid, d_nk, status);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const __nv_bfloat16* hidden, const int32_t* idx,
                               const int32_t* d_nk, int chunk_index, int chunk_rows, int H,
                               __nv_bfloat16* hc, int64_t N, int* status, cudaStream_t s) {
  const int vec = H / 8;
  gather_rows_kernel<<<blocks_for(chunk_rows, 8), 256, 0, s>>>(
      reinterpret_cast<const uint4*>(hidden), idx, d_nk, chunk_index, chunk_rows, vec,
      reinterpret_cast<uint4*>(hc), N, status);
  return cudaGetLastError();
}

cudaError_t launch_merge(const float4* part, int num_vt, const int32_t* d_nk, int chunk_index,
                         int chunk_rows, int want_entropy, float* lp_c, float* ent_c,
                         float* lse_c, float4* raw_c, cudaStream_t s) {
  merge_kernel<<<blocks_for(chunk_rows, kMergeRows), 256, 0, s>>>(
      part, num_vt, d_nk, chunk_index, chunk_rows, want_entropy, lp_c, ent_c, lse_c, raw_c);
  return cudaGetLastError();
}

cudaError_t launch_merge_shards(const float4* partials, int num_shards, const uint8_t* keep,
                                int64_t N, int want_entropy, float* lp, float* ent, float* lse,
                                cudaStream_t s) {
  merge_shards_kernel<<<blocks_for(N, 256), 256, 0, s>>>(partials, num_shards, keep, N,
                                                         want_entropy, lp, ent, lse);
  return cudaGetLastError();
}

cudaError_t launch_expand4(const uint8_t* keep, const int32_t* idx, const int32_t* d_nk, int64_t N,
                           const float4* src, float4* dst, int* status, cudaStream_t s) {
  expand4_kernel<<<blocks_for(N, 256), 256, 0, s>>>(keep, idx, d_nk, N, src, dst, status);
  return cudaGetLastError();
}

cudaError_t launch_expand3(const uint8_t* keep, const int32_t* idx, const int32_t* d_nk,
                           int64_t N, const float* a_c, const float* b_c, const float* c_c,
                           float* a, float* b, float* c, const uint8_t* lvalid, int* status,
                           cudaStream_t s) {
  // compact rows may reach N rounded up to 256 in block-sparse mode
  expand3_kernel<<<blocks_for((N + 255) / 256 * 256, 256), 256, 0, s>>>(
      keep, idx, d_nk, N, a_c, b_c, c_c, a, b, c, lvalid, status);
  return cudaGetLastError();
}

cudaError_t launch_expand(const float* src, const int32_t* idx, const int32_t* d_nk, int64_t N,
                          float* dst, int32_t* status, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(dst, 0, static_cast<size_t>(N) * sizeof(float), s);
  if (e != cudaSuccess) return e;
  scatter_vals_kernel<<<blocks_for(N, 256), 256, 0, s>>>(src, idx, d_nk, N, dst, status);
  return cudaGetLastError();
}

cudaError_t launch_gather_vec(const int32_t* idx, const int32_t* d_nk, int64_t N, const float* a,
                              const float* b, const float* c, const float* d, float* a_c,
                              float* b_c, float* c_c, float* d_c, int* status, cudaStream_t s) {
  gather_vec_kernel<<<blocks_for((N + 255) / 256 * 256, 256), 256, 0, s>>>(
      idx, d_nk, a, b, c, d, a_c, b_c, c_c, d_c, N, status);
  return cudaGetLastError();
}

cudaError_t launch_dh_reduce(const float* part, const int32_t* d_nk, int chunk_index,
                             int chunk_rows, int H, int tile_m, int tile_n, int workers, int num_kb,
                             int max_split, int fill_pct, const int32_t* idx,
                             const uint8_t* lvalid, __nv_bfloat16* dhidden, int64_t N,
                             int* status, cudaStream_t s) {
  // the chunk's largest tile grid (its rows are known only on the device);
  // blocks past the chunk's tiles, and of tiles taken whole, return
  const int64_t tiles = static_cast<int64_t>((chunk_rows + tile_m - 1) / tile_m) *
                        ((H + tile_n - 1) / tile_n);
  const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(tile_m / 32));
  dh_reduce_kernel<<<grid, 256, 0, s>>>(
      reinterpret_cast<const float4*>(part), d_nk, chunk_index, chunk_rows, H, tile_m, tile_n,
      workers, num_kb, max_split, fill_pct, idx, lvalid, reinterpret_cast<uint2*>(dhidden), N,
      status);
  return cudaGetLastError();
}

cudaError_t launch_zero_skipped_rows(const uint8_t* keep, int64_t N, int H,
                                     __nv_bfloat16* dhidden, cudaStream_t s) {
  zero_skipped_rows_kernel<<<blocks_for(N, 8), 256, 0, s>>>(keep, N, H / 8,
                                                           reinterpret_cast<uint4*>(dhidden));
  return cudaGetLastError();
}

}  // namespace lmhead
