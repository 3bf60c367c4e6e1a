// Internal interfaces between the C-ABI layer and the kernels.
#pragma once

#include <cstdint>
#include <initializer_list>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace lmhead {

// True when every non-null pointer is device memory of the current device
// (or managed memory).  A host pointer or another GPU's memory passed as a
// kernel buffer would make the kernels fault; the entry points refuse it
// with LMHEAD_EINVAL instead.
inline bool device_ptrs_ok(std::initializer_list<const void*> ptrs) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  for (const void* ptr : ptrs) {
    if (ptr == nullptr) continue;
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
      cudaGetLastError();  // not a sticky error: clear it
      return false;
    }
    if (a.type == cudaMemoryTypeManaged) continue;
    if (a.type != cudaMemoryTypeDevice || a.device != dev) return false;
  }
  return true;
}

// Debug builds (-DLMHEAD_DEBUG): every index the kernels derive from data is
// checked before the access it guards; a failed check records LMHEAD_EBOUNDS
// (7) in the status word and the access is skipped, so a wrong index shows up
// as a status instead of as a stray memory access.  Release builds compile the
// checks out (LM_DCHECK is then the constant true).
#ifdef LMHEAD_DEBUG
__device__ __forceinline__ bool lm_index_ok(bool ok, int* status) {
  if (!ok && status != nullptr) atomicCAS(status, 0, 7);
  return ok;
}
#define LM_DCHECK(cond, status) lm_index_ok((cond), (status))
#else
#define LM_DCHECK(cond, status) true
#endif

// Tile shape of the tcgen05 GEMM: 128 x 256 fp32 accumulator in TMEM,
// 64-element (128-byte) K steps staged by TMA with the 128-byte swizzle.
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kGemmThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kABytes = kBM * kBK * 2;
constexpr int kBBytes = kBN * kBK * 2;

// The four contractions of the path.
//   kFwd: Z = Hc W^T  -> per-row online-softmax partials per 256-column tile
//   kDz : Z = Hc W^T  -> dZ (bf16) from the recomputed logits
//   kDh : dHc = dZ W  -> rows scattered to dhidden (bf16)
//   kDw : dW (+)= dZ^T Hc (fp32)
enum GemmMode : int { kFwd = 0, kDz = 1, kDh = 2, kDw = 3 };

// Output staging of the kDz / kDw epilogues: per epilogue warp two 4 KB
// buffers, each one TMA box of 32 rows x 128 bytes (128-byte swizzle).
constexpr int kOutBoxBytes = 32 * 128;
constexpr int kOutStageBytes = 4 * 2 * kOutBoxBytes;
constexpr int out_stage_bytes(int mode) {
  return (mode == kDz || mode == kDw) ? kOutStageBytes : 0;
}
template <int MODE>
constexpr int gemm_smem_bytes() {
  return kStages * (kABytes + kBBytes) + out_stage_bytes(MODE) + 1024 + 256;
}

struct TcGemmParams {
  const int32_t* d_nk;      // device Nk
  int chunk_index;          // which chunk of the kept rows (see chunk_span)
  int chunk_rows;           // C: most rows per chunk (multiple of 256)
  int V;
  int H;
  int group_m;              // M tiles per raster block, 0 = none (see tile_coords)
  int group_n;              // N tiles per raster group when group_m == 0
  int64_t n_rows;           // N, rows of the batch (index checks of debug builds)
  int* status;              // device status word
  // epilogue operands (compact, indexed by compact row)
  const int32_t* targets_c;
  const int32_t* idx;
  const float* lse_c;
  const float* ent_c;
  const float* glp_c;
  const float* gent_c;      // nullable: metric-only entropy
  int want_entropy;
  float4* part;             // kFwd: [ceil(V/kBN)][C] (m, s, u, t)
  __nv_bfloat16* dhidden;   // kDh: [N, H]
  int beta;                 // kDw: 1 = add to dW (the output map's tensor)
  float* dh_part;           // kDh: [max_split][C][H] fp32 partial sums of split
                            //   tiles, by part (work_schedule)
  int max_split;            // kDh: most K parts of a tile (1 = never split K)
  int split_fill_pct;       // kDh: split only below this fill of the worker slots
  int stall;                // fault injection: the producer issues no loads, so
                            //   the pipeline waits run out (device ETIMEOUT)
  // Block-sparse mode (tile skipping in place): the "compact rows" are the
  // rows of the active 256-row tiles of the batch, read from hidden directly.
  const int32_t* tile_list; // active tiles (row / 256), or nullptr (compaction)
  const uint8_t* lvalid;    // per compact row: 1 if it is a kept row
};

// tma_c is the output map of kDz (dZ chunk, bf16, boxes of 32 rows x 64
// columns) and kDw (dW, fp32, boxes of 32 rows x 32 columns), both with the
// 128-byte swizzle; the other contractions do not read it.
template <int MODE>
cudaError_t launch_tc_gemm(const CUtensorMap& tma_a, const CUtensorMap& tma_b,
                           const CUtensorMap& tma_c, const TcGemmParams& p, int grid,
                           cudaStream_t stream);

// The same contractions on CTA pairs (cta_group::2, tc_gemm2.cuh): tiles of
// 256 rows x NSUB * 256 columns (NSUB = 1: two double-buffered 256-column
// accumulators; NSUB = 2: one 512-column accumulator).  `grid` must be even;
// the B maps use 128-row boxes for K-major B (each CTA stages half of every
// 256-column block of B).
template <int MODE, int NSUB>
cudaError_t launch_tc_gemm_pair(const CUtensorMap& tma_a, const CUtensorMap& tma_b,
                                const CUtensorMap& tma_c, const TcGemmParams& p, int grid,
                                cudaStream_t stream);

// The Nk kept rows are cut into ceil(Nk / C) chunks of equal size rounded up
// to 256 rows (so no chunk is much shorter than the others and the per-chunk
// cost of the weight-gradient update stays hidden behind its MMAs).  Chunk c
// covers compact rows [start, start + rows); rows == 0 past the last chunk.
// Computed on the device from Nk, so the host never waits for Nk.
__host__ __device__ __forceinline__ void chunk_span(int nk, int C, int c, int& start, int& rows) {
  if (nk <= 0) {
    start = 0;
    rows = 0;
    return;
  }
  const int nchunks = (nk + C - 1) / C;
  if (c >= nchunks) {
    start = nk;
    rows = 0;
    return;
  }
  const int per = (nk + nchunks - 1) / nchunks;
  const int cb = (per + 255) & ~255;  // <= C because C is a multiple of 256
  start = c * cb;
  rows = nk - start < cb ? nk - start : cb;
}

// Work schedule of one persistent GEMM launch over `tiles` output tiles of
// `num_kb` K blocks each, taken by `workers` persistent workers (CTA pairs or
// CTAs) in units of one tile and a range of its K blocks.  Worker w takes
// units w, w + W, w + 2W, ..., so the units in flight at any time are
// neighbours in unit order and walk their K ranges in step: the operand
// slices they share are read from DRAM once and then from L2.
//
// Plain: every unit is one whole tile.  Every contraction but dHidden, and
// dHidden when the last wave of tiles fills at least fill_pct of the worker
// slots (measured on GB300, a partly idle last wave costs less than its share
// of tiles: the few workers left run faster).
//
// Split tail (dHidden otherwise; K = V is long and the tile grid small): the
// tiles of the whole waves stay whole, and each of the R tiles of the last
// wave is cut into S equal K parts, so the last wave takes 1/S of a whole
// tile's time (S in 2 .. max_split, chosen for the fewest tail rounds per
// part; R * S units may take more than one round).  Parts with the same index
// share their K range, so the tail walks K in step too.  Its tiles get S fp32
// partial sums, slot p for part p, that the dHidden reduction adds in slot
// order; whole tiles write their bf16 rows to dhidden directly.  (Cutting the
// iterations into equal ranges per worker instead -- stream-K -- balances the
// waves exactly, but each worker then starts at its own K offset: measured on
// the half-kept 64K-token step, dHidden fetched so much more from DRAM that
// the step took 3.5% longer.)
struct WorkSched {
  int tiles = 0;
  int num_kb = 0;
  int workers = 0;
  int full = 0;        // tiles taken whole: 0 .. full-1 (all tiles when split == 1)
  int split = 1;       // K parts of each tail tile full .. tiles-1

  __host__ __device__ __forceinline__ int units() const {
    return full + (tiles - full) * split;
  }
  // Units (workers' partial sums) of tile t: 1 for a tile taken whole.
  __host__ __device__ __forceinline__ int tile_slots(int t) const {
    return t < full ? 1 : split;
  }
};

__host__ __device__ __forceinline__ WorkSched work_schedule(int tiles, int workers, int num_kb,
                                                            bool may_split, int max_split,
                                                            int fill_pct) {
  WorkSched s;
  s.tiles = tiles;
  s.num_kb = num_kb;
  s.workers = workers;
  s.full = tiles;
  if (!may_split || tiles <= 0 || workers <= 0 || max_split < 2 || num_kb < 2) return s;
  const long long slots = static_cast<long long>((tiles + workers - 1) / workers) * workers;
  if (static_cast<long long>(tiles) * 100 >= slots * fill_pct) return s;
  const int rem = tiles % workers;  // > 0: the last wave is not full
  // tail time in units of a whole tile's time: ceil(rem * S / W) rounds of 1/S
  int best = 1;
  long long best_rounds = 1;  // rounds of the unsplit tail
  for (int S = 2; S <= max_split && S <= num_kb; ++S) {
    const long long rounds = (static_cast<long long>(rem) * S + workers - 1) / workers;
    if (rounds * best < best_rounds * S) {  // rounds / S < best_rounds / best
      best = S;
      best_rounds = rounds;
    }
  }
  if (best == 1) return s;
  s.full = tiles - rem;
  s.split = best;
  return s;
}

// One unit of a worker's work: K blocks [kb0, kb1) of tile `tile`, part
// `slot` of the `slots` parts the tile is cut into.
struct WorkSeg {
  int tile, kb0, kb1, slot, slots;
};

// Walks one worker's units in order.  The producer, the MMA issuer and the
// epilogue of a worker each walk them with their own iterator, so all three
// see the same sequence.
struct SegIter {
  WorkSched s;
  int u;

  __host__ __device__ __forceinline__ SegIter(const WorkSched& sched, int w) : s(sched), u(w) {}
  // Fills g with the next unit; false when the worker has no more work.
  __host__ __device__ __forceinline__ bool next(WorkSeg& g) {
    if (u >= s.units()) return false;
    if (u < s.full) {
      g = WorkSeg{u, 0, s.num_kb, 0, 1};
    } else {
      const int rem = s.tiles - s.full;
      const int part = (u - s.full) / rem;
      g.tile = s.full + (u - s.full - part * rem);
      g.kb0 = static_cast<int>(static_cast<int64_t>(part) * s.num_kb / s.split);
      g.kb1 = static_cast<int>(static_cast<int64_t>(part + 1) * s.num_kb / s.split);
      g.slot = part;
      g.slots = s.split;
    }
    u += s.workers;
    return true;
  }
};

// Block-sparse mode: row of the hidden states behind compact row (cstart + lrow),
// where the compact rows are the rows of the active 256-row tiles in order.
__device__ __forceinline__ int sparse_row(const int32_t* tile_list, int cstart, int lrow) {
  const int l = cstart + lrow;
  return tile_list[l >> 8] * 256 + (l & 255);
}

// Rows counted by one block of the compaction scan (rowops.cu).
constexpr int kCompactRowsPerBlock = 4096;

// Row kernels (rowops.cu).
cudaError_t launch_build_keep(const float* c0, const float* c1, const float* c2,
                              const int32_t* offsets, int n_seq, int64_t N, uint8_t* keep,
                              cudaStream_t s);
// Targets are checked against [0, V_valid) and stored minus t_offset.
cudaError_t launch_compact(const uint8_t* keep, const int64_t* targets, int64_t N,
                           int64_t V_valid, int64_t t_offset, int32_t* idx, int32_t* targets_c,
                           int32_t* d_nk, int32_t* counts, int* status, cudaStream_t s);
// Block-sparse mode: active 256-row tiles (any kept row), compacted to
// tile_list[0..Na) with Na at d_na; then the per-compact-row arrays for the
// Na * 256 rows of those tiles: idx (row of the batch, clamped to N-1),
// targets_c (checked against [0, V_valid), minus t_offset), lvalid (kept
// row), and d_nk = Na * 256.
cudaError_t launch_tile_scan(const uint8_t* keep, const int64_t* targets, int64_t N,
                             int64_t V_valid, int64_t t_offset, uint8_t* tile_flags,
                             int32_t* tile_list, int32_t* d_na, int32_t* counts, int32_t* idx,
                             int32_t* targets_c, uint8_t* lvalid, int32_t* d_nk, int* status,
                             cudaStream_t s);
// (N and status serve the index checks of debug builds.)
cudaError_t launch_gather_rows(const __nv_bfloat16* hidden, const int32_t* idx,
                               const int32_t* d_nk, int chunk_index, int chunk_rows, int H,
                               __nv_bfloat16* hc, int64_t N, int* status, cudaStream_t s);
cudaError_t launch_merge(const float4* part, int num_vt, const int32_t* d_nk, int chunk_index,
                         int chunk_rows, int want_entropy, float* lp_c, float* ent_c,
                         float* lse_c, float4* raw_c, cudaStream_t s);
cudaError_t launch_merge_shards(const float4* partials, int num_shards, const uint8_t* keep,
                                int64_t N, int want_entropy, float* lp, float* ent, float* lse,
                                cudaStream_t s);
cudaError_t launch_expand4(const uint8_t* keep, const int32_t* idx, const int32_t* d_nk, int64_t N,
                           const float4* src, float4* dst, int* status, cudaStream_t s);
cudaError_t launch_expand3(const uint8_t* keep, const int32_t* idx, const int32_t* d_nk,
                           int64_t N, const float* a_c, const float* b_c, const float* c_c,
                           float* a, float* b, float* c, const uint8_t* lvalid, int* status,
                           cudaStream_t s);
cudaError_t launch_expand(const float* src, const int32_t* idx, const int32_t* d_nk, int64_t N,
                          float* dst, int32_t* status, cudaStream_t s);
cudaError_t launch_gather_vec(const int32_t* idx, const int32_t* d_nk, int64_t N,
                              const float* a, const float* b, const float* c, const float* d,
                              float* a_c, float* b_c, float* c_c, float* d_c, int* status,
                              cudaStream_t s);
// Sum of the dHidden partials of the chunk's split tail tiles
// (work_schedule), rows scattered to dhidden[idx] as bf16; tiles taken whole
// were written by the contraction itself.
cudaError_t launch_dh_reduce(const float* part, const int32_t* d_nk, int chunk_index,
                             int chunk_rows, int H, int tile_m, int tile_n, int workers, int num_kb,
                             int max_split, int fill_pct, const int32_t* idx,
                             const uint8_t* lvalid, __nv_bfloat16* dhidden, int64_t N,
                             int* status, cudaStream_t s);
cudaError_t launch_zero_skipped_rows(const uint8_t* keep, int64_t N, int H,
                                     __nv_bfloat16* dhidden, cudaStream_t s);

// Scoring of existing logits (logits_sls.cu); dtype 0 = bf16, 1 = float32.
cudaError_t launch_sls_fwd(const void* logits, int dtype, int64_t ld, const int64_t* targets,
                           const uint8_t* keep, int64_t N, int V, int want_entropy, float* lp,
                           float* ent, float* lse, int* status, cudaStream_t s);
cudaError_t launch_sls_bwd(const void* logits, int dtype, int64_t ld, const int64_t* targets,
                           const uint8_t* keep, int64_t N, int V, const float* lse,
                           const float* ent, const float* g_lp, const float* g_ent, void* dz,
                           int64_t ld_out, int* status, cudaStream_t s);

int device_sm_count();

}  // namespace lmhead
