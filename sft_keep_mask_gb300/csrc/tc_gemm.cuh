// Persistent tcgen05 GEMM for the four contractions of the fused LM head,
// with the epilogue of each contraction fused in.
//
// D[M, N] = A[M, K] * B[N, K]^T, bf16 operands staged in shared memory by TMA
// (128-byte swizzle), fp32 accumulator in tensor memory.  One CTA per SM; it
// walks the tiles t = blockIdx.x, blockIdx.x + gridDim.x, ...
//
//   warp 0      TMA producer: a ring of kStages (A, B) stages
//   warp 1      TMEM owner and MMA issuer (one thread): 4 MMAs of
//               128 x 256 x 16 per 64-wide K step, into one of two 256-column
//               accumulators, so the epilogue of tile i overlaps the MMAs of
//               tile i+1
//   warps 2..5  epilogue: warp w reads TMEM lanes 32*(w%4) .. +31, i.e. one
//               accumulator row per thread, 32 columns per tcgen05.ld; kDz /
//               kDw stage their output in shared memory for TMA writes
//
// Operand majors per contraction (K-major = K contiguous in global memory):
//   kFwd, kDz : A = Hc [rows, H] K-major,  B = W [V, H] K-major
//   kDh       : A = dZ [rows, V] K-major,  B = W [V, H] MN-major (H contiguous)
//   kDw       : A = dZ [rows, V] MN-major (V contiguous),
//               B = Hc [rows, H] MN-major (H contiguous)
//
// The logits never leave the SM in the forward: the kFwd epilogue reduces
// each 128 x 256 tile to per-row (max, sum exp, sum exp * (z - max), target
// logit) -- the single fused projection of SkyRL pull request #2374
// ("How it works"), with the entropy -(p log p) of its gemini-code-assist
// review accumulated online in a numerically safe form.
#pragma once

#include <atomic>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace lmhead {

template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tma_a,
                   const __grid_constant__ CUtensorMap tma_b,
                   const __grid_constant__ CUtensorMap tma_c, const TcGemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint8_t* sOut = sB + kStages * kBBytes;  // kDz / kDw output staging
  uint64_t* full = reinterpret_cast<uint64_t*>(sOut + out_stage_bytes(MODE));
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  int cstart, rows_valid, M, N, K;
  if (!gemm_extents<MODE>(p, cstart, rows_valid, M, N, K)) return;
  const int num_m = (M + kBM - 1) / kBM;
  const int num_n = (N + kBN - 1) / kBN;
  const int num_kb = (K + kBK - 1) / kBK;
  const int num_tiles = num_m * num_n;
  const int worker = static_cast<int>(blockIdx.x);
  const WorkSched sched = work_schedule(num_tiles, static_cast<int>(gridDim.x), num_kb,
                                        MODE == kDh, p.max_split, p.split_fill_pct);
  WorkSeg seg;
  if (!SegIter(sched, worker).next(seg)) return;  // no work for this CTA

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tma_a);
    tma_prefetch_desc(&tma_b);
    if (out_stage_bytes(MODE) > 0) tma_prefetch_desc(&tma_c);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      SegIter segs(sched, worker);
      for (WorkSeg g; !p.stall && segs.next(g);) {
        int mt, nt;
        tile_coords(g.tile, num_m, num_n, p.group_m, p.group_n, mt, nt);
        bool ok = true;
        for (int kb = g.kb0; kb < g.kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status, kSiteProducerEmpty)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[stage], kABytes + kBBytes);
          uint8_t* a_dst = sA + stage * kABytes;
          uint8_t* b_dst = sB + stage * kBBytes;
          const int k0 = kb * kBK;
          if (MODE == kDw) {
            // A MN-major: dZ[k rows, m cols]; two 64-column boxes
            tma_load_2d(a_dst, &tma_a, &full[stage], mt * kBM, k0);
            tma_load_2d(a_dst + 8192, &tma_a, &full[stage], mt * kBM + 64, k0);
          } else {
            const int ay = (MODE != kDh && p.tile_list != nullptr)
                               ? sparse_row(p.tile_list, cstart, mt * kBM) : mt * kBM;
            tma_load_2d(a_dst, &tma_a, &full[stage], k0, ay);
          }
          if (MODE == kDh || MODE == kDw) {
            // B MN-major: [k rows, n cols]; four 64-column boxes
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tma_load_2d(b_dst + j * 8192, &tma_b, &full[stage], nt * kBN + 64 * j,
                          (MODE == kDw && p.tile_list != nullptr)
                              ? sparse_row(p.tile_list, cstart, k0) : k0);
          } else {
            tma_load_2d(b_dst, &tma_b, &full[stage], k0, nt * kBN);
          }
          ++issued;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      // Let every load that was issued land before the CTA exits.
      for (int s = 0; s < kStages; ++s) {
        const uint32_t uses = issued / kStages + (static_cast<uint32_t>(s) < issued % kStages ? 1u : 0u);
        if (uses > 0) mbar_wait_drain(&full[s], (uses - 1u) & 1u, p.status, kSiteProducerDrain);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr bool a_mn = (MODE == kDw);
      constexpr bool b_mn = (MODE == kDh || MODE == kDw);
      constexpr uint32_t idesc = idesc_bf16(kBM, kBN, a_mn, b_mn);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      SegIter segs(sched, worker);
      for (WorkSeg g; ok && num_kb > 0 && segs.next(g); ++it) {
        const int kb0 = g.kb0;
        const int kb1 = g.kb1;

        const int acc = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        if (!mbar_wait(&tempty[acc], (use & 1u) ^ 1u, abort_flag, p.status, kSiteIssuerTmemEmpty))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status, kSiteIssuerFull)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_addr(sA + stage * kABytes);
          const uint32_t b_addr = smem_addr(sB + stage * kBBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t ad = a_mn ? smem_desc_sw128(a_addr + k * 2048, 8192, 1024)
                                     : smem_desc_sw128(a_addr + k * 32, 16, 1024);
            const uint64_t bd = b_mn ? smem_desc_sw128(b_addr + k * 2048, 8192, 1024)
                                     : smem_desc_sw128(b_addr + k * 32, 16, 1024);
            umma_bf16(d_tmem, ad, bd, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
          }
          umma_commit(&empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
      }
      // No MMA may still be running when the accumulators are released.
      umma_commit(drain);
      mbar_wait_drain(drain, 0, p.status, kSiteIssuerDrain);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int row_local = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    OutStage os{&tma_c, sOut + (warp - 2) * 2 * kOutBoxBytes, 0u};
    int it = 0;
    SegIter segs(sched, worker);
    for (WorkSeg g; segs.next(g); ++it) {
      int mt, nt;
      tile_coords(g.tile, num_m, num_n, p.group_m, p.group_n, mt, nt);
      const int acc = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      if (num_kb > 0) {
        if (!mbar_wait(&tfull[acc], use & 1u, abort_flag, p.status, kSiteEpilogueFull)) break;
        tc_fence_after();
      }
      const uint32_t tbase = tmem_base + lane_off + static_cast<uint32_t>(acc * kBN);
      uint64_t* te = &tempty[acc];
      epilogue_tile<MODE>(p, tbase, mt * kBM + row_local, nt, cstart, rows_valid, num_kb > 0, g.slot, g.slots, os, [&] {
        tc_fence_before();
        mbar_arrive(te);
      });
    }
    // the output writes have finished before the CTA's shared memory goes
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

template <int MODE>
cudaError_t launch_tc_gemm(const CUtensorMap& tma_a, const CUtensorMap& tma_b,
                           const CUtensorMap& tma_c, const TcGemmParams& p, int grid,
                           cudaStream_t stream) {
  // the shared-memory opt-in is per device: set it once on each device used
  static std::atomic<bool> configured[64];  // zero-initialised (static storage)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(tc_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             gemm_smem_bytes<MODE>());
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_release);
  }
  tc_gemm_kernel<MODE><<<grid, kGemmThreads, gemm_smem_bytes<MODE>(), stream>>>(tma_a, tma_b, tma_c,
                                                                              p);
  return cudaGetLastError();
}

}  // namespace lmhead
