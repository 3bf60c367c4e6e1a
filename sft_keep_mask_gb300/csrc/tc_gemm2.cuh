// Persistent tcgen05 GEMM over CTA pairs (clusters of two CTAs on two SMs).
//
// Same contraction and epilogues as the one-CTA kernel (tc_gemm.cuh), with
// tiles computed by `tcgen05.mma.cta_group::2`: each CTA of the pair stages
// its 128-row half of A and its 128-row half of every 256-column block of B,
// the even CTA issues the MMAs for both, and each CTA's tensor memory
// receives its 128 accumulator rows.  Two tile widths (NSUB 256-column
// blocks per tile):
//
//   NSUB = 1  256 x 256 tiles, two 256-column accumulators, so the epilogue
//             of tile i overlaps the MMAs of tile i + 1; 32 KB per CTA and K
//             step, six stages.  Every operand byte fetched from L2 feeds 1.5
//             times the FLOPs of the one-CTA tile.
//   NSUB = 2  256 x 512 tiles in one 512-column accumulator (all of TMEM):
//             each 64-wide K step issues two N = 256 MMAs that share the A
//             half, so a K step stages 48 KB per CTA for twice the FLOPs --
//             a quarter fewer operand bytes per FLOP than NSUB = 1 -- and, with
//             twice the output in flight, the column operand streams past
//             half as often.  The accumulator is released in two 256-column
//             halves, so the next tile's MMAs into the first half overlap the
//             epilogue's drain of the second; the drain of the first half is
//             not overlapped, which pays where K is long (dHidden: K = V; dW:
//             K = the chunk's rows).  Four stages.
//
//   warp 0      TMA producer of this CTA's halves; both CTAs count the bytes
//               on the even CTA's full barrier
//   warp 1      TMEM allocation (both CTAs, collectively) and, in the even
//               CTA, the MMA issuer; its commits arrive on the barriers of
//               both CTAs (tcgen05.commit with a CTA mask: an mbarrier
//               arrive, no memory is read)
//   warps 2..5  epilogue of this CTA's 128 rows; one elected lane per warp
//               releases the accumulator on the even CTA's barrier and, for
//               kDz / kDw, issues the warp's TMA output writes
#pragma once

#include <atomic>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace lmhead {

constexpr int kPairABytes = 128 * kBK * 2;   // this CTA's half of A
constexpr int kPairBBytes = 128 * kBK * 2;   // this CTA's half of one 256-column block of B
template <int NSUB>
constexpr int pair_stages() {
  return NSUB == 1 ? 6 : 4;
}
template <int MODE, int NSUB>
constexpr int pair_smem_bytes() {
  return pair_stages<NSUB>() * (kPairABytes + NSUB * kPairBBytes) + out_stage_bytes(MODE) + 1024 +
         256;
}
static_assert(pair_smem_bytes<kDz, 2>() <= 232448, "wide tile stages exceed shared memory");
constexpr int kPairTileM = 256;

template <int MODE, int NSUB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGemmThreads, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tma_a,
                        const __grid_constant__ CUtensorMap tma_b,
                        const __grid_constant__ CUtensorMap tma_c, const TcGemmParams p) {
  constexpr int kStg = pair_stages<NSUB>();
  constexpr int kBStage = NSUB * kPairBBytes;   // this CTA's B bytes per stage
  constexpr int kTileN = NSUB * kBN;            // columns of a tile
  constexpr int kNumAcc = NSUB == 1 ? 2 : 1;    // accumulators in the 512 TMEM columns
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStg * kPairABytes;
  uint8_t* sOut = sB + kStg * kBStage;  // kDz / kDw output staging
  uint64_t* full = reinterpret_cast<uint64_t*>(sOut + out_stage_bytes(MODE));
  uint64_t* empty = full + kStg;
  uint64_t* tfull = empty + kStg;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int num_pairs = static_cast<int>(gridDim.x >> 1);

  int cstart, rows_valid, M, N, K;
  if (!gemm_extents<MODE>(p, cstart, rows_valid, M, N, K)) return;  // uniform over the grid
  const int num_m = (M + kPairTileM - 1) / kPairTileM;
  const int num_n = (N + kTileN - 1) / kTileN;
  const int num_kb = (K + kBK - 1) / kBK;
  const int num_tiles = num_m * num_n;
  const WorkSched sched =
      work_schedule(num_tiles, num_pairs, num_kb, MODE == kDh, p.max_split, p.split_fill_pct);
  WorkSeg seg;
  if (!SegIter(sched, pair).next(seg)) return;  // no work: both CTAs of the pair leave together

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStg; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);  // 4 epilogue warps in each CTA
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
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      const int half = static_cast<int>(rank) * 128;
      SegIter segs(sched, pair);
      for (WorkSeg g; !p.stall && segs.next(g);) {
        int mt, nt;
        tile_coords(g.tile, num_m, num_n, p.group_m, p.group_n, mt, nt);
        bool ok = true;
        for (int kb = g.kb0; kb < g.kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status, kSiteProducerEmpty)) { ok = false; break; }
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * (kPairABytes + kBStage));
          const uint32_t bar = map_to_cta(smem_addr(&full[stage]), 0);
          uint8_t* a_dst = sA + stage * kPairABytes;
          uint8_t* b_dst = sB + stage * kBStage;
          const int k0 = kb * kBK;
          const int m0 = mt * kPairTileM + half;
          if (MODE == kDw) {
            tma_load_2d_pair(a_dst, &tma_a, bar, m0, k0);
            tma_load_2d_pair(a_dst + 8192, &tma_a, bar, m0 + 64, k0);
          } else {
            // block-sparse: the compact rows are read in place from hidden
            const int ay = (MODE != kDh && p.tile_list != nullptr)
                               ? sparse_row(p.tile_list, cstart, m0) : m0;
            tma_load_2d_pair(a_dst, &tma_a, bar, k0, ay);
          }
#pragma unroll
          for (int h = 0; h < NSUB; ++h) {
            // this CTA's 128 columns of the tile's h-th 256-column block
            const int n0 = nt * kTileN + h * kBN + half;
            uint8_t* bh = b_dst + h * kPairBBytes;
            if (MODE == kDh || MODE == kDw) {
              const int by = (MODE == kDw && p.tile_list != nullptr)
                                 ? sparse_row(p.tile_list, cstart, k0) : k0;
              tma_load_2d_pair(bh, &tma_b, bar, n0, by);
              tma_load_2d_pair(bh + 8192, &tma_b, bar, n0 + 64, by);
            } else {
              tma_load_2d_pair(bh, &tma_b, bar, k0, n0);
            }
          }
          ++issued;
          if (++stage == kStg) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      // The even CTA sees every load of the pair complete on its full
      // barriers; let them land before it exits.
      if (leader) {
        for (int s = 0; s < kStg; ++s) {
          const uint32_t uses =
              issued / kStg + (static_cast<uint32_t>(s) < issued % kStg ? 1u : 0u);
          if (uses > 0) mbar_wait_drain(&full[s], (uses - 1u) & 1u, p.status, kSiteProducerDrain);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (leader && lane == 0) {
      constexpr bool a_mn = (MODE == kDw);
      constexpr bool b_mn = (MODE == kDh || MODE == kDw);
      constexpr uint32_t idesc = idesc_bf16(kPairTileM, kBN, a_mn, b_mn);  // one N = 256 block
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      SegIter segs(sched, pair);
      for (WorkSeg g; ok && num_kb > 0 && segs.next(g); ++it) {
        const int kb0 = g.kb0;
        const int kb1 = g.kb1;

        // the MMAs of one K step into one 256-column block of the accumulator
        auto issue = [&](int st, int kbv, int h, uint32_t d_tmem) {
          const uint32_t a_addr = smem_addr(sA + st * kPairABytes);
          const uint32_t bh = smem_addr(sB + st * kBStage) + static_cast<uint32_t>(h * kPairBBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t ad = a_mn ? smem_desc_sw128(a_addr + k * 2048, 8192, 1024)
                                     : smem_desc_sw128(a_addr + k * 32, 16, 1024);
            const uint64_t bd = b_mn ? smem_desc_sw128(bh + k * 2048, 8192, 1024)
                                     : smem_desc_sw128(bh + k * 32, 16, 1024);
            umma_bf16_pair(d_tmem + static_cast<uint32_t>(h * kBN), ad, bd, idesc,
                           (kbv != kb0 || k != 0) ? 1u : 0u);
          }
        };
        if (NSUB == 1) {
          const int acc = it & 1;
          const uint32_t use = static_cast<uint32_t>(it >> 1);
          if (!mbar_wait(&tempty[acc], (use & 1u) ^ 1u, abort_flag, p.status,
                         kSiteIssuerTmemEmpty))
            break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(&full[stage], phase, abort_flag, p.status, kSiteIssuerFull)) { ok = false; break; }
            tc_fence_after();
            issue(stage, kb, 0, d_tmem);
            umma_commit_pair(&empty[stage], 0x3);
            if (++stage == kStg) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          umma_commit_pair(&tfull[acc], 0x3);
        } else {
          // One 512-column accumulator released in two 256-column halves
          // (tempty[0], tempty[1]) as the previous tile's epilogue drains
          // them.  The first-half MMAs of each K step start as soon as half 0
          // is free; the second-half MMAs of the filled stages are held, in K
          // order, until half 1 is free, and a stage is released only after
          // both halves have read it.  When every stage is held the issuer
          // waits for half 1, so the producer always gets a stage back.
          const uint32_t par = (static_cast<uint32_t>(it) & 1u) ^ 1u;
          if (!mbar_wait(&tempty[0], par, abort_flag, p.status, kSiteIssuerTmemEmpty)) break;
          tc_fence_after();
          bool hi = mbar_test_wait(&tempty[1], par);
          int held = 0, hstage = 0, hkb = 0;  // held stages: count, first stage, its K block
          auto release_held = [&]() {
            for (int i = 0; i < held; ++i) {
              const int st = (hstage + i) % kStg;
              issue(st, hkb + i, 1, tmem_base);
              umma_commit_pair(&empty[st], 0x3);
            }
            held = 0;
          };
          if (hi) tc_fence_after();
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait(&full[stage], phase, abort_flag, p.status, kSiteIssuerFull)) { ok = false; break; }
            tc_fence_after();
            issue(stage, kb, 0, tmem_base);
            if (!hi) {
              hi = mbar_test_wait(&tempty[1], par);
              if (!hi && held + 1 == kStg) {
                if (!mbar_wait(&tempty[1], par, abort_flag, p.status, kSiteIssuerTmemEmpty)) {
                  ok = false;
                  break;
                }
                hi = true;
              }
              if (hi) tc_fence_after();
            }
            if (hi) {
              release_held();
              issue(stage, kb, 1, tmem_base);
              umma_commit_pair(&empty[stage], 0x3);
            } else {
              if (held == 0) {
                hstage = stage;
                hkb = kb;
              }
              ++held;
            }
            if (++stage == kStg) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;
          if (held > 0) {
            if (!mbar_wait(&tempty[1], par, abort_flag, p.status, kSiteIssuerTmemEmpty)) break;
            tc_fence_after();
            release_held();
          }
          umma_commit_pair(&tfull[0], 0x3);
        }
      }
      umma_commit_pair(drain, 0x1);
      mbar_wait_drain(drain, 0, p.status, kSiteIssuerDrain);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int row_local = static_cast<int>(rank) * 128 + q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    OutStage os{&tma_c, sOut + (warp - 2) * 2 * kOutBoxBytes, 0u};
    int it = 0;
    SegIter segs(sched, pair);
    for (WorkSeg g; segs.next(g); ++it) {
      int mt, nt;
      tile_coords(g.tile, num_m, num_n, p.group_m, p.group_n, mt, nt);
      const int acc = it % kNumAcc;
      const uint32_t use = static_cast<uint32_t>(it / kNumAcc);
      if (num_kb > 0) {
        if (!mbar_wait(&tfull[acc], use & 1u, abort_flag, p.status, kSiteEpilogueFull)) break;
        tc_fence_after();
      }
      const uint32_t tbase = tmem_base + lane_off + static_cast<uint32_t>(acc * kBN);
      // the tile's 256-column blocks in turn, each released right after its
      // last TMEM load (one accumulator of two halves when NSUB = 2)
#pragma unroll 1
      for (int h = 0; h < NSUB; ++h) {
        const uint32_t te = map_to_cta(smem_addr(&tempty[NSUB == 1 ? acc : h]), 0);
        epilogue_tile<MODE>(p, tbase + static_cast<uint32_t>(h * kBN), mt * kPairTileM + row_local,
                            nt * NSUB + h, cstart, rows_valid, num_kb > 0, g.slot, g.slots, os, [&] {
                              tc_fence_before();
                              __syncwarp();
                              if (lane == 0) mbar_arrive_cluster(te);
                            });
      }
    }
    // the output writes have finished before the CTA's shared memory goes
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync();  // the pair's MMAs and loads are finished in both CTAs
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

template <int MODE, int NSUB>
cudaError_t launch_tc_gemm_pair(const CUtensorMap& tma_a, const CUtensorMap& tma_b,
                                const CUtensorMap& tma_c, const TcGemmParams& p, int grid,
                                cudaStream_t stream) {
  // the shared-memory opt-in is per device: set it once on each device used
  static std::atomic<bool> configured[64];  // zero-initialised (static storage)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(tc_gemm_pair_kernel<MODE, NSUB>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             pair_smem_bytes<MODE, NSUB>());
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_release);
  }
  tc_gemm_pair_kernel<MODE, NSUB><<<grid, kGemmThreads, pair_smem_bytes<MODE, NSUB>(), stream>>>(
      tma_a, tma_b, tma_c, p);
  return cudaGetLastError();
}

}  // namespace lmhead
