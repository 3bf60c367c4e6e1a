// Persistent tcgen05 GEMM over clusters of four CTAs: two CTA pairs that
// share their A operand through TMA multicast.
//
// Same contractions, tiles and epilogues as the CTA-pair kernel
// (tc_gemm2.cuh): each pair computes a 256 x 256 tile with
// `tcgen05.mma.cta_group::2`.  The two pairs of a cluster take the same 256
// rows of A and two neighbouring column tiles (2j and 2j + 1), so every A
// byte is fetched from L2 once for both pairs: CTA r (cluster rank) loads the
// (r >> 1)-th 64-row quarter of A-half (r & 1) and multicasts it to the CTA
// holding that half in each pair (ranks r & 1 and (r & 1) + 2).  Per K step a
// cluster then reads 96 KB from L2 instead of 128 KB; under a power limit
// the operand traffic is energy that the tensor cores get back.
//
// Barriers: the full barrier of each pair's even CTA counts the bytes landing
// in both CTAs of its pair (its half of A from two sources, both halves of B)
// -- 64 KB per K step, as in the pair kernel.  A stage is refilled only after
// both pairs have consumed it: every MMA commit of either pair arrives on the
// empty barriers of all four CTAs (count 2).  Accumulator barriers stay per
// pair.  dHidden splits its K range by the same rule as the pair kernel,
// counting units of two column tiles and clusters as the workers.
#pragma once

#include <atomic>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace lmhead {

constexpr int kQuadStages = 6;
constexpr int kQuadABytes = 128 * kBK * 2;   // this CTA's half of A (two 64-row quarters)
constexpr int kQuadBBytes = 128 * kBK * 2;   // this CTA's half of B
template <int MODE>
constexpr int quad_smem_bytes() {
  return kQuadStages * (kQuadABytes + kQuadBBytes) + out_stage_bytes(MODE) + 1024 + 256;
}

template <int MODE>
__global__ void __cluster_dims__(4, 1, 1) __launch_bounds__(kGemmThreads, 1)
    tc_gemm_quad_kernel(const __grid_constant__ CUtensorMap tma_a,
                        const __grid_constant__ CUtensorMap tma_b,
                        const __grid_constant__ CUtensorMap tma_c, const TcGemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kQuadStages * kQuadABytes;
  uint8_t* sOut = sB + kQuadStages * kQuadBBytes;  // kDz / kDw output staging
  uint64_t* full = reinterpret_cast<uint64_t*>(sOut + out_stage_bytes(MODE));
  uint64_t* empty = full + kQuadStages;
  uint64_t* tfull = empty + kQuadStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t half = rank & 1u;          // which half of the pair's rows / columns
  const uint32_t pq = rank >> 1;            // which pair of the cluster
  const uint32_t pair_lead = rank & ~1u;    // the pair's even CTA (issues its MMAs)
  const uint16_t pair_mask = static_cast<uint16_t>(0x3u << (2u * pq));
  const bool leader = half == 0;
  const int cluster = static_cast<int>(blockIdx.x >> 2);
  const int num_clusters = static_cast<int>(gridDim.x >> 2);

  int cstart, rows_valid, M, N, K;
  if (!gemm_extents<MODE>(p, cstart, rows_valid, M, N, K)) return;  // uniform over the grid
  const int num_m = (M + kPairTileM - 1) / kPairTileM;
  const int num_n = (N + kBN - 1) / kBN;
  const int num_np = (num_n + 1) / 2;       // column-tile pairs
  const int num_kb = (K + kBK - 1) / kBK;
  const int num_base = num_m * num_np;
  const int splits =
      MODE == kDh ? dh_split_count(num_base, num_clusters, num_kb, p.max_split, p.split_fill_pct) : 1;
  const int num_units = num_base * splits;
  if (cluster >= num_units) return;  // the four CTAs of the cluster leave together

  if (threadIdx.x == 0) {
    for (int s = 0; s < kQuadStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 2);  // one commit from each pair
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);  // 4 epilogue warps in each CTA of the pair
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
  cluster_sync();  // barriers of all four CTAs initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      const uint16_t a_mask = static_cast<uint16_t>((1u << half) | (1u << (half + 2u)));
      for (int u = cluster; u < num_units && !p.stall; u += num_clusters) {
        const int sidx = u / num_base;
        const int kb0 = static_cast<int>(static_cast<int64_t>(sidx) * num_kb / splits);
        const int kb1 = static_cast<int>(static_cast<int64_t>(sidx + 1) * num_kb / splits);
        int mt, ntp;
        tile_coords(u % num_base, num_m, num_np, p.group_m, p.group_n, mt, ntp);
        const int nt = 2 * ntp + static_cast<int>(pq);
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * (kQuadABytes + kQuadBBytes));
          const uint32_t bar = map_to_cta(smem_addr(&full[stage]), pair_lead);
          uint8_t* a_dst = sA + stage * kQuadABytes + pq * 8192;  // this CTA's quarter
          uint8_t* b_dst = sB + stage * kQuadBBytes;
          const int k0 = kb * kBK;
          const int m0 = mt * kPairTileM + static_cast<int>(half) * 128 + static_cast<int>(pq) * 64;
          const int n0 = nt * kBN + static_cast<int>(half) * 128;
          if (MODE == kDw) {
            tma_load_2d_pair_mc(a_dst, &tma_a, bar, m0, k0, a_mask);
          } else {
            tma_load_2d_pair_mc(a_dst, &tma_a, bar, k0, m0, a_mask);
          }
          if (MODE == kDh || MODE == kDw) {
            tma_load_2d_pair(b_dst, &tma_b, bar, n0, k0);
            tma_load_2d_pair(b_dst + 8192, &tma_b, bar, n0 + 64, k0);
          } else {
            tma_load_2d_pair(b_dst, &tma_b, bar, k0, n0);
          }
          ++issued;
          if (++stage == kQuadStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      // The even CTA of each pair sees every load landing in its pair
      // complete on its full barriers; let them land before it exits.
      if (leader) {
        for (int s = 0; s < kQuadStages; ++s) {
          const uint32_t uses =
              issued / kQuadStages + (static_cast<uint32_t>(s) < issued % kQuadStages ? 1u : 0u);
          if (uses > 0) mbar_wait_drain(&full[s], (uses - 1u) & 1u, p.status);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (leader && lane == 0) {
      constexpr bool a_mn = (MODE == kDw);
      constexpr bool b_mn = (MODE == kDh || MODE == kDw);
      constexpr uint32_t idesc = idesc_bf16(kPairTileM, kBN, a_mn, b_mn);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int u = cluster; u < num_units && ok && num_kb > 0; u += num_clusters, ++it) {
        const int sidx = u / num_base;
        const int kb0 = static_cast<int>(static_cast<int64_t>(sidx) * num_kb / splits);
        const int kb1 = static_cast<int>(static_cast<int64_t>(sidx + 1) * num_kb / splits);
        const int acc = it & 1;
        const uint32_t use = static_cast<uint32_t>(it >> 1);
        if (!mbar_wait(&tempty[acc], (use & 1u) ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_addr = smem_addr(sA + stage * kQuadABytes);
          const uint32_t b_addr = smem_addr(sB + stage * kQuadBBytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t ad = a_mn ? smem_desc_sw128(a_addr + k * 2048, 8192, 1024)
                                     : smem_desc_sw128(a_addr + k * 32, 16, 1024);
            const uint64_t bd = b_mn ? smem_desc_sw128(b_addr + k * 2048, 8192, 1024)
                                     : smem_desc_sw128(b_addr + k * 32, 16, 1024);
            umma_bf16_pair(d_tmem, ad, bd, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
          }
          umma_commit_pair(&empty[stage], 0xF);  // both pairs' producers wait for it
          if (++stage == kQuadStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit_pair(&tfull[acc], pair_mask);
      }
      umma_commit_pair(drain, static_cast<uint16_t>(1u << rank));
      mbar_wait_drain(drain, 0, p.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const int row_local = static_cast<int>(half) * 128 + q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    OutStage os{&tma_c, sOut + (warp - 2) * 2 * kOutBoxBytes, 0u};
    int it = 0;
    for (int u = cluster; u < num_units; u += num_clusters, ++it) {
      const int sidx = u / num_base;
      int mt, ntp;
      tile_coords(u % num_base, num_m, num_np, p.group_m, p.group_n, mt, ntp);
      const int nt = 2 * ntp + static_cast<int>(pq);
      const int acc = it & 1;
      const uint32_t use = static_cast<uint32_t>(it >> 1);
      if (num_kb > 0) {
        if (!mbar_wait(&tfull[acc], use & 1u, abort_flag, p.status)) break;
        tc_fence_after();
      }
      const uint32_t tbase = tmem_base + lane_off + static_cast<uint32_t>(acc * kBN);
      const uint32_t te = map_to_cta(smem_addr(&tempty[acc]), pair_lead);
      // (the second pair's column tile may lie past N when N has an odd
      // number of tiles: the epilogues write nothing past N)
      epilogue_tile<MODE>(p, tbase, mt * kPairTileM + row_local, nt, cstart, rows_valid,
                          num_kb > 0, sidx, splits, os, [&] {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive_cluster(te);
                          });
    }
    // the output writes have finished before the CTA's shared memory goes
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  cluster_sync();  // every MMA and every (multicast) load of the cluster is done
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

// Clusters of four that fit on the device at once with this kernel's shared
// memory (not every GPC holds a multiple of four SMs), cached per device.
template <int MODE>
int quad_max_clusters(int dev) {
  static std::atomic<int> cached[64];  // zero-initialised (static storage)
  if (dev < 0 || dev >= 64) return 0;
  int n = cached[dev].load(std::memory_order_acquire);
  if (n == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(4, 1, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = quad_smem_bytes<MODE>();
    if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_quad_kernel<MODE>, &cfg) != cudaSuccess ||
        n < 1) {
      cudaGetLastError();
      return 0;
    }
    cached[dev].store(n, std::memory_order_release);
  }
  return n;
}

template <int MODE>
cudaError_t launch_tc_gemm_quad(const CUtensorMap& tma_a, const CUtensorMap& tma_b,
                                const CUtensorMap& tma_c, const TcGemmParams& p,
                                int64_t units, cudaStream_t stream, int* clusters_out) {
  static std::atomic<bool> configured[64];  // zero-initialised (static storage)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(tc_gemm_quad_kernel<MODE>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, quad_smem_bytes<MODE>());
    if (e != cudaSuccess) return e;
    configured[dev].store(true, std::memory_order_release);
  }
  const int maxc = quad_max_clusters<MODE>(dev);
  if (maxc < 1) return cudaErrorLaunchOutOfResources;
  const int64_t clusters = units < maxc ? (units < 1 ? 1 : units) : maxc;
  if (clusters_out != nullptr) *clusters_out = static_cast<int>(clusters);
  tc_gemm_quad_kernel<MODE><<<static_cast<unsigned>(4 * clusters), kGemmThreads,
                              quad_smem_bytes<MODE>(), stream>>>(tma_a, tma_b, tma_c, p);
  return cudaGetLastError();
}

}  // namespace lmhead
