// fgemm_kernel_pair.cuh -- classical GEMM on CTA pairs (tcgen05 cta_group::2).
//
// A cluster of two CTAs computes one 256 x BN output tile: the even CTA's MMA
// thread issues M = 256 MMAs that read 128 rows of A and BN/2 columns of B from
// each CTA's shared memory and accumulate into 128 TMEM lanes of each CTA.
// Per CTA that halves the B operand traffic of a 128 x BN tile (shared-memory
// reads per MMA cycle drop from 96 to 64 bytes at BN = 256), and a 256 x 128
// pair tile is as cheap to feed as a 128 x 256 single-CTA tile.
//
// Barriers: each CTA's producer loads its own halves with TMA and counts the
// bytes on the EVEN CTA's full[s] barrier (cluster address), which expects the
// bytes of both; the MMA thread's commits arrive on empty[s] and tfull[b] in
// both CTAs (multicast); both CTAs' epilogue warps arrive on the even CTA's
// tempty[b] (8 arrivals).  Waits are bounded as in the single-CTA kernel.
#pragma once

#include <algorithm>

#include "fgemm_kernel.cuh"

namespace fgemm {

template <int BN>
struct PairCfg {
  static constexpr int kABytes = kBM * kBK * 2;        // this CTA's 128 rows of A
  static constexpr int kBBytes = kBK * (BN / 2) * 2;   // this CTA's BN/2 columns of B
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = BN == 256 ? 6 : 8;
  static constexpr int kTmemCols = BN == 256 ? 512 : 256;
  static constexpr int kBarBytes = 256;
  // One extra B half after the barriers: the MMA reads BN/2 columns of B per
  // CTA; the slack keeps even a full-width read of the last stage inside this
  // CTA's shared memory.
  static constexpr int kSlackBytes = kBBytes;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kBarBytes + kSlackBytes;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert(2 * BN <= kTmemCols, "two accumulator buffers must fit in TMEM");
  static_assert((2 * kStages + 5) * 8 + 4 <= kBarBytes, "barrier area too small");
};

template <int BN>
__global__ void __launch_bounds__(256, 1) fgemm_kernel_pair(const __grid_constant__ KernelParams p) {
  using PC = PairCfg<BN>;
  constexpr int S = PC::kStages;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  const uint32_t sA0 = base;
  const uint32_t sB0 = base + S * PC::kABytes;
  const uint32_t bar0 = base + S * PC::kStageBytes;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + S * PC::kStageBytes + 8 * (2 * S + 5));
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull = [&](uint32_t b) { return bar0 + 8u * (2 * S + b); };
  auto tempty = [&](uint32_t b) { return bar0 + 8u * (2 * S + 2 + b); };
  const uint32_t drain = bar0 + 8u * (2 * S + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(full(s), 1);
      ptx::mbar_init(empty(s), 1);
    }
    for (uint32_t b = 0; b < 2; ++b) {
      ptx::mbar_init(tfull(b), 1);
      ptx::mbar_init(tempty(b), 8);
    }
    ptx::mbar_init(drain, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), PC::kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();  // both CTAs' barriers exist before any remote arrive
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------- TMA producer (both CTAs)
    if (lane == 0) {
      ptx::prefetch_tmap(&p.tmap_a);
      ptx::prefetch_tmap(&p.tmap_b);
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      constexpr int HALF = BN / 2;
      for (int unit = cluster; ok && unit < p.num_units; unit += nclusters) {
        int tm, tn;
        unit_coords(p, unit, tm, tn);
        const int ay = tm * (2 * kBM) + static_cast<int>(rank) * kBM;
        int bx[BN / 128];
#pragma unroll
        for (int q = 0; q < BN / 128; ++q) {
          const int qc = static_cast<int>(rank) * HALF + q * 64;  // column inside the pair tile
          if (p.epi == kEpiSwiglu)
            bx[q] = qc < HALF ? tn * HALF + qc : p.n_out + tn * HALF + (qc - HALF);
          else
            bx[q] = tn * BN + qc;
        }
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_one(empty(s), ph ^ 1u, p, 0)) {
            ok = false;
            break;
          }
          const uint32_t fb = ptx::mapa(full(s), 0);
          if (leader) ptx::mbar_arrive_expect_tx(full(s), 2 * PC::kStageBytes);
          ptx::tma_load_2d_pair(sA0 + s * PC::kABytes, &p.tmap_a, kb * kBK, ay, fb);
#pragma unroll
          for (int q = 0; q < BN / 128; ++q)
            ptx::tma_load_2d_pair(sB0 + s * PC::kBBytes + q * 8192, &p.tmap_b, bx[q], kb * kBK, fb);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok && leader) {
        for (int i = 0; i < S; ++i) {
          if (--s < 0) {
            s = S - 1;
            ph ^= 1u;
          }
          wait_bounded(full(s), ph, p, err_code(0), false);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------- MMA issuer (even CTA only)
    if (lane == 0 && leader) {
      int s = 0;
      uint32_t ph = 0, acc_it = 0;
      bool ok = true;
      for (int unit = cluster; ok && unit < p.num_units; unit += nclusters) {
        const uint32_t buf = acc_it & 1u, aph = (acc_it >> 1) & 1u;
        ++acc_it;
        if (!wait_one(tempty(buf), aph ^ 1u, p, 1)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t dt = tmem_base + buf * BN;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_one(full(s), ph, p, 1)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t ad = ptx::sdesc(sA0 + s * PC::kABytes, 16, 1024);
          const uint64_t bd = ptx::sdesc(sB0 + s * PC::kBBytes, 8192, 1024);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            ptx::mma_f16_pair(dt, ad + static_cast<uint64_t>(k * 2), bd + static_cast<uint64_t>(k * 128),
                              p.idesc, (kb | k) != 0 ? 1u : 0u);
          ptx::mma_commit_pair(empty(s), 0x3);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (ok) ptx::mma_commit_pair(tfull(buf), 0x3);
      }
      ptx::mma_commit_pair(drain, 0x1);
      wait_bounded(drain, 0, p, err_code(1), false);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------- epilogue (both CTAs)
    const int ew = warp - 4;
    const int r = ew * 32 + lane;
    uint32_t acc_it = 0;
    bool ok = true;
    for (int unit = cluster; ok && unit < p.num_units; unit += nclusters) {
      int tm, tn;
      unit_coords(p, unit, tm, tn);
      const uint32_t buf = acc_it & 1u, aph = (acc_it >> 1) & 1u;
      ++acc_it;
      if (!wait_warp(tfull(buf), aph, p, 2)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + buf * BN;
      epilogue_classical<BN>(p, tbase, tm * (2 * kBM) + static_cast<int>(rank) * kBM, tn, r);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa(tempty(buf), 0));
    }
  }

  ptx::tc_fence_before();
  ptx::cluster_sync();  // no CTA leaves while its peer may still signal it
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc_pair(tmem_base, PC::kTmemCols);
}

template <int BN>
cudaError_t launch_gemm_pair_t(const KernelParams& p, int max_clusters, cudaStream_t stream) {
  auto kern = fgemm_kernel_pair<BN>;
  constexpr int smem = PairCfg<BN>::kSmemBytes;
  static unsigned long long configured = 0;
  static int clusters_fit[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!(configured & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * std::max(max_clusters, 1), 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    clusters_fit[dev & 63] = n > 0 ? n : 1;
    configured |= bit;
  }
  const int clusters = std::min(std::min(max_clusters, clusters_fit[dev & 63]), p.num_units);
  cfg.gridDim = dim3(2 * std::max(clusters, 1), 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace fgemm
