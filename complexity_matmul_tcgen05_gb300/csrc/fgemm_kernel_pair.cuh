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
  static constexpr int kBarBytes = 1024;  // barriers, padded to keep what follows 1024-aligned
  // After the barriers: the epilogue warps' staging areas for TMA stores of
  // C (4 KB each).  The region is at least one B half long: the MMA reads
  // BN/2 columns of B per CTA, and this keeps even a full-width read of the
  // last stage inside this CTA's shared memory.
  static constexpr int kStagingOff = kStages * kStageBytes + kBarBytes;
  static constexpr int kStagingBytes = 4 * 4096;
  static constexpr int kSlackBytes = kBBytes > kStagingBytes ? kBBytes : kStagingBytes;
  static constexpr int kSmemBytes = 1024 + kStagingOff + kSlackBytes;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert(2 * BN <= kTmemCols, "two accumulator buffers must fit in TMEM");
  static_assert((2 * kStages + 6) * 8 + 4 <= kBarBytes, "barrier area too small");
  static_assert(kStageBytes >= 4096, "the last tile's second half stages in the pipeline buffers");
};

// One piece of a K-split tile, for this thread's row r of the CTA's 128 rows:
// store the piece's fp32 partial (layout [col/4][row][4]: a lane moves 16
// bytes of its row, a warp 512 contiguous bytes), then count the arrival on
// the (tile, rank, warp) counter.  A warp that is not the last for its 32
// rows hands the TMEM buffer back at once.  The last one sums the pieces in
// piece order (its own from TMEM, the others from the workspace), applies the
// ordinary epilogue to the sum, then hands the buffer back.  Hands the buffer
// back itself (arrives on `tempty_remote`).
template <int BN>
__device__ __forceinline__ void epilogue_split_piece(const KernelParams& p, uint32_t tbase, int row0,
                                                     int tn, int r, const WorkItem& w,
                                                     uint32_t rank, int ew,
                                                     uint32_t tempty_remote) {
  const int lane = threadIdx.x & 31;
  const int t = w.unit;  // the split region is units [0, split_tiles)
  constexpr size_t kSlot = static_cast<size_t>(kBM) * BN;
  const size_t piece_stride = 2 * kSlot;  // slots are [tile][piece][rank]
  float* tile_ws = p.split_ws + (static_cast<size_t>(t) * p.split_pieces * 2 + rank) * kSlot;
  float4* mine = reinterpret_cast<float4*>(tile_ws + static_cast<size_t>(w.piece) * piece_stride);
  auto release = [&]() {
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive_cluster(tempty_remote);
  };
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    uint32_t ar[32];
    ptx::tmem_ld_32x32b_x32(tbase + c * 32, ar);
    ptx::tmem_wait_ld();
    ptx::tmem_regs_ready(ar);
    float4* dst = mine + static_cast<size_t>(c * 8) * kBM + r;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      __stcg(dst + q * kBM, make_float4(__uint_as_float(ar[4 * q + 0]), __uint_as_float(ar[4 * q + 1]),
                                        __uint_as_float(ar[4 * q + 2]), __uint_as_float(ar[4 * q + 3])));
  }
  __threadfence();
  __syncwarp();
  const bool last = count_arrival(p, p.split_ctr + (static_cast<size_t>(t) * 2 + rank) * 4 + ew, w.npieces);
  if (!last) {
    release();
    return;
  }
  __threadfence();
  const int row = row0 + r;
  const bool row_ok = row < p.M;
  // v = sum over pieces q = 0 .. npieces-1 (in that order) of TMEM column
  // block [col, col + 32) of piece q; this piece's own values come from TMEM.
  auto load_sum = [&](int col, float (&v)[32]) {
    uint32_t ar[32];
    ptx::tmem_ld_32x32b_x32(tbase + col, ar);
    ptx::tmem_wait_ld();
    ptx::tmem_regs_ready(ar);
#pragma unroll 1
    for (int q = 0; q < w.npieces; ++q) {
      float x[32];
      if (q == w.piece) {
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(ar[j]);
      } else {
        const float4* src = reinterpret_cast<const float4*>(tile_ws + static_cast<size_t>(q) * piece_stride) +
                            static_cast<size_t>(col / 4) * kBM + r;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 f = __ldcg(src + i * kBM);
          x[4 * i + 0] = f.x;
          x[4 * i + 1] = f.y;
          x[4 * i + 2] = f.z;
          x[4 * i + 3] = f.w;
        }
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = q == 0 ? x[j] : v[j] + x[j];
    }
  };
  if (p.epi == kEpiSwiglu) {
    constexpr int HALF = BN / 2;
#pragma unroll 1
    for (int c = 0; c < HALF / 32; ++c) {
      const int col0 = tn * HALF + c * 32;
      float g[32], u[32];
      load_sum(c * 32, g);
      load_sum(HALF + c * 32, u);
      finish_swiglu_warp(p, col0, g, u);
      if (row_ok && col0 < p.n_out) store_row32(p, row, col0, g);
    }
  } else {
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
      const int col0 = tn * BN + c * 32;
      float v[32];
      load_sum(c * 32, v);
      float b[32];
      bias32(p, 0, col0, b);
      finish_plain(p, b, v);
      if (row_ok && col0 < p.n_out) store_row32(p, row, col0, v);
    }
  }
  release();
}

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
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + S * PC::kStageBytes + 8 * (2 * S + 6));
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull = [&](uint32_t b) { return bar0 + 8u * (2 * S + b); };
  auto tempty = [&](uint32_t b) { return bar0 + 8u * (2 * S + 2 + b); };
  const uint32_t drain = bar0 + 8u * (2 * S + 4);
  // completes (once per launch, in both CTAs) when every MMA of the pair's
  // last work item is done: what the warps helping with the last tile wait
  // for.  A parity wait on tfull could not serve them: with short K they get
  // there while that barrier is still two phases behind, and a parity wait
  // that far back returns at once.
  const uint32_t lastfull = bar0 + 8u * (2 * S + 5);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;
  const int n_items = work_item_count(p.num_units, p.split_tiles, p.split_pieces, nclusters, cluster);

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
    ptx::mbar_init(lastfull, 1);
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
      WorkItem w;
      for (int n = 0; ok && work_item(p.num_units, p.split_tiles, p.split_pieces, nclusters, p.k_blocks, cluster, n, w);
           ++n) {
        int tm, tn;
        unit_coords(p, w.unit, tm, tn);
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
        for (int kb = w.k0; kb < w.k1; ++kb) {
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
      WorkItem w;
      for (int n = 0; ok && work_item(p.num_units, p.split_tiles, p.split_pieces, nclusters, p.k_blocks, cluster, n, w);
           ++n) {
        const uint32_t buf = acc_it & 1u, aph = (acc_it >> 1) & 1u;
        ++acc_it;
        if (!wait_one(tempty(buf), aph ^ 1u, p, 1)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t dt = tmem_base + buf * BN;
        for (int kb = w.k0; kb < w.k1; ++kb) {
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
                              p.idesc, (kb != w.k0 || k != 0) ? 1u : 0u);
          ptx::mma_commit_pair(empty(s), 0x3);
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (ok) ptx::mma_commit_pair(tfull(buf), 0x3);
      }
      if (ok && n_items > 0) ptx::mma_commit_pair(lastfull, 0x3);
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
    WorkItem w;
    const int last_n = n_items - 1;
    StageOut so{base_ptr + PC::kStagingOff + ew * 4096, base + PC::kStagingOff + ew * 4096, 0};
    for (int n = 0; ok && work_item(p.num_units, p.split_tiles, p.split_pieces, nclusters, p.k_blocks, cluster, n, w);
         ++n) {
      int tm, tn;
      unit_coords(p, w.unit, tm, tn);
      const uint32_t buf = acc_it & 1u, aph = (acc_it >> 1) & 1u;
      ++acc_it;
      if (!wait_warp(tfull(buf), aph, p, 2)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + buf * BN;
      const int row0 = tm * (2 * kBM) + static_cast<int>(rank) * kBM;
      if (w.npieces > 1) {  // arrives on tempty itself, before the pieces' sum
        epilogue_split_piece<BN>(p, tbase, row0, tn, r, w, rank, ew, ptx::mapa(tempty(buf), 0));
        continue;
      }
      if (n == last_n)  // warps 0-3 finish the other half of the columns
        epilogue_classical<BN, 1>(p, tbase, row0, tn, r, &so);
      else
        epilogue_classical<BN>(p, tbase, row0, tn, r, &so);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa(tempty(buf), 0));
    }
    stage_drain();
  }

  // ------------------------------------------- last tile, second half
  // Nothing overlaps the last tile's epilogue, so the producer, MMA and
  // spare warps (one per TMEM lane quarter, like warps 4-7) take half of its
  // columns.  They meet first, so that the spare warps start their bounded
  // wait only once the producer and the MMA issuer are done.
  if (warp < 4) ptx::named_bar_sync(1, 128);
  if (warp < 4 && n_items > 0) {
    WorkItem w;
    work_item(p.num_units, p.split_tiles, p.split_pieces, nclusters, p.k_blocks, cluster, n_items - 1, w);
    if (w.npieces == 1) {
      const uint32_t it = static_cast<uint32_t>(n_items - 1);
      const uint32_t buf = it & 1u;
      if (wait_warp(lastfull, 0, p, 2)) {
        ptx::tc_fence_after();
        int tm, tn;
        unit_coords(p, w.unit, tm, tn);
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + buf * BN;
        const int row0 = tm * (2 * kBM) + static_cast<int>(rank) * kBM;
        // every MMA has read its operands by now: stage in the pipeline buffers
        StageOut so{base_ptr + warp * 4096, base + warp * 4096, 0};
        epilogue_classical<BN, 2>(p, tbase, row0, tn, warp * 32 + lane, &so);
        stage_drain();
      }
    }
  }

  ptx::tc_fence_before();
  ptx::cluster_sync();  // no CTA leaves while its peer may still signal it
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc_pair(tmem_base, PC::kTmemCols);
}

// Launch configuration of the classical pair kernel; on first use per device
// it also sets the shared-memory limit and records how many clusters fit.
template <int BN>
cudaError_t pair_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute (&attr)[1], int& fit,
                        cudaStream_t stream) {
  auto kern = fgemm_kernel_pair<BN>;
  constexpr int smem = PairCfg<BN>::kSmemBytes;
  static unsigned long long configured = 0;
  static int clusters_fit[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  cfg = cudaLaunchConfig_t{};
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
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * std::max(sms / 2, 1), 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    clusters_fit[dev & 63] = std::min(n > 0 ? n : 1, std::max(sms / 2, 1));
    configured |= bit;
  }
  fit = clusters_fit[dev & 63];
  return cudaSuccess;
}

template <int BN>
int gemm_pair_clusters_fit_t() {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  int fit = 0;
  return pair_config<BN>(cfg, attr, fit, nullptr) == cudaSuccess ? fit : 0;
}

template <int BN>
cudaError_t launch_gemm_pair_t(const KernelParams& p, int clusters, cudaStream_t stream) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  int fit = 0;
  cudaError_t e = pair_config<BN>(cfg, attr, fit, stream);
  if (e != cudaSuccess) return e;
  if (clusters < 1 || clusters > fit) return cudaErrorInvalidValue;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  return cudaLaunchKernelEx(&cfg, fgemm_kernel_pair<BN>, p);
}

}  // namespace fgemm
