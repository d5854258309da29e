// fgemm_kern_skinny.cu -- small-M classical GEMM (M <= 64), bound by
// streaming B from HBM.
//
// With M this small, a 128-row tensor-core tile of C is mostly padding, and
// the shared memory it takes is better spent keeping more of B in flight.
// This kernel computes C^T = B^T A^T instead: the MMA's 128 rows run over
// 128 columns of C (B^T, read MN-major straight from row-major B) and its
// N = mp columns over the M rows of C (A^T, read K-major from row-major A,
// rows past M zero-filled by the copy engine).  A stage is 16 KB of B plus
// mp x 128 bytes of A, so 8 to 11 stages of B are in flight per SM.
//
// The K blocks of all column tiles are shared out evenly over the CTAs
// (stream_k_item): no SM idles in a partial last wave.  Each piece of a tile
// that several CTAs share stores its fp32 partial (128 x mp, small at these
// sizes); the last piece to finish sums the pieces in piece order and applies
// the epilogue.  Epilogues: none, scale + bias, SiLU (bias indexed by column).
//
// Warp roles as in the other kernels: warp 0 TMA producer, warp 1 MMA issuer,
// warps 4..7 epilogue (TMEM lanes = the tile's 128 columns).  Every mbarrier
// wait is bounded.
#include <algorithm>

#include "fgemm_kernel.cuh"

namespace fgemm {

template <int MP>
struct SkinnyCfg {
  static constexpr int kBtBytes = 128 * kBK * 2;  // B^T tile: 128 columns x 64 K, two 64-column boxes
  static constexpr int kAtBytes = MP * kBK * 2;   // A^T tile: MP rows x 64 K
  static constexpr int kStageBytes = kBtBytes + kAtBytes;
  static constexpr int kStages = (200 * 1024) / kStageBytes < 12 ? (200 * 1024) / kStageBytes : 12;
  static constexpr int kTmemCols = 2 * MP < 32 ? 32 : 2 * MP;  // two accumulators of MP columns
  static constexpr int kBarBytes = 256;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kBarBytes;
  static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert((2 * kStages + 5) * 8 + 4 <= kBarBytes, "barrier area too small");
};

// Slot of piece q of this work item's tile (see stream_k_slot).
__device__ __forceinline__ size_t skinny_slot(const KernelParams& p, const WorkItem& w, int q) {
  return static_cast<size_t>(stream_k_slot(p.num_units, p.k_blocks, gridDim.x, w.unit,
                                           static_cast<int>(blockIdx.x) - w.piece + q));
}

// The epilogue of one piece for this thread's column n = n0 + r: acc[m] holds
// C^T[n][m], m < MP.  A tile with one piece is finished at once; otherwise the
// piece's partial is stored and the last piece of the tile finishes it.  The
// tile's arrival counters sit with the slot of its piece 0 (4 per slot, one
// per epilogue warp).
template <int MP>
__device__ __forceinline__ void skinny_finish(const KernelParams& p, int n0, int r, const WorkItem& w,
                                              int ew, float (&acc)[MP]) {
  if (w.npieces > 1) {
    constexpr size_t kSlot = static_cast<size_t>(128) * MP;
    float4* mine = reinterpret_cast<float4*>(p.split_ws + skinny_slot(p, w, w.piece) * kSlot) + r;
#pragma unroll
    for (int q = 0; q < MP / 4; ++q)
      __stcg(mine + q * 128, make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]));
    __threadfence();
    __syncwarp();
    const bool last = count_arrival(p, p.split_ctr + skinny_slot(p, w, 0) * 4 + ew, w.npieces);
    if (!last) return;
    __threadfence();
    // sum the pieces in piece order (this piece's own values from registers);
    // the loads of kBatch pieces are in flight together
    constexpr int kBatch = MP == 16 ? 4 : (MP == 32 ? 2 : 1);
    float sum[MP];
#pragma unroll 1
    for (int q0 = 0; q0 < w.npieces; q0 += kBatch) {
      float x[kBatch][MP];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int q = q0 + b;
        if (q >= w.npieces) continue;
        if (q == w.piece) {
#pragma unroll
          for (int m = 0; m < MP; ++m) x[b][m] = acc[m];
        } else {
          const float4* src =
              reinterpret_cast<const float4*>(p.split_ws + skinny_slot(p, w, q) * kSlot) + r;
#pragma unroll
          for (int i = 0; i < MP / 4; ++i) {
            const float4 f = __ldcg(src + i * 128);
            x[b][4 * i] = f.x;
            x[b][4 * i + 1] = f.y;
            x[b][4 * i + 2] = f.z;
            x[b][4 * i + 3] = f.w;
          }
        }
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int q = q0 + b;
        if (q >= w.npieces) continue;
#pragma unroll
        for (int m = 0; m < MP; ++m) sum[m] = q == 0 ? x[b][m] : sum[m] + x[b][m];
      }
    }
#pragma unroll
    for (int m = 0; m < MP; ++m) acc[m] = sum[m];
  }
  const int n = n0 + r;
  if (n >= p.n_out) return;
  const float b = p.bias ? ld_bias(p, n) : 0.0f;
  uint16_t* dst = p.C + n;
#pragma unroll
  for (int m = 0; m < MP; ++m) {
    if (m < p.M) {
      float v = p.alpha * acc[m] + b;
      if (p.epi == kEpiSilu) v = silu(v);
      dst[static_cast<long long>(m) * p.ldc] = pack1(v, p.is_bf16);
    }
  }
}

template <int MP>
__global__ void __launch_bounds__(256, 1) fgemm_kernel_skinny(const __grid_constant__ KernelParams p) {
  using SC = SkinnyCfg<MP>;
  constexpr int S = SC::kStages;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  auto sBt = [&](int s) { return base + s * SC::kStageBytes; };
  auto sAt = [&](int s) { return base + s * SC::kStageBytes + SC::kBtBytes; };
  const uint32_t bar0 = base + S * SC::kStageBytes;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + S * SC::kStageBytes + 8 * (2 * S + 5));
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull = [&](uint32_t b) { return bar0 + 8u * (2 * S + b); };
  auto tempty = [&](uint32_t b) { return bar0 + 8u * (2 * S + 2 + b); };
  const uint32_t drain = bar0 + 8u * (2 * S + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int tiles = p.num_units;
  const int ctas = gridDim.x;
  const int cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(full(s), 1);
      ptx::mbar_init(empty(s), 1);
    }
    for (uint32_t b = 0; b < 2; ++b) {
      ptx::mbar_init(tfull(b), 1);
      ptx::mbar_init(tempty(b), 4);
    }
    ptx::mbar_init(drain, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), SC::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::prefetch_tmap(&p.tmap_a);
      ptx::prefetch_tmap(&p.tmap_b);
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      WorkItem w;
      for (int n = 0; ok && stream_k_item(tiles, p.k_blocks, ctas, cta, n, w); ++n) {
        const int n0 = w.unit * 128;
        for (int kb = w.k0; kb < w.k1; ++kb) {
          if (!wait_one(empty(s), ph ^ 1u, p, 0)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(full(s), SC::kStageBytes);
          ptx::tma_load_2d(sBt(s), &p.tmap_b, n0, kb * kBK, full(s));
          ptx::tma_load_2d(sBt(s) + 8192, &p.tmap_b, n0 + 64, kb * kBK, full(s));
          ptx::tma_load_2d(sAt(s), &p.tmap_a, kb * kBK, 0, full(s));
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
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
    // ------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0, acc_it = 0;
      bool ok = true;
      WorkItem w;
      for (int n = 0; ok && stream_k_item(tiles, p.k_blocks, ctas, cta, n, w); ++n) {
        const uint32_t buf = acc_it & 1u, aph = (acc_it >> 1) & 1u;
        ++acc_it;
        if (!wait_one(tempty(buf), aph ^ 1u, p, 1)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t dt = tmem_base + buf * MP;
        for (int kb = w.k0; kb < w.k1; ++kb) {
          if (!wait_one(full(s), ph, p, 1)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          // A operand: B^T, MN-major (64-column boxes 8 KB apart, 8-K-row groups 1 KB apart);
          // B operand: A^T, K-major (128-byte rows, 8-row groups 1 KB apart)
          const uint64_t ad = ptx::sdesc(sBt(s), 8192, 1024);
          const uint64_t bd = ptx::sdesc(sAt(s), 16, 1024);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            ptx::mma_f16(dt, ad + static_cast<uint64_t>(k * 128), bd + static_cast<uint64_t>(k * 2),
                         p.idesc, (kb != w.k0 || k != 0) ? 1u : 0u);
          ptx::mma_commit(empty(s));
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (ok) ptx::mma_commit(tfull(buf));
      }
      ptx::mma_commit(drain);
      wait_bounded(drain, 0, p, err_code(1), false);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------- epilogue
    const int ew = warp - 4;
    const int r = ew * 32 + lane;
    uint32_t acc_it = 0;
    WorkItem w;
    for (int n = 0; stream_k_item(tiles, p.k_blocks, ctas, cta, n, w); ++n) {
      const uint32_t buf = acc_it & 1u, aph = (acc_it >> 1) & 1u;
      ++acc_it;
      if (!wait_warp(tfull(buf), aph, p, 2)) break;
      ptx::tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + buf * MP;
      float acc[MP];
#pragma unroll
      for (int g = 0; g < MP / 16; ++g) {
        uint32_t a16[16];
        ptx::tmem_ld_32x32b_x16(tbase + g * 16, a16);
        ptx::tmem_wait_ld();
        ptx::tmem_regs_ready16(a16);
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[g * 16 + j] = __uint_as_float(a16[j]);
      }
      // the accumulator is in registers: hand the TMEM buffer back first
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(tempty(buf));
      skinny_finish<MP>(p, w.unit * 128, r, w, ew, acc);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem_base, SC::kTmemCols);
}

template <int MP>
cudaError_t launch_skinny_t(const KernelParams& p, int grid, cudaStream_t stream) {
  auto kern = fgemm_kernel_skinny<MP>;
  constexpr int smem = SkinnyCfg<MP>::kSmemBytes;
  static unsigned long long configured = 0;  // per-device bit
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(configured & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured |= bit;
  }
  kern<<<grid, 256, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_gemm_skinny(int mp, const KernelParams& p, int grid, cudaStream_t stream) {
  switch (mp) {
    case 16: return launch_skinny_t<16>(p, grid, stream);
    case 32: return launch_skinny_t<32>(p, grid, stream);
    case 64: return launch_skinny_t<64>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fgemm
