// fgemm_kern_lcma.cu -- one Strassen-like level (Strassen's or Winograd's
// scheme) on CTA pairs, with the summed operands streamed through HBM
// (FalconGEMM summary, "Methodology" items 1 and 3).
//
// Two launches:
//  1. lcma_form_kernel forms every summed operand of the scheme once from the
//     2 x 2 blocks of A and B (e.g. A11 + A22, B12 - B22): each element is the
//     fp32 sum of the exact 16-bit inputs, rounded once to the input type,
//     written to handle-owned temporaries.  It reads A and B once and writes
//     each temporary once: a streaming, HBM-bound kernel.
//  2. fgemm_kernel_pair_lcma runs the seven block products in one persistent
//     launch on CTA pairs: 256 x BN tiles of the half-size block space, on
//     the classical pair mainloop (TMA -> 128-byte-swizzled shared-memory ring
//     -> tcgen05.mma cta_group::2 -> double-buffered TMEM), so the tensor
//     pipe sees the same operand stream as a classical product.  The work
//     units (output position, product), position-major, are shared out in
//     equal contiguous ranges over the pairs.  The epilogue warps fold each
//     product's accumulator into per-CTA fp32 partial tiles of the output
//     blocks it feeds (C11 = M1 + M4 - M5 + M7, ...) with TMA bulk stores
//     (first contribution) and bulk reduce-adds performed at the L2, so no
//     load latency sits in the fold.  After the last product of a position
//     they apply alpha / bias / activation to every block and store C.  A
//     position whose products fall in two pairs' ranges is finished by the
//     last pair to arrive (a generation-tagged counter), which adds the
//     pairs' partials in pair order: the result does not depend on timing.
//
// Why the sums go through HBM on this chip: the classical 256 x 256 pair
// mainloop already keeps the shared-memory port and the tensor pipe near
// their limits, and forming sums on chip adds operand traffic to the same
// port (the register and TMA-staged on-chip forms of this library measure
// 4-7x slower than the classical kernel).  The pre-pass moves
// (4 + ntemp) blocks of A and of B once through HBM, a few percent of the
// products' time at the large shapes where one level saves 1/8 of the MACs.
#include <algorithm>

#include "fgemm_kernel.cuh"

namespace fgemm {

// ------------------------------------------------------ operand formation

// Block (q >> 1, q & 1) of a 2 x 2 split of a rows x cols sub-block grid.
__device__ __forceinline__ const uint4* form_src(const LcmaFormJob& J, int q, int r) {
  const uint16_t* base = J.src + static_cast<long long>((q >> 1) * J.rows + r) * J.ld +
                         static_cast<long long>(q & 1) * J.cols;
  return reinterpret_cast<const uint4*>(base);
}

// One warp per row and 32 column groups of 8 elements (16 bytes) per warp:
// the four blocks' 16 bytes are loaded once, every temporary's 16 bytes
// formed and stored.  blockIdx.z selects the matrix (A or B).
__global__ void __launch_bounds__(256) lcma_form_kernel(const __grid_constant__ LcmaFormParams P) {
  const LcmaFormJob& J = P.job[blockIdx.z];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cols8 = J.cols >> 3;
  const int c8 = blockIdx.x * 32 + lane;
  if (J.ntemp == 0 || c8 >= cols8) return;
  const long long plane = static_cast<long long>(J.rows) * J.cols;
#pragma unroll 1
  for (int r = blockIdx.y * 8 + warp; r < J.rows; r += gridDim.y * 8) {
    uint4 raw[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      raw[q] = (J.block_mask >> q) & 1u ? __ldg(form_src(J, q, r) + c8) : make_uint4(0, 0, 0, 0);
    uint16_t* dst = J.dst + static_cast<long long>(r) * J.cols + c8 * 8;
#pragma unroll 1
    for (int t = 0; t < J.ntemp; ++t) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int cf = J.coef[t][q];
        if (cf != 0) {
          float f[8];
          unpack8(raw[q], f, P.is_bf16);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] += cf > 0 ? f[i] : -f[i];
        }
      }
      *reinterpret_cast<uint4*>(dst + t * plane) =
          make_uint4(pack2(acc[0], acc[1], P.is_bf16), pack2(acc[2], acc[3], P.is_bf16),
                     pack2(acc[4], acc[5], P.is_bf16), pack2(acc[6], acc[7], P.is_bf16));
    }
  }
}

cudaError_t launch_lcma_form(const LcmaFormParams& f, int num_sms, cudaStream_t stream) {
  int max_cols8 = 0, max_rows = 0;
  for (int j = 0; j < 2; ++j) {
    if (f.job[j].ntemp == 0) continue;
    max_cols8 = std::max(max_cols8, f.job[j].cols / 8);
    max_rows = std::max(max_rows, f.job[j].rows);
  }
  if (max_cols8 == 0) return cudaSuccess;
  const int gx = (max_cols8 + 31) / 32;
  // about 16 blocks of 8 warps per SM over both matrices, each warp looping over rows
  const int gy = std::max(1, std::min((max_rows + 7) / 8, std::max(1, num_sms * 8 / gx)));
  lcma_form_kernel<<<dim3(gx, std::min(gy, 65535), 2), 256, 0, stream>>>(f);
  return cudaGetLastError();
}

// ------------------------------------------------------- product kernel

template <int BN>
struct LcmaCfg {
  static constexpr int kABytes = kBM * kBK * 2;        // this CTA's 128 rows of A
  static constexpr int kBBytes = kBK * (BN / 2) * 2;   // this CTA's BN/2 columns of B
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = BN == 256 ? 6 : 8;
  static constexpr int kTmemCols = BN == 256 ? 512 : 256;
  static constexpr int kBarBytes = 1024;
  // After the barriers: per epilogue warp two 4 KB buffers of 32 rows x 32
  // fp32 values, the sources of the bulk stores / reduce-adds of the fold.
  // The region is longer than a B half, so even a full-width MMA read of the
  // last stage stays inside this CTA's shared memory.
  static constexpr int kStagingOff = kStages * kStageBytes + kBarBytes;
  static constexpr int kStagingBytes = 4 * 2 * 4096;
  static constexpr int kSmemBytes = 1024 + kStagingOff + kStagingBytes;
  static constexpr int kChunks = BN / 32;
  static constexpr int kBlocks = 4;  // output blocks of one level
  static_assert(kStagingBytes >= kBBytes, "slack past the last stage");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert(2 * BN <= kTmemCols, "two accumulator buffers must fit in TMEM");
  static_assert((2 * kStages + 5) * 8 + 4 <= kBarBytes, "barrier area too small");
};

// The contiguous range of units [lo, hi) of pair c (equal shares, +-1).
__device__ __forceinline__ void lcma_range(long long units, int pairs, int c, long long& lo,
                                           long long& hi) {
  lo = static_cast<long long>(c) * units / pairs;
  hi = static_cast<long long>(c + 1) * units / pairs;
}

// Partial slot of output position `pos` on a pair whose units are [lo, hi):
// 0 for its first position, 1 for its last, 2 for the ones between.
__device__ __forceinline__ int lcma_slot(long long lo, long long hi, int np, long long pos) {
  if (pos == lo / np) return 0;
  if (pos == (hi - 1) / np) return 1;
  return 2;
}

__device__ __forceinline__ long long lmax(long long a, long long b) { return a > b ? a : b; }
__device__ __forceinline__ long long lmin(long long a, long long b) { return a < b ? a : b; }

// Output blocks that products [k0, k1) of the scheme feed.
__device__ __forceinline__ uint32_t lcma_block_mask(const LcmaParams& L, int k0, int k1) {
  uint32_t m = 0;
  for (int k = k0; k < k1; ++k)
    for (int t = 0; t < L.prod[k].nc; ++t) m |= 1u << (L.prod[k].c[t] & kTermIndexMask);
  return m;
}

// The 32 x 32 fp32 values warp `ew` of CTA `cta` holds for chunk c of output
// block blk in slot s: 4 KB, row lane at lane * 32.
template <int BN>
__device__ __forceinline__ float* lcma_part(float* ws, int cta, int s, int blk, int c, int ew) {
  using LC = LcmaCfg<BN>;
  const size_t per_cta = static_cast<size_t>(3) * LC::kBlocks * kBM * BN;
  return ws + static_cast<size_t>(cta) * per_cta +
         ((static_cast<size_t>(s) * LC::kBlocks + blk) * LC::kChunks + c) * (kBM * 32) +
         static_cast<size_t>(ew) * 1024;
}

// v[j] (+)= row `lane` of a 32 x 32 partial.
__device__ __forceinline__ void lcma_load_row(const float* part, int lane, float (&v)[32], bool add) {
  const float4* src = reinterpret_cast<const float4*>(part + lane * 32);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 f = __ldcg(src + q);
    if (add) {
      v[4 * q + 0] += f.x; v[4 * q + 1] += f.y; v[4 * q + 2] += f.z; v[4 * q + 3] += f.w;
    } else {
      v[4 * q + 0] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
    }
  }
}

// Finishes output position (tm, tn) for this warp's 32 rows of this CTA:
// for every output block and 32-column chunk, the sum in pair order of the
// partials of pairs [c0, c1] that fed the block, then alpha / bias /
// activation and the store of C.  Every pair's partial lies in its slot for
// this position.
template <int BN>
__device__ void lcma_finish(const LcmaParams& L, int pairs, int c0, int c1, long long pos, int tm,
                            int tn, uint32_t rank, int ew) {
  using LC = LcmaCfg<BN>;
  const KernelParams& p = L.k;
  const int lane = threadIdx.x & 31;
  const int np = p.num_products;
  int slot[8];
  uint32_t mask[8];
  const int ns = c1 - c0 + 1;  // at most 8 pairs share a position (7 products)
  for (int i = 0; i < ns; ++i) {
    long long lo, hi;
    lcma_range(L.units, pairs, c0 + i, lo, hi);
    const long long u0 = pos * np;
    const int k0 = static_cast<int>(lmax(lo, u0) - u0);
    const int k1 = static_cast<int>(lmin(hi, u0 + np) - u0);
    slot[i] = lcma_slot(lo, hi, np, pos);
    mask[i] = lcma_block_mask(L, k0, k1);
  }
  auto gather = [&](int blk, int c, float (&v)[32]) {
    bool any = false;
    for (int i = 0; i < ns; ++i) {
      if (!((mask[i] >> blk) & 1u)) continue;
      const int cta = 2 * (c0 + i) + static_cast<int>(rank);
      lcma_load_row(lcma_part<BN>(p.workspace, cta, slot[i], blk, c, ew), lane, v, any);
      any = true;
    }
    if (!any) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 0.0f;
    }
  };
  const int row_in = tm * (2 * kBM) + static_cast<int>(rank) * kBM + ew * 32 + lane;
  if (p.epi == kEpiSwiglu) {
    // gate = output blocks (r, 0), up = (r, 1): the halves of the N split
#pragma unroll 1
    for (int sr = 0; sr < 2; ++sr) {
#pragma unroll 1
      for (int c = 0; c < LC::kChunks; ++c) {
        float g[32], u[32];
        gather(sr * 2, c, g);
        gather(sr * 2 + 1, c, u);
        const int col0 = tn * BN + c * 32;
        finish_swiglu_warp(p, col0, g, u);
        store_row32(p, sr * p.sub_m + row_in, col0, g);
      }
    }
  } else {
#pragma unroll 1
    for (int blk = 0; blk < LC::kBlocks; ++blk) {
#pragma unroll 1
      for (int c = 0; c < LC::kChunks; ++c) {
        float v[32];
        gather(blk, c, v);
        const int col0 = (blk & 1) * p.sub_n + tn * BN + c * 32;
        float b[32];
        bias32(p, 0, col0, b);
        finish_plain(p, b, v);
        store_row32(p, (blk >> 1) * p.sub_m + row_in, col0, v);
      }
    }
  }
}

template <int BN>
__global__ void __launch_bounds__(256, 1) fgemm_kernel_pair_lcma(const __grid_constant__ LcmaParams L) {
  using LC = LcmaCfg<BN>;
  constexpr int S = LC::kStages;
  const KernelParams& p = L.k;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  const uint32_t sA0 = base;
  const uint32_t sB0 = base + S * LC::kABytes;
  const uint32_t bar0 = base + S * LC::kStageBytes;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + S * LC::kStageBytes + 8 * (2 * S + 5));
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
  const int pairs = gridDim.x >> 1;
  const int np = p.num_products;
  long long lo, hi;
  lcma_range(L.units, pairs, cluster, lo, hi);

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
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), LC::kTmemCols);
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
      ptx::prefetch_tmap(&L.tmap_ta);
      ptx::prefetch_tmap(&L.tmap_tb);
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (long long u = lo; ok && u < hi; ++u) {
        const long long pos = u / np;
        const LcmaProduct& P = L.prod[u - pos * np];
        int tm, tn;
        unit_coords(p, static_cast<int>(pos), tm, tn);
        const CUtensorMap* amap = P.a_temp ? &L.tmap_ta : &p.tmap_a;
        const CUtensorMap* bmap = P.b_temp ? &L.tmap_tb : &p.tmap_b;
        const int ay = (P.a_temp ? P.a_idx : (P.a_idx >> 1)) * p.sub_m + tm * (2 * kBM) +
                       static_cast<int>(rank) * kBM;
        const int ax = P.a_temp ? 0 : (P.a_idx & 1) * p.sub_k;
        const int by = (P.b_temp ? P.b_idx : (P.b_idx >> 1)) * p.sub_k;
        const int bx = (P.b_temp ? 0 : (P.b_idx & 1) * p.sub_n) + tn * BN +
                       static_cast<int>(rank) * (BN / 2);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_one(empty(s), ph ^ 1u, p, 0)) {
            ok = false;
            break;
          }
          const uint32_t fb = ptx::mapa(full(s), 0);
          if (leader) ptx::mbar_arrive_expect_tx(full(s), 2 * LC::kStageBytes);
          ptx::tma_load_2d_pair(sA0 + s * LC::kABytes, amap, ax + kb * kBK, ay, fb);
#pragma unroll
          for (int q = 0; q < BN / 128; ++q)
            ptx::tma_load_2d_pair(sB0 + s * LC::kBBytes + q * 8192, bmap, bx + q * 64, by + kb * kBK, fb);
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
      for (long long u = lo; ok && u < hi; ++u) {
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
          const uint64_t ad = ptx::sdesc(sA0 + s * LC::kABytes, 16, 1024);
          const uint64_t bd = ptx::sdesc(sB0 + s * LC::kBBytes, 8192, 1024);
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
    uint8_t* stg = base_ptr + LC::kStagingOff + ew * 8192;
    const uint32_t stg_addr = base + LC::kStagingOff + ew * 8192;
    uint32_t acc_it = 0, nbulk = 0;
    uint32_t written = 0;  // output blocks of the current position this pair has stored
    bool ok = true;
    for (long long u = lo; ok && u < hi; ++u) {
      const long long pos = u / np;
      const int pr = static_cast<int>(u - pos * np);
      const long long u0 = pos * np;
      const int k_lo = static_cast<int>(lmax(lo, u0) - u0);
      const int k_hi = static_cast<int>(lmin(hi, u0 + np) - u0);
      const int slot = lcma_slot(lo, hi, np, pos);
      const uint32_t buf = acc_it & 1u, aph = (acc_it >> 1) & 1u;
      ++acc_it;
      if (pr == k_lo) written = 0;
      // the previous product's bulk operations have landed before this one
      // adds to the same partials (a fixed order of the fp32 additions)
      if (lane == 0) ptx::bulk_wait<0>();
      __syncwarp();
      if (!wait_warp(tfull(buf), aph, p, 2)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + buf * BN;
      const LcmaProduct& P = L.prod[pr];
      const int nc = P.nc;
      uint32_t first_bits = 0;
      for (int t = 0; t < nc; ++t) {
        const int blk = P.c[t] & kTermIndexMask;
        if (!((written >> blk) & 1u)) first_bits |= 1u << t;
        written |= 1u << blk;
      }
#pragma unroll 1
      for (int c = 0; c < LC::kChunks; ++c) {
        uint32_t ar[32];
        ptx::tmem_ld_32x32b_x32(tbase + c * 32, ar);
        ptx::tmem_wait_ld();
        ptx::tmem_regs_ready(ar);
#pragma unroll 1
        for (int t = 0; t < nc; ++t) {
          const uint32_t sb = nbulk & 1u;
          // the bulk operation that read this buffer two operations ago is done reading
          if (lane == 0) ptx::bulk_wait_read<1>();
          __syncwarp();
          const float sg = (P.c[t] & kTermNeg) ? -1.0f : 1.0f;
          float4* row = reinterpret_cast<float4*>(stg + sb * 4096 + lane * 128);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            row[q] = make_float4(sg * __uint_as_float(ar[4 * q + 0]), sg * __uint_as_float(ar[4 * q + 1]),
                                 sg * __uint_as_float(ar[4 * q + 2]), sg * __uint_as_float(ar[4 * q + 3]));
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            float* dst = lcma_part<BN>(p.workspace, static_cast<int>(blockIdx.x), slot,
                                       P.c[t] & kTermIndexMask, c, ew);
            if ((first_bits >> t) & 1u)
              ptx::bulk_store(dst, stg_addr + sb * 4096, 4096);
            else
              ptx::bulk_reduce_add_f32(dst, stg_addr + sb * 4096, 4096);
            ptx::bulk_commit();
          }
          ++nbulk;
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa(tempty(buf), 0));
      if (pr != k_hi - 1) continue;
      // the pair's last product of this position: its partials are complete
      if (lane == 0) ptx::bulk_wait<0>();
      __syncwarp();
      ptx::fence_proxy_async_global();
      int tm, tn;
      unit_coords(p, static_cast<int>(pos), tm, tn);
      if (k_lo == 0 && k_hi == np) {
        lcma_finish<BN>(L, pairs, cluster, cluster, pos, tm, tn, rank, ew);
        continue;
      }
      const int c0 = stream_k_owner(u0, L.units, pairs);
      const int c1 = stream_k_owner(u0 + np - 1, L.units, pairs);
      __threadfence();
      __syncwarp();
      const bool last = count_arrival(p, p.split_ctr + (static_cast<size_t>(pos) * 2 + rank) * 4 + ew,
                                      c1 - c0 + 1);
      if (!last) continue;
      __threadfence();
      ptx::fence_proxy_async_global();
      lcma_finish<BN>(L, pairs, c0, c1, pos, tm, tn, rank, ew);
    }
    if (lane == 0) ptx::bulk_wait<0>();
    __syncwarp();
  }

  ptx::tc_fence_before();
  ptx::cluster_sync();  // no CTA leaves while its peer may still signal it
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc_pair(tmem_base, LC::kTmemCols);
}

template <int BN>
cudaError_t lcma_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute (&attr)[1], int& fit,
                        cudaStream_t stream) {
  auto kern = fgemm_kernel_pair_lcma<BN>;
  constexpr int smem = LcmaCfg<BN>::kSmemBytes;
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

int lcma_pair_clusters_fit(int bn) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  int fit = 0;
  cudaError_t e = bn == 256   ? lcma_config<256>(cfg, attr, fit, nullptr)
                  : bn == 128 ? lcma_config<128>(cfg, attr, fit, nullptr)
                              : cudaErrorInvalidValue;
  return e == cudaSuccess ? fit : 0;
}

template <int BN>
cudaError_t launch_lcma_pair_t(const LcmaParams& L, int clusters, cudaStream_t stream) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  int fit = 0;
  cudaError_t e = lcma_config<BN>(cfg, attr, fit, stream);
  if (e != cudaSuccess) return e;
  if (clusters < 1 || clusters > fit || static_cast<long long>(clusters) > L.units)
    return cudaErrorInvalidValue;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  return cudaLaunchKernelEx(&cfg, fgemm_kernel_pair_lcma<BN>, L);
}

cudaError_t launch_lcma_pair(int bn, const LcmaParams& L, int clusters, cudaStream_t stream) {
  switch (bn) {
    case 128: return launch_lcma_pair_t<128>(L, clusters, stream);
    case 256: return launch_lcma_pair_t<256>(L, clusters, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fgemm
