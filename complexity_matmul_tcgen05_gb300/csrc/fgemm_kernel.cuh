// fgemm_kernel.cuh -- persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
// One kernel template covers both forms of the product:
//   DEPTH == 0  classical: C tile = A row block x B column block.
//   DEPTH >= 1  Strassen-like (FalconGEMM summary, "Methodology" items 1 and
//               3): each output-tile position of the (M, N) >> DEPTH block
//               space runs the 7^DEPTH block products one after another; the
//               operand sums (e.g. A11 + A22, B12 - B22) are formed on chip
//               by dedicated warps straight into the shared-memory operand
//               buffers, and every product's accumulator is folded into the
//               output blocks it contributes to by the epilogue (per-CTA fp32
//               partial tiles), which also applies the final scale / bias /
//               activation once the last product is in.
//
// Warp roles (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer: raw operand tiles -> shared-memory ring
//   warp 1      MMA issuer (one thread): tcgen05.mma into TMEM; owns TMEM
//   warps 2,3   (Strassen) operand-sum warps, with warps 8..15
//   warps 4..7  epilogue: tcgen05.ld -> fp32 math -> rounded stores
// The TMEM accumulator is double-buffered, so the epilogue of one tile (or
// product) runs while the MMAs of the next are in flight (the overlap the
// PingPong GEMM note describes, done here with TMEM buffers instead of two
// consumer warpgroups).
//
// Every mbarrier wait is bounded (globaltimer); on expiry the kernel latches
// an error code in p.err and every role leaves its loop, so the CTA still
// reaches its teardown and frees its TMEM.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fgemm_internal.h"
#include "fgemm_ptx.cuh"

namespace fgemm {

template <int BN>
struct TileCfg {
  static constexpr int kABytes = kBM * kBK * 2;  // 16 KB: 128 rows x 128 bytes
  static constexpr int kBBytes = kBK * BN * 2;   // BN/64 boxes of 64 K-rows x 128 bytes
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = BN == 256 ? 4 : (BN == 128 ? 6 : 8);
  static constexpr int kTmemCols = BN == 256 ? 512 : (BN == 128 ? 256 : 128);
  static constexpr int kBarBytes = 256;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kBarBytes;
  static_assert(2 * BN <= kTmemCols, "two accumulator buffers must fit in TMEM");
  static_assert((2 * kStages + 5) * 8 + 4 <= kBarBytes, "barrier area too small");
};

template <int DEPTH>
struct RoleCfg {
  // Strassen: warps 2, 3 and 8..15 form operand sums (10 warps).
  static constexpr int kSumWarps = DEPTH == 0 ? 0 : 10;
  static constexpr int kThreads = DEPTH == 0 ? 256 : 512;
};

// ------------------------------------------------------------ small helpers

__device__ __forceinline__ uint32_t err_code(int role) {
  return kErrTimeout | (static_cast<uint32_t>(role) << 24) | (blockIdx.x & 0xFFFFFFu);
}

// Bounded wait on one mbarrier phase by the calling thread.  Gives up when
// the kernel's error word is set by another role (honor_err) or when
// p.spin_ns elapses (then latches `code`).
static __device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const KernelParams& p,
                                          uint32_t code, bool honor_err) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
#pragma unroll 1
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (ptx::mbar_try_wait(bar, parity)) return true;
    if (honor_err && *reinterpret_cast<volatile unsigned int*>(p.err) != 0u) return false;
    if (ptx::globaltimer() - t0 > p.spin_ns) {
      atomicCAS(p.err, 0u, code);
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_one(uint32_t bar, uint32_t parity, const KernelParams& p,
                                         int role) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  return wait_bounded(bar, parity, p, err_code(role), true);
}

// Whole-warp wait; the outcome is made warp-uniform.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const KernelParams& p,
                                          int role) {
  bool ok = wait_one(bar, parity, p, role);
  return __all_sync(0xFFFFFFFFu, ok);
}

// Counts one arrival of a split piece on `ctr` (by lane 0 of the calling
// warp) and tells the whole warp whether it was the last of `npieces`.  The
// counter holds gen << 8 | arrivals.  A counter tagged with another
// generation (left by a launch that ended on an error) counts as zero
// arrivals, and the last arrival resets the counter to zero arrivals of this
// generation, so a replay of the same launch (a CUDA graph) counts from zero
// again.  Warp-collective.
__device__ __forceinline__ bool count_arrival(const KernelParams& p, unsigned int* ctr, int npieces) {
  const int lane = threadIdx.x & 31;
  unsigned int count = 0;
  if (lane == 0) {
    const unsigned int gen = p.split_gen;
    unsigned int cur = *reinterpret_cast<volatile unsigned int*>(ctr);
#pragma unroll 1
    for (int it = 0; it < (1 << 20); ++it) {
      const unsigned int next = (cur >> 8) == gen ? cur + 1u : ((gen << 8) | 1u);
      const unsigned int prev = atomicCAS(ctr, cur, next);
      if (prev == cur) {
        count = next & 0xFFu;
        break;
      }
      cur = prev;
    }
    if (count == 0)
      atomicCAS(p.err, 0u, err_code(2));
    else if (count == static_cast<unsigned int>(npieces))
      atomicExch(ctr, gen << 8);
  }
  count = __shfl_sync(0xFFFFFFFFu, count, 0);
  return count == static_cast<unsigned int>(npieces);
}

__device__ __forceinline__ void unit_coords(const KernelParams& p, int unit, int& tm, int& tn) {
  const int G = p.raster_group;
  const int per_group = G * p.tiles_n;
  const int g = unit / per_group;
  const int first_m = g * G;
  const int gsz = min(p.tiles_m - first_m, G);
  const int r = unit - g * per_group;
  tm = first_m + r % gsz;
  tn = r / gsz;
}

__device__ __forceinline__ float h2f(uint32_t h, int is_bf16) {
  return is_bf16 ? __uint_as_float(h << 16) : __half2float(__ushort_as_half((unsigned short)h));
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, int is_bf16) {
  if (is_bf16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint16_t pack1(float v, int is_bf16) {
  return is_bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(v))
                 : __half_as_ushort(__float2half_rn(v));
}

__device__ __forceinline__ float silu(float v) { return v / (1.0f + __expf(-v)); }

// The value a float becomes when stored in the output type.
__device__ __forceinline__ float round_out(float v, int is_bf16) {
  return h2f(pack1(v, is_bf16), is_bf16);
}

// RMSNorm row scale from an earlier product's block sums of squares:
// 1 / sqrt(sum_p sumsq_in[p][row] / n + eps), summed in block order.
__device__ __forceinline__ float rms_row_scale(const KernelParams& p, int row) {
  float ss = 0.0f;
#pragma unroll 4
  for (int q = 0; q < p.sumsq_parts; ++q) ss += __ldg(p.sumsq_in + static_cast<size_t>(q) * p.M + row);
  return 1.0f / sqrtf(ss * p.rms_inv_n + p.rms_eps);
}

__device__ __forceinline__ float ld_bias(const KernelParams& p, int col) {
  return h2f(__ldg(p.bias + col), p.is_bf16);
}

// Writes 32 consecutive outputs of one row, clipping at n_out.
__device__ __forceinline__ void store_row32(const KernelParams& p, int row, int col0,
                                            const float (&v)[32]) {
  uint16_t* dst = p.C + static_cast<long long>(row) * p.ldc + col0;
  const int n = p.n_out - col0;
  if (n >= 32) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      d4[q] = make_uint4(pack2(v[8 * q + 0], v[8 * q + 1], p.is_bf16),
                         pack2(v[8 * q + 2], v[8 * q + 3], p.is_bf16),
                         pack2(v[8 * q + 4], v[8 * q + 5], p.is_bf16),
                         pack2(v[8 * q + 6], v[8 * q + 7], p.is_bf16));
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < n) dst[j] = pack1(v[j], p.is_bf16);
  }
}

// A warp's staging area for TMA stores of C: two 2 KB buffers of 32 rows x
// 32 columns (64-byte rows, 16-byte chunk j of row t at chunk j ^ ((t >> 1) & 3),
// the 64-byte swizzle of p.tmap_c), used in turn.
struct StageOut {
  uint8_t* ptr;   // generic address of the first buffer
  uint32_t addr;  // shared-space address of the first buffer (1024-aligned)
  uint32_t it;    // buffers filled so far
};

// Stores the warp's 32 rows x 32 columns (row wrow0 + lane holds v) through
// the staging area: wait until the buffer's previous store has read it,
// write this lane's row, then lane 0 issues the TMA store.  The tensor map
// clips rows >= M and columns >= n_out.  Warp-collective.
__device__ __forceinline__ void stage_store32(const KernelParams& p, StageOut& so, int wrow0, int col0,
                                              const float (&v)[32]) {
  const int lane = threadIdx.x & 31;
  const uint32_t off = (so.it & 1u) * 2048u;
  if (lane == 0) ptx::bulk_wait_read<1>();
  __syncwarp();
  uint8_t* row = so.ptr + off + lane * 64;
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<uint4*>(row + ((q ^ sw) << 4)) =
        make_uint4(pack2(v[8 * q + 0], v[8 * q + 1], p.is_bf16), pack2(v[8 * q + 2], v[8 * q + 3], p.is_bf16),
                   pack2(v[8 * q + 4], v[8 * q + 5], p.is_bf16), pack2(v[8 * q + 6], v[8 * q + 7], p.is_bf16));
  ptx::fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    ptx::tma_store_2d(&p.tmap_c, so.addr + off, col0, wrow0);
    ptx::bulk_commit();
  }
  ++so.it;
}

// Waits until every TMA store of the staging area has completed.
__device__ __forceinline__ void stage_drain() {
  if ((threadIdx.x & 31) == 0) ptx::bulk_wait<0>();
  __syncwarp();
}

// b[j] = bias[base + min(col0 + j, n_out - 1)] (0 without a bias), for every
// lane of the warp: each lane loads one entry and the warp exchanges them by
// shuffles.  Warp-collective: call it outside row-dependent branches.
__device__ __forceinline__ void bias32(const KernelParams& p, int base, int col0, float (&b)[32]) {
  if (!p.bias) {
#pragma unroll
    for (int j = 0; j < 32; ++j) b[j] = 0.0f;
    return;
  }
  const int lane = threadIdx.x & 31;
  const float mine = ld_bias(p, base + min(col0 + lane, p.n_out - 1));
#pragma unroll
  for (int j = 0; j < 32; ++j) b[j] = __shfl_sync(0xFFFFFFFFu, mine, j);
}

// v[j] = act(alpha * x[j] + b[j]) for the non-gated epilogues.
__device__ __forceinline__ void finish_plain(const KernelParams& p, const float (&b)[32],
                                             float (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    float x = p.alpha * v[j] + b[j];
    if (p.epi == kEpiSilu) x = silu(x);
    v[j] = x;
  }
}

// g[j] = silu(alpha * g + bg[j]) * (alpha * u + bu[j]).
__device__ __forceinline__ void finish_swiglu(const KernelParams& p, const float (&bg)[32],
                                              const float (&bu)[32], float (&g)[32],
                                              const float (&u)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) g[j] = silu(p.alpha * g[j] + bg[j]) * (p.alpha * u[j] + bu[j]);
}

// finish_swiglu with one bias array live at a time (for the 128-register
// Strassen kernels).  Warp-collective like bias32.
__device__ __forceinline__ void finish_swiglu_warp(const KernelParams& p, int col0, float (&g)[32],
                                                   const float (&u)[32]) {
  float b[32];
  bias32(p, 0, col0, b);
#pragma unroll
  for (int j = 0; j < 32; ++j) g[j] = silu(p.alpha * g[j] + b[j]);
  bias32(p, p.n_out, col0, b);
#pragma unroll
  for (int j = 0; j < 32; ++j) g[j] *= p.alpha * u[j] + b[j];
}

// ------------------------------------------------------------ epilogues

// Classical tile: the accumulator in TMEM columns [tbase, tbase + BN).  For
// SwiGLU the tile's first BN/2 columns hold gate columns and the last BN/2
// the matching up columns (the producer loads them side by side).  Every
// bias entry the tile needs is loaded up front (one per lane per 32-column
// chunk, kept as raw 16-bit values and converted when used, so no wait on
// them precedes the first TMEM load; broadcast by shuffles), and for the
// plain epilogues the TMEM load of the next chunk is in flight while the
// current one is finished and stored.  RMSNorm statistics (CODA section of
// the PingPong GEMM / CODA note): with p.sumsq_in the accumulator row is first
// scaled by 1 / sqrt(mean of squares + eps) of an earlier product's row; with
// p.sumsq_out the sums of squares of the stored values of each 64-column
// block are written out, in column order within the block.  RMS selects the
// variant with those statistics at compile time, so the plain epilogue pays
// nothing for them.
// PART selects the 32-column chunks this warp finishes: 0 all of them, 1 the
// first half, 2 the second half (two warps sharing one tile's rows).  With a
// staging area (so != nullptr) C goes out by TMA stores, else by each lane
// storing its row.
template <int BN, bool RMS, int PART>
__device__ __forceinline__ void epilogue_classical_t(const KernelParams& p, uint32_t tbase, int row0,
                                                     int tn, int r, StageOut* so) {
  const int lane = threadIdx.x & 31;
  const int row = row0 + r;
  const bool row_ok = row < p.M;
  const int wrow0 = row - lane;
  auto emit = [&](int col0, const float (&v)[32]) {
    if (so) {
      if (wrow0 < p.M && col0 < p.n_out) stage_store32(p, *so, wrow0, col0, v);
    } else if (row_ok && col0 < p.n_out) {
      store_row32(p, row, col0, v);
    }
  };
  // RMSNorm: the scale of this row (1 without statistics in), and the
  // running sum of squares of the stored outputs of one 64-column block
  const float rs = (RMS && p.sumsq_in && row_ok) ? rms_row_scale(p, row) : 1.0f;
  float ss = 0.0f;
  auto add_sumsq = [&](int c, int col0, const float (&v)[32]) {
    if constexpr (RMS) {
      if (!p.sumsq_out) return;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float q = round_out(v[j], p.is_bf16);
        if (col0 + j < p.n_out) ss += q * q;
      }
      if ((c & 1) && row_ok && col0 - 32 < p.n_out) {  // end of the block [col0 - 32, col0 + 32)
        p.sumsq_out[static_cast<size_t>((col0 - 32) >> 6) * p.M + row] = ss;
        ss = 0.0f;
      }
    }
  };
  if (p.epi == kEpiSwiglu) {
    constexpr int HALF = BN / 2;
    constexpr int CH = HALF / 32;
    constexpr int CB = PART == 2 ? CH / 2 : 0, CE = PART == 1 ? CH / 2 : CH;
    float bg[CH], bu[CH];
#pragma unroll
    for (int c = CB; c < CE; ++c) {
      const int col = min(tn * HALF + c * 32 + lane, p.n_out - 1);
      bg[c] = p.bias ? ld_bias(p, col) : 0.0f;
      bu[c] = p.bias ? ld_bias(p, p.n_out + col) : 0.0f;
    }
#pragma unroll
    for (int c = CB; c < CE; ++c) {
      uint32_t gr[32], ur[32];
      ptx::tmem_ld_32x32b_x32(tbase + c * 32, gr);
      ptx::tmem_ld_32x32b_x32(tbase + HALF + c * 32, ur);
      ptx::tmem_wait_ld();
      ptx::tmem_regs_ready(gr);
      ptx::tmem_regs_ready(ur);
      const int col0 = tn * HALF + c * 32;
      float g[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float ga = RMS ? rs * __uint_as_float(gr[j]) : __uint_as_float(gr[j]);
        const float ua = RMS ? rs * __uint_as_float(ur[j]) : __uint_as_float(ur[j]);
        const float gv = p.alpha * ga + __shfl_sync(0xFFFFFFFFu, bg[c], j);
        const float uv = p.alpha * ua + __shfl_sync(0xFFFFFFFFu, bu[c], j);
        g[j] = silu(gv) * uv;
      }
      emit(col0, g);
      add_sumsq(c, col0, g);
    }
  } else {
    constexpr int CH = BN / 32;
    constexpr int CB = PART == 2 ? CH / 2 : 0, CE = PART == 1 ? CH / 2 : CH;
    uint32_t bl[CH];  // raw 16-bit bias values, converted when used
#pragma unroll
    for (int c = CB; c < CE; ++c)
      bl[c] = p.bias ? __ldg(p.bias + min(tn * BN + c * 32 + lane, p.n_out - 1)) : 0u;
    auto finish = [&](int c, const uint32_t (&ar)[32]) {
      const int col0 = tn * BN + c * 32;
      const float bf = h2f(bl[c], p.is_bf16);
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float a = RMS ? rs * __uint_as_float(ar[j]) : __uint_as_float(ar[j]);
        float x = p.alpha * a + __shfl_sync(0xFFFFFFFFu, bf, j);
        if (p.epi == kEpiSilu) x = silu(x);
        v[j] = x;
      }
      emit(col0, v);
      add_sumsq(c, col0, v);
    };
    uint32_t ra[32], rb[32];
    ptx::tmem_ld_32x32b_x32(tbase + CB * 32, ra);
    ptx::tmem_wait_ld();
    ptx::tmem_regs_ready(ra);
#pragma unroll
    for (int c = CB; c < CE; c += 2) {  // CB and CE are even for every tile width
      ptx::tmem_ld_32x32b_x32(tbase + (c + 1) * 32, rb);
      finish(c, ra);
      ptx::tmem_wait_ld();
      ptx::tmem_regs_ready(rb);
      if (c + 2 < CE) ptx::tmem_ld_32x32b_x32(tbase + (c + 2) * 32, ra);
      finish(c + 1, rb);
      if (c + 2 < CE) {
        ptx::tmem_wait_ld();
        ptx::tmem_regs_ready(ra);
      }
    }
  }
}

template <int BN, int PART = 0>
__device__ __forceinline__ void epilogue_classical(const KernelParams& p, uint32_t tbase, int row0,
                                                   int tn, int r, StageOut* so = nullptr) {
  if (p.sumsq_in || p.sumsq_out)
    epilogue_classical_t<BN, true, PART>(p, tbase, row0, tn, r, so);
  else
    epilogue_classical_t<BN, false, PART>(p, tbase, row0, tn, r, so);
}

// Strassen product `pr` for the 128 rows starting at row0 (inside each
// output block) of column tile tn: fold +-acc into the per-CTA fp32
// partial tiles of the output blocks it feeds; after the last product, apply
// the epilogue to every block and store C.  Workspace layout per CTA:
// [block][32-column chunk][128 rows][32 floats], so a warp's 32 rows of one
// chunk are 4 KB contiguous.  Every element is read and written only by the
// thread that owns its row, in program order.
template <int BN, int DEPTH>
__device__ __forceinline__ void epilogue_strassen(const KernelParams& p, const StrassenTable& tab,
                                                  uint32_t tbase, int row0,
                                                  int tn, int pr, int r, float* ws) {
  constexpr int G = 1 << DEPTH;
  constexpr int CH = BN / 32;
  const int nc = tab.nc[pr];
  const bool last = pr == p.num_products - 1;
  auto slot_ptr = [&](int slot, int c) {
    return reinterpret_cast<float4*>(ws + ((static_cast<size_t>(slot) * CH + c) * kBM + r) * 32);
  };
#pragma unroll 1
  for (int c = 0; c < CH; ++c) {
    uint32_t ar[32];
    ptx::tmem_ld_32x32b_x32(tbase + c * 32, ar);
    ptx::tmem_wait_ld();
#pragma unroll 1
    for (int t = 0; t < nc; ++t) {
      const uint8_t code = tab.c[pr][t];
      float4* w = slot_ptr(code & kTermIndexMask, c);
      const float sg = (code & kTermNeg) ? -1.0f : 1.0f;
      if (code & kTermFirst) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          w[q] = make_float4(sg * __uint_as_float(ar[4 * q + 0]), sg * __uint_as_float(ar[4 * q + 1]),
                             sg * __uint_as_float(ar[4 * q + 2]), sg * __uint_as_float(ar[4 * q + 3]));
      } else {
        float4 x[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) x[q] = w[q];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          x[q].x += sg * __uint_as_float(ar[4 * q + 0]);
          x[q].y += sg * __uint_as_float(ar[4 * q + 1]);
          x[q].z += sg * __uint_as_float(ar[4 * q + 2]);
          x[q].w += sg * __uint_as_float(ar[4 * q + 3]);
          w[q] = x[q];
        }
      }
    }
    if (!last) continue;
    if (p.epi == kEpiSwiglu) {
#pragma unroll 1
      for (int sr = 0; sr < G; ++sr) {
#pragma unroll 1
        for (int sc = 0; sc < G / 2; ++sc) {
          const float4* wg = slot_ptr(sr * G + sc, c);
          const float4* wu = slot_ptr(sr * G + sc + G / 2, c);
          float g[32], u[32];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 a = wg[q], b = wu[q];
            g[4 * q + 0] = a.x; g[4 * q + 1] = a.y; g[4 * q + 2] = a.z; g[4 * q + 3] = a.w;
            u[4 * q + 0] = b.x; u[4 * q + 1] = b.y; u[4 * q + 2] = b.z; u[4 * q + 3] = b.w;
          }
          const int row = sr * p.sub_m + row0 + r;
          const int col0 = sc * p.sub_n + tn * BN + c * 32;
          finish_swiglu_warp(p, col0, g, u);
          store_row32(p, row, col0, g);
        }
      }
    } else {
#pragma unroll 1
      for (int s = 0; s < G * G; ++s) {
        const float4* w = slot_ptr(s, c);
        float v[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 a = w[q];
          v[4 * q + 0] = a.x; v[4 * q + 1] = a.y; v[4 * q + 2] = a.z; v[4 * q + 3] = a.w;
        }
        const int row = (s >> DEPTH) * p.sub_m + row0 + r;
        const int col0 = (s & (G - 1)) * p.sub_n + tn * BN + c * 32;
        float b[32];
        bias32(p, 0, col0, b);
        finish_plain(p, b, v);
        store_row32(p, row, col0, v);
      }
    }
  }
}

// ------------------------------------------------- on-chip operand sums

// 8 packed 16-bit values -> 8 floats.
__device__ __forceinline__ void unpack8(const uint4& x, float (&f)[8], int is_bf16) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i + 0] = h2f(w[i] & 0xFFFFu, is_bf16);
    f[2 * i + 1] = h2f(w[i] >> 16, is_bf16);
  }
}

// Forms the product's summed operands for one K block: A sum (128 rows x 64)
// and/or B sum (64 rows x BN), each element sum_t sign_t * src_t computed in
// fp32 from the exact 16-bit inputs and rounded once (RNE), written into the
// 128-byte-swizzled operand buffers.  A and B chunks (16 bytes = 8 elements)
// form one work list so every thread keeps U chunks x terms loads in flight
// before it stores anything (the loads come from L2; their latency, not
// bandwidth, is what limits this stage).  TERMS bounds the source blocks of
// one formed operand: 2^DEPTH for the Strassen tables, 4 for the one-level
// Winograd table (whose expanded operands have up to four blocks).
template <int BN, int DEPTH, int TERMS>
__device__ __forceinline__ void form_operands(const KernelParams& p, const StrassenTable& tab, uint8_t* sA,
                                              uint8_t* sB,
                                              int pr, int tm, int tn, int kb, int tid,
                                              int nthreads) {
  constexpr int T = TERMS;                 // terms per formed operand (at most)
  constexpr int G = 1 << DEPTH;            // blocks per dimension
  constexpr int U = T == 2 ? 8 : 4;        // chunks per thread in flight: U * T loads
  constexpr int CPR = BN / 8;              // 16-byte chunks per K-row of the B tile
  const int na = tab.na[pr], nb = tab.nb[pr];
  const int nA = na > 1 ? kBM * 8 : 0;
  const int nB = nb > 1 ? kBK * CPR : 0;
  const int total = nA + nB;
  if (total == 0) return;
  const uint16_t* srcA[T];
  const uint16_t* srcB[T];
  float sgA[T], sgB[T];
#pragma unroll
  for (int t = 0; t < T; ++t) {
    const uint8_t ca = tab.a[pr][t < na ? t : 0];
    const int qa = ca & kTermIndexMask;
    srcA[t] = p.A + static_cast<long long>((qa >> DEPTH) * p.sub_m + tm * kBM) * p.lda +
              (qa & (G - 1)) * p.sub_k + kb * kBK;
    sgA[t] = (ca & kTermNeg) ? -1.0f : 1.0f;
    const uint8_t cb = tab.b[pr][t < nb ? t : 0];
    const int qb = cb & kTermIndexMask;
    srcB[t] = p.B + static_cast<long long>((qb >> DEPTH) * p.sub_k + kb * kBK) * p.ldb +
              (qb & (G - 1)) * p.sub_n + tn * BN;
    sgB[t] = (cb & kTermNeg) ? -1.0f : 1.0f;
  }
  const long long lda = p.lda, ldb = p.ldb;
  const int is_bf16 = p.is_bf16;
#pragma unroll 1
  for (int ch0 = tid; ch0 < total; ch0 += U * nthreads) {
    uint4 v[U][T];
    uint32_t soff[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int ch = ch0 + u * nthreads;
      if (ch < nA) {
        const int row = ch >> 3, c8 = ch & 7;
        const long long goff = row * lda + c8 * 8;
        soff[u] = static_cast<uint32_t>(row * 128 + ((c8 ^ (row & 7)) << 4));
#pragma unroll
        for (int t = 0; t < T; ++t)
          if (t < na) v[u][t] = __ldg(reinterpret_cast<const uint4*>(srcA[t] + goff));
      } else if (ch < total) {
        const int cb = ch - nA;
        const int row = cb / CPR, c = cb % CPR;
        const long long goff = row * ldb + c * 8;
        soff[u] = static_cast<uint32_t>((c >> 3) * 8192 + row * 128 + (((c & 7) ^ (row & 7)) << 4));
#pragma unroll
        for (int t = 0; t < T; ++t)
          if (t < nb) v[u][t] = __ldg(reinterpret_cast<const uint4*>(srcB[t] + goff));
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int ch = ch0 + u * nthreads;
      if (ch < total) {
        const bool is_a = ch < nA;
        const int nt = is_a ? na : nb;
        float acc[8], f[8];
        unpack8(v[u][0], acc, is_bf16);
        const float s0 = is_a ? sgA[0] : sgB[0];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] *= s0;
#pragma unroll
        for (int t = 1; t < T; ++t) {
          if (t < nt) {
            const float st = is_a ? sgA[t] : sgB[t];
            unpack8(v[u][t], f, is_bf16);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] += st * f[i];
          }
        }
        *reinterpret_cast<uint4*>((is_a ? sA : sB) + soff[u]) =
            make_uint4(pack2(acc[0], acc[1], is_bf16), pack2(acc[2], acc[3], is_bf16),
                       pack2(acc[4], acc[5], is_bf16), pack2(acc[6], acc[7], is_bf16));
      }
    }
  }
}

// ---------------------------------------------------------------- kernel

// Launch arguments by depth: the classical kernel takes KernelParams, the
// Strassen kernels StrassenParams.  A classical instantiation gets an unused
// table reference so that the shared code compiles.
template <int DEPTH>
struct KernelArgs {
  using type = StrassenParams;
};
template <>
struct KernelArgs<0> {
  using type = KernelParams;
};
static __device__ StrassenTable g_no_table;
__device__ __forceinline__ const KernelParams& kernel_params(const KernelParams& a) { return a; }
__device__ __forceinline__ const KernelParams& kernel_params(const StrassenParams& a) { return a.k; }
__device__ __forceinline__ const StrassenTable& kernel_table(const KernelParams&) { return g_no_table; }
__device__ __forceinline__ const StrassenTable& kernel_table(const StrassenParams& a) { return a.tab; }

template <int BN, int DEPTH, int TERMS = (1 << DEPTH)>
__global__ void __launch_bounds__(RoleCfg<DEPTH>::kThreads, 1)
    fgemm_kernel(const __grid_constant__ typename KernelArgs<DEPTH>::type args) {
  const KernelParams& p = kernel_params(args);
  const StrassenTable& tab = kernel_table(args);
  using TC = TileCfg<BN>;
  constexpr int S = TC::kStages;
  constexpr int kSumWarps = RoleCfg<DEPTH>::kSumWarps;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw_addr);
  const uint32_t sA0 = base;
  const uint32_t sB0 = base + S * TC::kABytes;
  const uint32_t bar0 = base + S * TC::kStageBytes;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + S * TC::kStageBytes + 8 * (2 * S + 5));
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull = [&](uint32_t b) { return bar0 + 8u * (2 * S + b); };
  auto tempty = [&](uint32_t b) { return bar0 + 8u * (2 * S + 2 + b); };
  const uint32_t drain = bar0 + 8u * (2 * S + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int NP = DEPTH == 0 ? 1 : p.num_products;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(full(s), 1 + kSumWarps);
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
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), TC::kTmemCols);
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
      for (int unit = blockIdx.x; ok && unit < p.num_units; unit += gridDim.x) {
        int tm, tn;
        unit_coords(p, unit, tm, tn);
        for (int pr = 0; ok && pr < NP; ++pr) {
          bool a_raw = true, b_raw = true;
          int ax0 = 0, ay = tm * kBM, by0 = 0;
          int bx[BN / 64];
          if constexpr (DEPTH == 0) {
            if (p.epi == kEpiSwiglu) {
              constexpr int HALF = BN / 2;
#pragma unroll
              for (int q = 0; q < BN / 64; ++q) {
                const int qc = q * 64;
                bx[q] = qc < HALF ? tn * HALF + qc : p.n_out + tn * HALF + (qc - HALF);
              }
            } else {
#pragma unroll
              for (int q = 0; q < BN / 64; ++q) bx[q] = tn * BN + q * 64;
            }
          } else {
            a_raw = tab.na[pr] == 1;
            b_raw = tab.nb[pr] == 1;
            const int qa = tab.a[pr][0] & kTermIndexMask;
            const int qb = tab.b[pr][0] & kTermIndexMask;
            ay = (qa >> DEPTH) * p.sub_m + tm * kBM;
            ax0 = (qa & ((1 << DEPTH) - 1)) * p.sub_k;
            by0 = (qb >> DEPTH) * p.sub_k;
            const int bxb = (qb & ((1 << DEPTH) - 1)) * p.sub_n + tn * BN;
#pragma unroll
            for (int q = 0; q < BN / 64; ++q) bx[q] = bxb + q * 64;
          }
          const uint32_t tx = (a_raw ? TC::kABytes : 0) + (b_raw ? TC::kBBytes : 0);
          for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (!wait_one(empty(s), ph ^ 1u, p, 0)) {
              ok = false;
              break;
            }
            ptx::mbar_arrive_expect_tx(full(s), tx);
            if (a_raw) ptx::tma_load_2d(sA0 + s * TC::kABytes, &p.tmap_a, ax0 + kb * kBK, ay, full(s));
            if (b_raw) {
#pragma unroll
              for (int q = 0; q < BN / 64; ++q)
                ptx::tma_load_2d(sB0 + s * TC::kBBytes + q * 8192, &p.tmap_b, bx[q], by0 + kb * kBK,
                                 full(s));
            }
            if (++s == S) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
      }
      if (!ok) {
        // Let copies already in flight land before the CTA leaves: the last
        // S stages' full barriers (bounded, error word ignored).
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
      const uint32_t b_lbo = 8192;  // 64-column boxes of B are 8 KB apart
      for (int unit = blockIdx.x; ok && unit < p.num_units; unit += gridDim.x) {
        for (int pr = 0; ok && pr < NP; ++pr) {
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
            const uint64_t ad = ptx::sdesc(sA0 + s * TC::kABytes, 16, 1024);
            const uint64_t bd = ptx::sdesc(sB0 + s * TC::kBBytes, b_lbo, 1024);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              // K step of 16: +32 bytes inside the A swizzle row, +16 K-rows (2 KB) of B
              ptx::mma_f16(dt, ad + static_cast<uint64_t>(k * 2), bd + static_cast<uint64_t>(k * 128),
                           p.idesc, (kb | k) != 0 ? 1u : 0u);
            }
            ptx::mma_commit(empty(s));
            if (++s == S) {
              s = 0;
              ph ^= 1u;
            }
          }
          if (ok) ptx::mma_commit(tfull(buf));
        }
      }
      // Every MMA this thread issued is complete before TMEM is released.
      ptx::mma_commit(drain);
      wait_bounded(drain, 0, p, err_code(1), false);
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    // --------------------------------------------------------- epilogue
    const int ew = warp - 4;  // TMEM lane quarter this warp may access
    const int r = ew * 32 + lane;
    float* ws = nullptr;
    if constexpr (DEPTH > 0)
      ws = p.workspace + static_cast<size_t>(blockIdx.x) * (1 << (2 * DEPTH)) * kBM * BN;
    uint32_t acc_it = 0;
    bool ok = true;
    for (int unit = blockIdx.x; ok && unit < p.num_units; unit += gridDim.x) {
      int tm, tn;
      unit_coords(p, unit, tm, tn);
      for (int pr = 0; pr < NP; ++pr) {
        const uint32_t buf = acc_it & 1u, aph = (acc_it >> 1) & 1u;
        ++acc_it;
        if (!wait_warp(tfull(buf), aph, p, 2)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t tbase = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + buf * BN;
        if constexpr (DEPTH == 0) {
          epilogue_classical<BN>(p, tbase, tm * kBM, tn, r);
        } else {
          epilogue_strassen<BN, DEPTH>(p, tab, tbase, tm * kBM, tn, pr, r, ws);
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(tempty(buf));
      }
    }
  } else if (DEPTH > 0 && (warp == 2 || warp == 3 || warp >= 8)) {
    // ------------------------------------------------ operand-sum warps
    const int sw = warp < 4 ? warp - 2 : warp - 6;
    const int tid = sw * 32 + lane;
    constexpr int NT = kSumWarps * 32;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int unit = blockIdx.x; ok && unit < p.num_units; unit += gridDim.x) {
      int tm, tn;
      unit_coords(p, unit, tm, tn);
      for (int pr = 0; ok && pr < NP; ++pr) {
        const bool a_sum = tab.na[pr] > 1;
        const bool b_sum = tab.nb[pr] > 1;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_warp(empty(s), ph ^ 1u, p, 3)) {
            ok = false;
            break;
          }
          if (a_sum || b_sum)
            form_operands<BN, DEPTH, TERMS>(p, tab, base_ptr + s * TC::kABytes,
                                     base_ptr + S * TC::kABytes + s * TC::kBBytes, pr, tm, tn, kb,
                                     tid, NT);
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(full(s));
          if (++s == S) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem_base, TC::kTmemCols);
}

template <int BN, int DEPTH, int TERMS = (1 << DEPTH)>
cudaError_t launch_gemm_t(const KernelParams& p, const StrassenTable* tab, int grid, cudaStream_t stream) {
  auto kern = fgemm_kernel<BN, DEPTH, TERMS>;
  constexpr int smem = TileCfg<BN>::kSmemBytes;
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
  if constexpr (DEPTH == 0) {
    (void)tab;
    kern<<<grid, RoleCfg<DEPTH>::kThreads, smem, stream>>>(p);
  } else {
    if (!tab) return cudaErrorInvalidValue;
    const StrassenParams args{p, *tab};
    kern<<<grid, RoleCfg<DEPTH>::kThreads, smem, stream>>>(args);
  }
  return cudaGetLastError();
}

}  // namespace fgemm
