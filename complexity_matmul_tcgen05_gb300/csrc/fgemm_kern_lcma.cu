// fgemm_kern_lcma.cu -- one Strassen-like level (Strassen's or Winograd's
// scheme), or two Strassen levels, on CTA pairs, with the summed operands
// streamed through HBM (FalconGEMM summary, "Methodology" items 1 and 3).
// Two levels (D == 2) follow the same two steps with the 16 quarter blocks:
// lcma_form2_kernel forms each side's 49 leaf operands (one rounding each),
// and the product kernel runs 49 quarter-size products per position and
// folds them into the 16 output blocks.
//
// Two steps:
//  1. Every summed operand of the scheme is formed once from the 2 x 2 blocks
//     of A and B (e.g. A11 + A22, B12 - B22): each element is the fp32 sum of
//     the exact 16-bit inputs, rounded once to the input type, written to
//     handle-owned temporaries, A and B read once and each temporary written
//     once.  Either lcma_form_kernel does it as a streaming launch before the
//     products, or, for a scheme whose first products read only blocks of A
//     and B (Winograd's A11 B11 and A12 B21), the product kernel's idle warps
//     do it while those run (lcma_form_bands).
//  2. fgemm_kernel_pair_lcma runs the seven block products in one persistent
//     launch on CTA pairs: 256 x BN tiles of the half-size block space, on
//     the classical pair mainloop (TMA -> 128-byte-swizzled shared-memory ring
//     -> tcgen05.mma cta_group::2 -> double-buffered TMEM), so the tensor
//     pipe sees the same operand stream as a classical product.  Each pair
//     runs whole output positions product by product (product 1 of all its
//     positions, then product 2, ...; the pairs in step on the same product,
//     so neighbouring positions share its operand panels in the L2, and
//     consecutive waves reuse them).  The epilogue warps
//     fold each product's accumulator into per-CTA fp32 partial tiles of the
//     output blocks it feeds (C11 = M1 + M4 - M5 + M7, ...): the first
//     contribution to a block is stored, the next ones are added by vector
//     atomic reductions performed at the L2 (no load latency in the fold),
//     and at a block's last contribution the epilogue reads the partial,
//     adds the accumulator, applies alpha / bias / activation and stores C.
//     The partial last wave's positions run as separate (product, position)
//     units shared out evenly over the pairs: each stores its accumulator,
//     and the last of a position's seven to finish (a generation-tagged
//     counter) has them combined in product order, by the idle warps, so the
//     result does not depend on timing.
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

// Row r of block (q >> D, q & (2^D - 1)) of a 2^D x 2^D split of src into
// rows x cols blocks.
template <int D>
__device__ __forceinline__ const uint4* form_src(const LcmaFormJob& J, int q, int r) {
  const uint16_t* base = J.src + static_cast<long long>((q >> D) * J.rows + r) * J.ld +
                         static_cast<long long>(q & ((1 << D) - 1)) * J.cols;
  return reinterpret_cast<const uint4*>(base);
}

// One level: forms every temporary of job J at the R rows r0, r0 + rstep,
// ... (rows past the last are skipped) for the 16-byte column group c8: the
// source blocks' 16 bytes are loaded once (4 R loads in flight), each
// temporary's 16 bytes formed in fp32 (sum of the exact 16-bit values, one
// RNE rounding) and stored.  The sums of one group are independent of every
// other group.
template <int R>
__device__ __forceinline__ void form_rows(const LcmaFormJob& J, int is_bf16, int r0, int rstep, int c8) {
  const long long plane = static_cast<long long>(J.rows) * J.cols;
  uint4 raw[R][4];
#pragma unroll
  for (int h = 0; h < R; ++h) {
    const int r = r0 + h * rstep;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      raw[h][q] = (r < J.rows && ((J.block_mask >> q) & 1u)) ? __ldg(form_src<1>(J, q, r) + c8)
                                                             : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int h = 0; h < R; ++h) {
    const int r = r0 + h * rstep;
    if (r >= J.rows) break;
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
          unpack8(raw[h][q], f, is_bf16);
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[i] += cf > 0 ? f[i] : -f[i];
        }
      }
      *reinterpret_cast<uint4*>(dst + t * plane) =
          make_uint4(pack2(acc[0], acc[1], is_bf16), pack2(acc[2], acc[3], is_bf16),
                     pack2(acc[4], acc[5], is_bf16), pack2(acc[6], acc[7], is_bf16));
    }
  }
}

// The one-level pre-pass as its own launch: one warp per pair of rows and
// 32 column groups of 8 elements (16 bytes) per warp; blockIdx.z selects the
// matrix (A or B).
__global__ void __launch_bounds__(256) lcma_form_kernel(const __grid_constant__ LcmaFormParams P) {
  const LcmaFormJob& J = P.job[blockIdx.z];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cols8 = J.cols >> 3;
  const int c8 = blockIdx.x * 32 + lane;
  if (J.ntemp == 0 || c8 >= cols8) return;
  const int step = gridDim.y * 8;
#pragma unroll 1
  for (int r0 = blockIdx.y * 8 + warp; r0 < J.rows; r0 += 2 * step) form_rows<2>(J, P.is_bf16, r0, step, c8);
}

// Two Strassen levels: product (p, q)'s operand on one side is
// sum_{i, j} c[p][i] c[q][j] X(i, j), X(i, j) quarter block (2 ri + rj,
// 2 ci + cj) for outer block i = (ri, ci) and inner block j = (rj, cj).  One
// thread per row and 16-byte column group: the 16 quarter blocks' 16 bytes
// are loaded once; for each outer combination p the four inner blocks
// Y_j = sum_i c[p][i] X(i, j) are summed in fp32, then each inner combination
// q of them, rounded once to the input type and stored as the temporary that
// holds (p, q) (the four operands that are a single block are read in
// place).  The coefficients are compile-time constants, so only the nonzero
// terms are added.
template <int Side>
__device__ __forceinline__ void form2_group(const LcmaFormJob& J, int is_bf16, int r, int c8) {
  uint4 raw[16];
#pragma unroll
  for (int q = 0; q < 16; ++q) raw[q] = __ldg(form_src<2>(J, q, r) + c8);
  const long long plane = static_cast<long long>(J.rows) * J.cols;
  uint16_t* dst = J.dst + static_cast<long long>(r) * J.cols + c8 * 8;
#pragma unroll
  for (int p = 0; p < 7; ++p) {
    float y[4][8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int e = 0; e < 8; ++e) y[j][e] = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = strassen_coef(Side, p, i);
        if (c == 0) continue;
        const int q16 = (2 * (i >> 1) + (j >> 1)) * 4 + 2 * (i & 1) + (j & 1);
        float f[8];
        unpack8(raw[q16], f, is_bf16);
#pragma unroll
        for (int e = 0; e < 8; ++e) y[j][e] += c > 0 ? f[e] : -f[e];
      }
    }
#pragma unroll
    for (int q = 0; q < 7; ++q) {
      const int t = J.leaf_temp[p * 7 + q];
      if (t < 0) continue;
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = strassen_coef(Side, q, j);
        if (c == 0) continue;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += c > 0 ? y[j][e] : -y[j][e];
      }
      *reinterpret_cast<uint4*>(dst + t * plane) =
          make_uint4(pack2(acc[0], acc[1], is_bf16), pack2(acc[2], acc[3], is_bf16),
                     pack2(acc[4], acc[5], is_bf16), pack2(acc[6], acc[7], is_bf16));
    }
  }
}

// The two-level pre-pass: one warp per row and 32 column groups;
// blockIdx.z selects the matrix (A or B).
__global__ void __launch_bounds__(256) lcma_form2_kernel(const __grid_constant__ LcmaFormParams P) {
  const LcmaFormJob& J = P.job[blockIdx.z];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c8 = blockIdx.x * 32 + lane;
  const int r = blockIdx.y * 8 + warp;
  if (J.ntemp == 0 || c8 >= (J.cols >> 3) || r >= J.rows) return;
  if (blockIdx.z == 0)
    form2_group<0>(J, P.is_bf16, r, c8);
  else
    form2_group<1>(J, P.is_bf16, r, c8);
}

cudaError_t launch_lcma_form(const LcmaFormParams& f, int depth, int num_sms, cudaStream_t stream) {
  int max_cols8 = 0, max_rows = 0;
  for (int j = 0; j < 2; ++j) {
    if (f.job[j].ntemp == 0) continue;
    max_cols8 = std::max(max_cols8, f.job[j].cols / 8);
    max_rows = std::max(max_rows, f.job[j].rows);
  }
  if (max_cols8 == 0) return cudaSuccess;
  const int gx = (max_cols8 + 31) / 32;
  if (depth == 2) {
    if ((max_rows + 7) / 8 > 65535) return cudaErrorInvalidValue;
    lcma_form2_kernel<<<dim3(gx, (max_rows + 7) / 8, 2), 256, 0, stream>>>(f);
    return cudaGetLastError();
  }
  // about 16 blocks of 8 warps per SM over both matrices, each warp looping over rows
  const int gy = std::max(1, std::min((max_rows + 7) / 8, std::max(1, num_sms * 8 / gx)));
  if (depth != 1) return cudaErrorInvalidValue;
  lcma_form_kernel<<<dim3(gx, std::min(gy, 65535), 2), 256, 0, stream>>>(f);
  return cudaGetLastError();
}

// ------------------------------------------------------- product kernel

template <int BN, int D>
struct LcmaCfg {
  static constexpr int kABytes = kBM * kBK * 2;        // this CTA's 128 rows of A
  static constexpr int kBBytes = kBK * (BN / 2) * 2;   // this CTA's BN/2 columns of B
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = BN == 256 ? 6 : 8;
  static constexpr int kTmemCols = BN == 256 ? 512 : 256;
  // The combination queue after the barriers: head, taken, epilogue warps
  // done, progress, then one word per job.  A tail unit hands at most
  // kMaxTerms groups x 4 warps of combinations, and a pair has fewer than
  // 7^D tail units.
  static constexpr int kQueueOff = 256;
  static constexpr int kQueueCap = D == 1 ? 128 : 1024;
  static constexpr int kBarBytes = D == 1 ? 1024 : 5120;
  // After the barriers, one B half of slack: even a full-width MMA read of
  // the last stage stays inside this CTA's shared memory.
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kBarBytes + kBBytes;
  static constexpr int kChunks = BN / 32;
  static constexpr int kBlocks = 1 << (2 * D);  // output blocks of D levels
  static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
  static_assert(kQueueOff + 4 * (4 + kQueueCap) <= kBarBytes, "combination queue does not fit");
  static_assert(kMaxTerms * 4 * 7 <= kQueueCap && (D == 1 || kMaxTerms * 4 * 49 <= kQueueCap),
                "a pair's tail jobs must fit the queue");
  static_assert(2 * BN <= kTmemCols, "two accumulator buffers must fit in TMEM");
  static_assert((2 * kStages + 5) * 8 + 4 <= kBarBytes, "barrier area too small");
};

// The schedule.  With P pairs and `positions` output positions (256 x BN
// tiles of the half-size block space, in rasterised order), the first
// W = floor(positions / P) waves are whole positions: pair c owns positions
// c, c + P, c + 2P, ... and runs them product by product, product 0 for all
// of them, then product 1, ...  At any moment the pairs work on the same
// product and on neighbouring positions, and consecutive waves of one
// product reuse its operand panels in the L2: each product is run like a
// classical product of its two operands.  Every position still sees its
// products in order, so its fold adds them in product order.
// The T = positions - W P positions of the partial last wave are cut into
// their 7 T units (product, position), product-major (unit t: product
// t / T, position W P + t mod T), shared out in equal contiguous ranges, one
// per pair.  A tail unit stores its accumulator; the last of a position's
// seven units to finish combines them, a chain of dependent loads that is
// long next to a unit's MMAs.  So a pair runs its tail units among its whole
// positions, after the whole positions' first `tail_at` products: the
// combinations then overlap the MMAs of the products that follow.  (With
// the temporaries formed in this kernel, tail_at leaves time for them to be
// stored first.)
struct LcmaItem {
  long long pos;   // output position (unit_coords order)
  int pr;          // product
  int slot;        // whole position: its index among the pair's whole positions
  long long tail;  // tail unit index, or -1 for a product of a whole position
};

struct LcmaSchedule {
  long long whole;   // W: whole positions per pair
  long long tail0;   // W * P: the first tail position
  long long tail_n;  // T: tail positions
  long long tlo, thi;  // this pair's tail units [tlo, thi)
  long long head;    // whole-position items before the tail units: W * tail_at
  __device__ LcmaSchedule(long long positions, int pairs, int np, int tail_at, int c) {
    whole = positions / pairs;
    tail0 = whole * pairs;
    tail_n = positions - tail0;
    const long long ut = tail_n * np;
    tlo = static_cast<long long>(c) * ut / pairs;
    thi = static_cast<long long>(c + 1) * ut / pairs;
    head = whole * min(max(tail_at, 0), np);
  }
  __device__ long long items(int np) const { return whole * np + (thi - tlo); }
  __device__ LcmaItem item(long long n, int np, int pairs, int c) const {
    LcmaItem it;
    const long long nt = thi - tlo;
    if (n >= head && n < head + nt) {
      it.slot = -1;
      it.tail = tlo + (n - head);
      it.pr = static_cast<int>(it.tail / tail_n);
      it.pos = tail0 + it.tail % tail_n;
    } else {
      const long long w = n < head ? n : n - nt;  // index among the whole-position items
      it.slot = static_cast<int>(w % whole);
      it.pos = c + it.slot * pairs;
      it.pr = static_cast<int>(w / whole);
      it.tail = -1;
    }
    return it;
  }
};

// fp32 tiles in global memory (a CTA's partial of one output block of one
// of its whole positions, or the accumulator of a tail unit): 128 rows x BN,
// laid out [32-column chunk][column quad: 8][row: 128][4], so that a warp's
// 16-byte accesses to one (chunk, quad) cover 512 contiguous bytes.  These
// return the chunk's base; row r's quad q is at index q * 128 + r.  A CTA's
// partials: `whole` slots (its whole positions) of the four blocks.
template <int BN, int D>
__device__ __forceinline__ float4* lcma_part(float* ws, long long whole, int cta, int slot, int blk, int c) {
  using LC = LcmaCfg<BN, D>;
  return reinterpret_cast<float4*>(
      ws + ((static_cast<size_t>(cta) * whole + slot) * LC::kBlocks + blk) * (kBM * BN) +
      static_cast<size_t>(c) * (kBM * 32));
}

template <int BN>
__device__ __forceinline__ float4* lcma_tail_part(float* ws, long long t, uint32_t rank, int c) {
  return reinterpret_cast<float4*>(ws + (static_cast<size_t>(t) * 2 + rank) * (kBM * BN) +
                                   static_cast<size_t>(c) * (kBM * 32));
}

// v[j] = (add ? v[j] : 0) + sg * row r of a 32-column chunk.
__device__ __forceinline__ void lcma_load_row(const float4* chunk, int r, float (&v)[32], bool add,
                                              float sg) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 f = __ldcg(chunk + q * kBM + r);
    if (add) {
      v[4 * q + 0] += sg * f.x; v[4 * q + 1] += sg * f.y; v[4 * q + 2] += sg * f.z; v[4 * q + 3] += sg * f.w;
    } else {
      v[4 * q + 0] = sg * f.x; v[4 * q + 1] = sg * f.y; v[4 * q + 2] = sg * f.z; v[4 * q + 3] = sg * f.w;
    }
  }
}

// Stores (or, add == true, atomically adds) sg * v (fp32 bit patterns) as
// row r of a chunk.  Every address of a partial is only ever written by one
// thread, whose operations on it take effect in program order, so the fp32
// additions happen in product order whatever the timing.
__device__ __forceinline__ void lcma_put_row(float4* chunk, int r, const uint32_t (&v)[32], float sg,
                                             bool add) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 f = make_float4(sg * __uint_as_float(v[4 * q + 0]), sg * __uint_as_float(v[4 * q + 1]),
                                 sg * __uint_as_float(v[4 * q + 2]), sg * __uint_as_float(v[4 * q + 3]));
    if (add)
      atomicAdd(chunk + q * kBM + r, f);
    else
      __stcg(chunk + q * kBM + r, f);
  }
}

// alpha / bias / activation of output block blk (or, for SwiGLU, of gate
// block 2 sr and up block 2 sr + 1 given as g and u) for 32 columns of chunk
// c of position (tm, tn), and the store of C by this thread's row.
template <int BN, int D>
__device__ __forceinline__ void lcma_emit(const KernelParams& p, int blk, int c, int tm, int tn,
                                          uint32_t rank, int r, float (&v)[32]) {
  const int col0 = (blk & ((1 << D) - 1)) * p.sub_n + tn * BN + c * 32;
  float b[32];
  bias32(p, 0, col0, b);
  finish_plain(p, b, v);
  store_row32(p, (blk >> D) * p.sub_m + tm * (2 * kBM) + static_cast<int>(rank) * kBM + r, col0, v);
}

template <int BN>
__device__ __forceinline__ void lcma_emit_swiglu(const KernelParams& p, int sr, int c, int tm, int tn,
                                                 uint32_t rank, int r, float (&g)[32], const float (&u)[32]) {
  const int col0 = tn * BN + c * 32;
  finish_swiglu_warp(p, col0, g, u);
  store_row32(p, sr * p.sub_m + tm * (2 * kBM) + static_cast<int>(rank) * kBM + r, col0, g);
}

// Finishes output group g of a tail position (its index among the T tail
// positions) for this warp's 32 rows of this CTA: output block g, or for
// SwiGLU block row g (gate block 2g, up block 2g + 1).  Every block is the
// sum, in product order with the scheme's signs, of the stored accumulators
// of the products that feed it, so the result does not depend on which unit
// finished last.
template <int BN, int D>
__device__ void lcma_finish_tail(const LcmaParams& L, long long tail_pos, long long tail_n, int g, int tm,
                                 int tn, uint32_t rank, int ew) {
  using LC = LcmaCfg<BN, D>;
  const KernelParams& p = L.k;
  const int r = ew * 32 + (threadIdx.x & 31);
  const int np = p.num_products;
  auto gather = [&](int blk, int c, float (&v)[32]) {
    bool any = false;
    for (int k = 0; k < np; ++k) {
      for (int t = 0; t < L.prod[k].nc; ++t) {
        const uint8_t code = L.prod[k].c[t];
        if ((code & kTermIndexMask) != blk) continue;
        lcma_load_row(lcma_tail_part<BN>(p.split_ws, k * tail_n + tail_pos, rank, c), r, v, any,
                      (code & kTermNeg) ? -1.0f : 1.0f);
        any = true;
      }
    }
    if (!any) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 0.0f;
    }
  };
  if (D == 1 && p.epi == kEpiSwiglu) {
#pragma unroll 1
    for (int c = 0; c < LC::kChunks; ++c) {
      float gv[32], uv[32];
      gather(g * 2, c, gv);
      gather(g * 2 + 1, c, uv);
      lcma_emit_swiglu<BN>(p, g, c, tm, tn, rank, r, gv, uv);
    }
  } else {
#pragma unroll 1
    for (int c = 0; c < LC::kChunks; ++c) {
      float v[32];
      gather(g, c, v);
      lcma_emit<BN, D>(p, g, c, tm, tn, rank, r, v);
    }
  }
}

// Operand formation inside the product kernel, by one warp: claims bands
// of kFormRows rows (the jobs' row counts are multiples of it) of job 0
// (A), then of job 1 (B), until none is left, forms each band's
// temporaries over the full width (four rows in flight per lane) and counts
// the band as stored.  The release: every lane's stores,
// then its fences (async proxy, GPU scope), then the warp barrier, then lane
// 0's increment.  A warp never waits for another CTA here, so every band a
// running CTA has claimed is stored whatever else runs on the GPU.
__device__ __forceinline__ void lcma_form_bands(const LcmaParams& L) {
  const int lane = threadIdx.x & 31;
  const int total = L.form_tasks[0] + L.form_tasks[1];
#pragma unroll 1
  while (true) {
    int t = 0;
    if (lane == 0) t = static_cast<int>(atomicAdd(L.form_ctr, 1u));
    t = __shfl_sync(0xFFFFFFFFu, t, 0);
    if (t >= total) break;
    const int j = t < L.form_tasks[0] ? 0 : 1;
    const LcmaFormJob& J = L.form.job[j];
    const int r0 = (t - (j ? L.form_tasks[0] : 0)) * kFormRows;
    const int r1 = r0 + kFormRows;  // the host asks for whole bands
    const int cols8 = J.cols >> 3;
#pragma unroll 1
    for (int r = r0; r < r1; r += 4)
#pragma unroll 1
      for (int c8 = lane; c8 < cols8; c8 += 32) form_rows<4>(J, L.form.is_bf16, r, 1, c8);
    ptx::fence_proxy_async_global();
    __threadfence();
    __syncwarp();
    if (lane == 0) atomicAdd(L.form_ctr + 1 + j, 1u);
  }
}

// Bounded wait of a producer until every band of job j is stored (then its
// later bulk-tensor loads see the temporaries).  Gives up when another role
// latched an error, or latches a timeout of the operand-sum role.
static __device__ __noinline__ bool lcma_wait_formed(const LcmaParams& L, int j) {
  const KernelParams& p = L.k;
  const unsigned int need = static_cast<unsigned int>(L.form_tasks[j]);
  const unsigned int* ctr = L.form_ctr + 1 + j;
  const uint64_t t0 = ptx::globaltimer();
#pragma unroll 1
  while (ptx::ld_acquire_gpu(ctr) < need) {
    if (*reinterpret_cast<volatile unsigned int*>(p.err) != 0u) return false;
    if (ptx::globaltimer() - t0 > p.spin_ns) {
      atomicCAS(p.err, 0u, err_code(3));
      return false;
    }
    __nanosleep(200);
  }
  ptx::fence_proxy_async_global();
  return true;
}

// The combinations of tail positions, run by warps 2 and 3 (idle once the
// operands are formed) so that the epilogue warps go on with the next
// accumulator.  An epilogue warp that finds it has the last unit of an
// output group appends a job (tail position, group, its warp index: the
// 32 rows to combine) to the CTA's queue in shared memory; a helper claims
// jobs in order and runs each.  The queue ends when all four epilogue
// warps have said they are done and every appended job is taken.  A helper
// may wait for its next job as long as the epilogue keeps finishing
// accumulators (queue word 3 counts them): its bound restarts at each one.
// It leaves on another role's error.
template <int BN, int D>
__device__ __forceinline__ void lcma_tail_helper(const LcmaParams& L, volatile uint32_t* q,
                                                 const LcmaSchedule& sched, uint32_t rank) {
  using LC = LcmaCfg<BN, D>;
  const KernelParams& p = L.k;
  const int lane = threadIdx.x & 31;
#pragma unroll 1
  while (true) {
    uint32_t i = 0, job = 0, quit = 0;
    if (lane == 0) {
      i = atomicAdd(const_cast<uint32_t*>(q + 1), 1u);
      uint64_t t0 = ptx::globaltimer();
      uint32_t beat = q[3];
#pragma unroll 1
      while (true) {
        if (i < static_cast<uint32_t>(LC::kQueueCap)) {
          job = q[4 + i];
          if (job != 0u) break;
        }
        if (q[2] == 4u && i >= q[0]) {  // done flags first: then the head is final
          quit = 1;
          break;
        }
        if (*reinterpret_cast<volatile unsigned int*>(p.err) != 0u) {
          quit = 1;
          break;
        }
        const uint32_t b = q[3];
        if (b != beat) {
          beat = b;
          t0 = ptx::globaltimer();
        } else if (ptx::globaltimer() - t0 > p.spin_ns) {
          atomicCAS(p.err, 0u, err_code(2));
          quit = 1;
          break;
        }
        __nanosleep(256);
      }
    }
    quit = __shfl_sync(0xFFFFFFFFu, quit, 0);
    job = __shfl_sync(0xFFFFFFFFu, job, 0);
    if (quit) break;
    __threadfence();  // the feeding units' stores, seen by the appending warp, are seen here
    const long long tail_pos = static_cast<long long>((job & 0x7FFFFFFFu) >> 6);
    int tm, tn;
    unit_coords(p, static_cast<int>(sched.tail0 + tail_pos), tm, tn);
    lcma_finish_tail<BN, D>(L, tail_pos, sched.tail_n, static_cast<int>((job >> 2) & 15u), tm, tn, rank,
                            static_cast<int>(job & 3u));
  }
}

template <int BN, int D>
__global__ void __launch_bounds__(256, 1) fgemm_kernel_pair_lcma(const __grid_constant__ LcmaParams L) {
  using LC = LcmaCfg<BN, D>;
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
  volatile uint32_t* queue = reinterpret_cast<volatile uint32_t*>(base_ptr + S * LC::kStageBytes + LC::kQueueOff);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1;
  const int pairs = gridDim.x >> 1;
  const int np = p.num_products;
  const LcmaSchedule sched(p.num_units, pairs, np, L.tail_at, cluster);
  const long long n_items = sched.items(np);

  for (int i = threadIdx.x; i < 4 + LC::kQueueCap; i += blockDim.x) queue[i] = 0u;
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
      // Where item n's operand tiles come from: the tensor maps and the
      // coordinates of this CTA's first K block.
      struct Src {
        const CUtensorMap* amap;
        const CUtensorMap* bmap;
        int ax, ay, bx, by;
      };
      auto source = [&](long long n) {
        const LcmaItem it = sched.item(n, np, pairs, cluster);
        const LcmaProduct& P = L.prod[it.pr];
        int tm, tn;
        unit_coords(p, static_cast<int>(it.pos), tm, tn);
        Src o;
        o.amap = P.a_temp ? &L.tmap_ta : &p.tmap_a;
        o.bmap = P.b_temp ? &L.tmap_tb : &p.tmap_b;
        constexpr int kCol = (1 << D) - 1;
        o.ay = (P.a_temp ? P.a_idx : (P.a_idx >> D)) * p.sub_m + tm * (2 * kBM) + static_cast<int>(rank) * kBM;
        o.ax = P.a_temp ? 0 : (P.a_idx & kCol) * p.sub_k;
        o.by = (P.b_temp ? P.b_idx : (P.b_idx >> D)) * p.sub_k;
        o.bx = (P.b_temp ? 0 : (P.b_idx & kCol) * p.sub_n) + tn * BN + static_cast<int>(rank) * (BN / 2);
        return o;
      };
      // sides whose temporaries this producer may read (the pre-pass formed
      // them before the launch, or this kernel has finished forming them)
      bool formed[2] = {L.form_tasks[0] == 0, L.form_tasks[1] == 0};
      for (long long n = 0; ok && n < n_items; ++n) {
        const Src cur = source(n);
        for (int j = 0; j < 2; ++j) {
          if (formed[j] || !(j == 0 ? cur.amap == &L.tmap_ta : cur.bmap == &L.tmap_tb)) continue;
          if (!lcma_wait_formed(L, j)) {
            ok = false;
            break;
          }
          formed[j] = true;
        }
        if (!ok) break;
        const CUtensorMap* amap = cur.amap;
        const CUtensorMap* bmap = cur.bmap;
        const int ax = cur.ax, ay = cur.ay, bx = cur.bx, by = cur.by;
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
      for (long long n = 0; ok && n < n_items; ++n) {
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
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------- operand formation (both CTAs)
    if (L.form_tasks[0] + L.form_tasks[1] > 0) lcma_form_bands(L);
    // ------------------------------------------- tail combinations (both CTAs)
    lcma_tail_helper<BN, D>(L, queue, sched, rank);
  } else if (warp >= 4) {
    // ------------------------------------------- epilogue (both CTAs)
    const int ew = warp - 4;
    const int r = ew * 32 + lane;
    uint32_t acc_it = 0;
    bool ok = true;
    for (long long n = 0; ok && n < n_items; ++n) {
      const LcmaItem it = sched.item(n, np, pairs, cluster);
      const uint32_t buf = acc_it & 1u, aph = (acc_it >> 1) & 1u;
      ++acc_it;
      if (!wait_warp(tfull(buf), aph, p, 2)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t tbase = tmem_base + (static_cast<uint32_t>(ew * 32) << 16) + buf * BN;
      const LcmaProduct& P = L.prod[it.pr];
      const int nc = P.nc;
      int tm, tn;
      unit_coords(p, static_cast<int>(it.pos), tm, tn);
#pragma unroll 1
      for (int c = 0; c < LC::kChunks; ++c) {
        uint32_t ar[32];
        ptx::tmem_ld_32x32b_x32(tbase + c * 32, ar);
        ptx::tmem_wait_ld();
        ptx::tmem_regs_ready(ar);
        if (it.tail >= 0) {  // a tail unit keeps its accumulator as it is
          lcma_put_row(lcma_tail_part<BN>(p.split_ws, it.tail, rank, c), r, ar, 1.0f, false);
          continue;
        }
        // fold into the partials of the blocks this product feeds, except
        // where it is the block's last contribution (finished below)
        for (int t = 0; t < nc; ++t) {
          const uint8_t code = P.c[t];
          if (code & kTermLast) continue;
          lcma_put_row(lcma_part<BN, D>(p.workspace, sched.whole, static_cast<int>(blockIdx.x), it.slot,
                                        code & kTermIndexMask, c),
                       r, ar,
                       (code & kTermNeg) ? -1.0f : 1.0f, !(code & kTermFirst));
        }
        if (!P.fin) continue;
        // the value of block blk once this product is in: its partial (the
        // earlier products, in order) plus this product's share, if any (the
        // chunk is read from TMEM again, so no copy of it stays live here)
        auto final_block = [&](int blk, float (&v)[32]) {
          bool fed = false, first = false;
          float sg = 1.0f;
          for (int t = 0; t < nc; ++t) {
            if ((P.c[t] & kTermIndexMask) != blk) continue;
            fed = true;
            first = (P.c[t] & kTermFirst) != 0;
            sg = (P.c[t] & kTermNeg) ? -1.0f : 1.0f;
          }
          if (!first)
            lcma_load_row(lcma_part<BN, D>(p.workspace, sched.whole, static_cast<int>(blockIdx.x), it.slot, blk, c),
                          r, v, false, 1.0f);
          if (fed) {
            uint32_t x[32];
            ptx::tmem_ld_32x32b_x32(tbase + c * 32, x);
            ptx::tmem_wait_ld();
            ptx::tmem_regs_ready(x);
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = first ? sg * __uint_as_float(x[j]) : v[j] + sg * __uint_as_float(x[j]);
          }
        };
        if (D == 1 && p.epi == kEpiSwiglu) {
#pragma unroll 1
          for (int sr = 0; sr < 2; ++sr) {
            if (!((P.fin >> sr) & 1u)) continue;
            float g[32], u[32];
            final_block(sr * 2, g);
            final_block(sr * 2 + 1, u);
            lcma_emit_swiglu<BN>(p, sr, c, tm, tn, rank, r, g, u);
          }
        } else {
#pragma unroll 1
          for (int blk = 0; blk < LC::kBlocks; ++blk) {
            if (!((P.fin >> blk) & 1u)) continue;
            float v[32];
            final_block(blk, v);
            lcma_emit<BN, D>(p, blk, c, tm, tn, rank, r, v);
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa(tempty(buf), 0));
      if (ew == 0 && lane == 0) queue[3] = static_cast<uint32_t>(n) + 1u;  // progress, for the helpers
      if (it.tail < 0) continue;
      // a tail unit: for every output group (block, or SwiGLU block row) it
      // feeds, the last of the group's feeding units to finish combines them
      const long long tail_pos = it.pos - sched.tail0;
      __threadfence();
      __syncwarp();
#pragma unroll 1
      for (int g = 0; g < LC::kBlocks; ++g) {
        if (!((P.groups >> g) & 1u)) continue;
        const bool last = count_arrival(
            p, p.split_ctr + ((static_cast<size_t>(tail_pos) * LC::kBlocks + g) * 2 + rank) * 4 + ew,
            L.group_pieces[g]);
        if (!last) continue;
        __threadfence();
        if (lane == 0) {
          const uint32_t slot = atomicAdd(const_cast<uint32_t*>(queue), 1u);
          if (slot < static_cast<uint32_t>(LC::kQueueCap))
            queue[4 + slot] = 0x80000000u | (static_cast<uint32_t>(tail_pos) << 6) |
                              (static_cast<uint32_t>(g) << 2) | static_cast<uint32_t>(ew);
          else
            atomicCAS(p.err, 0u, err_code(2));  // not reached: the host bounds the units per pair
        }
        __syncwarp();
      }
    }
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      atomicAdd(const_cast<uint32_t*>(queue + 2), 1u);
    }
  }

  ptx::tc_fence_before();
  ptx::cluster_sync();  // no CTA leaves while its peer may still signal it
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc_pair(tmem_base, LC::kTmemCols);
}

template <int BN, int D>
cudaError_t lcma_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute (&attr)[1], int& fit,
                        cudaStream_t stream) {
  auto kern = fgemm_kernel_pair_lcma<BN, D>;
  constexpr int smem = LcmaCfg<BN, D>::kSmemBytes;
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

int lcma_pair_clusters_fit(int bn, int depth) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  int fit = 0;
  cudaError_t e = cudaErrorInvalidValue;
  if (depth == 1)
    e = bn == 256 ? lcma_config<256, 1>(cfg, attr, fit, nullptr)
                  : (bn == 128 ? lcma_config<128, 1>(cfg, attr, fit, nullptr) : cudaErrorInvalidValue);
  else if (depth == 2)
    e = bn == 256 ? lcma_config<256, 2>(cfg, attr, fit, nullptr)
                  : (bn == 128 ? lcma_config<128, 2>(cfg, attr, fit, nullptr) : cudaErrorInvalidValue);
  return e == cudaSuccess ? fit : 0;
}

template <int BN, int D>
cudaError_t launch_lcma_pair_t(const LcmaParams& L, int clusters, cudaStream_t stream) {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  int fit = 0;
  cudaError_t e = lcma_config<BN, D>(cfg, attr, fit, stream);
  if (e != cudaSuccess) return e;
  if (clusters < 1 || clusters > fit || clusters > L.k.num_units * L.k.num_products ||
      L.k.num_products != (D == 1 ? 7 : 49) || (D == 2 && L.k.epi == kEpiSwiglu))
    return cudaErrorInvalidValue;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  return cudaLaunchKernelEx(&cfg, fgemm_kernel_pair_lcma<BN, D>, L);
}

cudaError_t launch_lcma_pair(int bn, int depth, const LcmaParams& L, int clusters, cudaStream_t stream) {
  if (depth == 1 && bn == 128) return launch_lcma_pair_t<128, 1>(L, clusters, stream);
  if (depth == 1 && bn == 256) return launch_lcma_pair_t<256, 1>(L, clusters, stream);
  if (depth == 2 && bn == 128) return launch_lcma_pair_t<128, 2>(L, clusters, stream);
  if (depth == 2 && bn == 256) return launch_lcma_pair_t<256, 2>(L, clusters, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fgemm
