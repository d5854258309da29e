// fgemm_internal.h -- definitions shared by the host API and the kernel
// translation units (not part of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fgemm {

constexpr int kBM = 128;          // output tile rows (tcgen05 M = 128, one CTA)
constexpr int kBK = 64;           // K per pipeline stage = one 128-byte swizzle row
constexpr int kMaxDepth = 2;      // Strassen recursion levels supported
constexpr int kMaxProducts = 49;  // 7^2
constexpr int kMaxTerms = 4;      // 2^depth source blocks per formed operand

// Term codes in the Strassen tables: bits [0,5) block index
// (row_block << depth | col_block) in the 2^depth x 2^depth block grid,
// bit 6 = first contribution to that output block, bit 7 = negative sign.
constexpr uint8_t kTermIndexMask = 0x1F;
constexpr uint8_t kTermFirst = 0x40;
constexpr uint8_t kTermNeg = 0x80;

// Product p multiplies (sum of a-terms of A) by (sum of b-terms of B) and adds
// its result, with the c-terms' signs, into output blocks.  For depth 0 there
// is one product with one term of each kind.
struct StrassenTable {
  uint8_t na[kMaxProducts];
  uint8_t nb[kMaxProducts];
  uint8_t nc[kMaxProducts];
  uint8_t a[kMaxProducts][kMaxTerms];
  uint8_t b[kMaxProducts][kMaxTerms];
  uint8_t c[kMaxProducts][kMaxTerms];
};

enum EpiKind : int { kEpiNone = 0, kEpiScaleBias = 1, kEpiSilu = 2, kEpiSwiglu = 3 };

struct KernelParams {
  CUtensorMap tmap_a;  // A: inner dim K, outer M, box {64, 128}, 128B swizzle
  CUtensorMap tmap_b;  // B: inner dim N, outer K, box {64, 64},  128B swizzle
  const uint16_t* A;
  const uint16_t* B;
  uint16_t* C;
  const uint16_t* bias;   // N entries (virtual column index) or nullptr
  float* workspace;       // Strassen partial tiles, 4^depth * 128 * BN floats per CTA
  unsigned int* err;      // device error word (0 = ok)
  long long lda, ldb, ldc;
  unsigned long long spin_ns;  // bound of every mbarrier wait
  int M, N, K;            // virtual GEMM: A is M x K, B is K x N
  int n_out;              // columns of C (N, or N/2 for SwiGLU)
  int sub_m, sub_n, sub_k;  // block sizes of one product (M, N, K >> depth)
  int tiles_m, tiles_n;   // output tile grid of one product (256-row tiles on CTA pairs)
  int num_units;          // tiles_m * tiles_n
  int k_blocks;           // ceil(sub_k / 64)
  int epi;                // EpiKind
  int is_bf16;
  int raster_group;       // tile rows per rasterisation group
  uint32_t idesc;         // tcgen05 instruction descriptor
  float alpha;
  int num_products;
  StrassenTable tab;
};

// Error word layout written by a kernel whose bounded wait ran out.
constexpr unsigned int kErrTimeout = 0x80000000u;
// bits [24,28): role (0 producer, 1 mma, 2 epilogue, 3 operand-sum), [0,24): block

size_t kernel_smem_bytes(int bn, int depth);
int kernel_threads(int depth);

// Launches the persistent GEMM kernel for tile width bn (64/128/256) and
// Strassen depth (0 = classical) with `grid` CTAs on `stream`.
cudaError_t launch_gemm(int bn, int depth, const KernelParams& p, int grid,
                        cudaStream_t stream);

// Classical kernel on CTA pairs: 256 x bn tiles (bn = 128 or 256), at most
// `max_clusters` pairs (fewer if fewer fit on the device at once).
cudaError_t launch_gemm_pair(int bn, const KernelParams& p, int max_clusters, cudaStream_t stream);

// One-level Strassen on CTA pairs (256 x bn tiles of the half-size block space).
cudaError_t launch_strassen_pair(int bn, const KernelParams& p, int max_clusters,
                                 cudaStream_t stream);

// The Strassen coefficient table of `depth` levels (0: one trivial product).
const StrassenTable& strassen_table(int depth);

// One block whose bounded wait on a never-completed mbarrier runs out.
cudaError_t launch_selftest_wait(const KernelParams& p, cudaStream_t stream);

// C[i][j] = epi(bias[j]) for K == 0 (the product is empty).
cudaError_t launch_k0_fill(const KernelParams& p, cudaStream_t stream);

}  // namespace fgemm
